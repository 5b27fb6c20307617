"""GPU parity of art_select_blocks (key-based block selection writing an ART
visit list) against the CPU oracle (oracle/select.py), through the C ABI.

The selected sets must match the oracle's, except for blocks whose oracle
score lies within a relative 1e-5 of the score at the cut (fp32 block sums on
the device, fp64 in the oracle); the order must be block 0, then descending
block index, then -1.
"""
import numpy as np
import pytest

import workloads as W
from oracle import select as S

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import kv_cache_early_gb300 as K  # noqa: E402

TIE_REL = 1e-5


def run_select(w, top_frac, keep_last, max_visit=None, order=0):
    dev = K.DeviceInputs(w)
    T_max = -(-w.max_pages_per_seq * w.page_size // w.block_size)
    need = min(T_max, int(np.ceil(top_frac * T_max)) + 1 + keep_last)
    mv = max_visit or need
    shape = K.make_shape(**dict(w.shape_dict(), max_visit=mv))
    vis = torch.full((w.batch, w.num_kv_heads, mv), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(K.art_select_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    K.art_select_blocks(dev.q, dev.k_cache, dev.block_table, dev.seq_lens, top_frac, keep_last, vis, shape, ws,
                        order=order)
    torch.cuda.synchronize()
    return vis.cpu().numpy().reshape(w.num_items, mv), K.art_read_device_status(ws)


def check(w, got, top_frac, keep_last, items=None):
    ref = S.select_blocks(w, top_frac, keep_last, items=items)
    ties = 0
    for it, (lst, sc) in ref.items():
        row = got[it]
        n = int((row >= 0).sum())
        assert (row[:n] >= 0).all() and (row[n:] == -1).all(), f"item {it}: -1 must end the list"
        dl = [int(x) for x in row[:n]]
        if lst == dl:
            continue
        T = len(sc)
        assert dl and dl[0] == 0 and all(a > b for a, b in zip(dl[1:], dl[2:])), f"item {it}: order {dl}"
        k = min(T, int(np.ceil(top_frac * T)))
        cut = np.sort(sc)[::-1][k - 1] if k > 0 else 0.0
        scale = max(abs(cut), float(np.abs(sc).mean()), 1e-30)
        for c in set(lst) ^ set(dl):
            assert abs(sc[c] - cut) <= TIE_REL * scale, f"item {it}: block {c} score {sc[c]} vs cut {cut}"
        ties += 1
    return ties


@pytest.mark.parametrize("k", [1, 2, 4, 5])
@pytest.mark.parametrize("frac,last", [(0.25, 8), (0.5, 0), (0.0, 3), (1.0, 0)])
def test_select_small(k, frac, last):
    w = W.config(k, small=True)
    got, st = run_select(w, frac, last)
    assert st == 0
    ties = check(w, got, frac, last)
    assert ties <= max(1, w.num_items // 10)


def test_select_reproduces_the_long_context_lists():
    """On the full long-context workload the device selection gives the lists
    the benchmark feeds to ART (built on the host in fp64)."""
    w = W.config(5)
    mv = w.visit_order.shape[-1]
    got, st = run_select(w, 0.25, 8, max_visit=None)
    assert st == 0
    items = np.arange(w.num_items)
    check(w, got, 0.25, 8, items=items)
    host = w.visit_order.reshape(w.num_items, -1)
    same = sum(int(np.array_equal(got[i][got[i] >= 0], host[i][host[i] >= 0])) for i in items)
    assert same >= w.num_items - 1, f"{same} of {w.num_items} lists equal"
    assert mv >= (got >= 0).sum(axis=1).max()


def test_select_edge_cases():
    w = W.build("select-edges", seed=71, dtype="bf16", batch=4, num_q_heads=8, num_kv_heads=2, head_dim=128,
                page_size=16, block_size=64, seq_lens=[0, 1, 65, 1000], paged="permuted", order=None)
    got, st = run_select(w, 0.3, 2)
    assert st == 0
    assert (got[0] == -1).all() and (got[1] == -1).all()        # seq_len 0: empty lists
    assert list(got[2][got[2] >= 0]) == [0] and list(got[3][got[3] >= 0]) == [0]  # one block
    check(w, got, 0.3, 2)
    # a page id outside the pool: that sequence's items get empty lists and a status bit
    w.block_table = w.block_table.copy()
    w.block_table[3, 5] = w.num_pages_total + 3
    got, st = run_select(w, 0.3, 2)
    assert "bad page id" in K.status_names(st)
    assert (got[6] == -1).all() and (got[7] == -1).all()
    check(w, got, 0.3, 2, items=[4, 5])


def test_select_then_decode_matches_host_lists():
    """ART over the device-selected lists equals ART over the host lists."""
    w = W.config(5, small=True)
    got, st = run_select(w, 0.25, 8)
    assert st == 0
    mv = w.visit_order.shape[-1]
    assert (got[:, mv:] == -1).all()
    got = np.ascontiguousarray(got[:, :mv])
    if not np.array_equal(got.reshape(w.visit_order.shape), w.visit_order):
        pytest.skip("a tie at the cut changed a list")
    dev = K.DeviceInputs(w)
    dev.art(1e-2, 1e-2, 2)
    torch.cuda.synchronize()
    a_out, a_bu = dev.out.float().cpu().numpy(), dev.blocks_used.cpu().numpy()
    dev.visit_order.copy_(torch.from_numpy(got.reshape(w.visit_order.shape)).cuda())
    dev.art(1e-2, 1e-2, 2)
    torch.cuda.synchronize()
    assert np.array_equal(dev.blocks_used.cpu().numpy(), a_bu)
    assert np.array_equal(dev.out.float().cpu().numpy(), a_out)


@pytest.mark.parametrize("k", [2, 4, 5])
def test_select_importance_order(k):
    """Order 1: block 0, then the kept blocks by descending score. Same kept set
    as order 0 (up to ties at the cut); the sequence must descend in the
    oracle's scores up to the tie tolerance."""
    w = W.config(k, small=True)
    got0, st0 = run_select(w, 0.25, 8)
    got1, st1 = run_select(w, 0.25, 8, order=1)
    assert st0 == 0 and st1 == 0
    ref = S.select_blocks(w, 0.25, 8, order="importance")
    for it, (lst, sc) in ref.items():
        d0 = [int(x) for x in got0[it] if x >= 0]
        d1 = [int(x) for x in got1[it] if x >= 0]
        assert sorted(d0) == sorted(d1), f"item {it}: kept sets differ between orders"
        if d1 == lst:
            continue
        assert d1[0] == 0
        scale = max(float(np.abs(sc).mean()), 1e-30)
        for a, b in zip(d1[1:], d1[2:]):
            assert sc[a] >= sc[b] - TIE_REL * scale, f"item {it}: {a} before {b}"
