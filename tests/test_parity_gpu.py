"""GPU parity: libart (through the C ABI) against the CPU oracle.

Small versions of the five decode workloads at sizes the oracle finishes in
seconds (several 64-token blocks, ragged tails, paged tables, GQA 1/4/7),
sweeps of the thresholds and patience, the edge cases (empty lists, zero
lengths, single blocks, bad device data), and the full-size workloads on
sampled items in the benchmark's launch configuration.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_harness import check_art, check_dense, compare, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS_SWEEP = [0.0, 1e-3, 1e-2, 5e-2]


@pytest.fixture(autouse=True, params=["one-cta", "units"])
def decode_path(request, monkeypatch):
    """Every test runs on both bf16 paths: one CTA per item, and the unit path
    (an item's list cut into units spread over many CTAs; fp32 and calls with
    more than 256 items always take the first)."""
    monkeypatch.setenv("ART_UNITS", "1" if request.param == "units" else "0")
    return request.param


@pytest.fixture(scope="module")
def small():
    return {k: W.config(k, small=True) for k in (1, 2, 3, 4, 5)}


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_dense_small(small, k):
    w = small[k]
    out, _, st, _ = run_gpu(w, "dense")
    assert st == 0
    check_dense(w, out, what=f"dense config {k}")


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("eps", EPS_SWEEP)
@pytest.mark.parametrize("patience", [1, 2])
def test_art_small(small, k, eps, patience):
    w = small[k]
    out, bu, st, _ = run_gpu(w, "art", eps, eps, patience)
    assert st == 0
    res = check_art(w, out, bu, eps, eps, patience, what=f"art config {k} eps {eps} p {patience}")
    if eps == 0.0:
        assert (bu == w.visit_lengths()).all()
    print(res)


def test_art_grid_ragged(small):
    """The threshold x patience grid of the ragged workload."""
    w = small[4]
    for eps, p in W.CONFIG4_GRID:
        out, bu, st, _ = run_gpu(w, "art", eps, eps, p)
        assert st == 0
        check_art(w, out, bu, eps, eps, p, what=f"grid eps {eps} p {p}")


def test_eps_zero_equals_dense(small, decode_path):
    w = small[2]
    dev = None
    out_d, _, _, dev = run_gpu(w, "dense")
    out_a, bu, st, _ = run_gpu(w, "art", 0.0, 0.0, 1, dev=dev)
    assert st == 0 and (bu == w.visit_lengths()).all()
    # eps = 0 never stops, so on either path ART folds the same blocks in the same
    # order with the same arithmetic as the dense twin (unit path: the same units,
    # merged the same way): the outputs are bit-identical
    np.testing.assert_array_equal(out_a, out_d)


def test_monotone_in_thresholds_and_patience(small):
    w = small[4]
    dev = None
    prev = None
    for eps in (1e-3, 3e-3, 1e-2, 3e-2, 0.1, 1.0):
        _, bu, _, dev = run_gpu(w, "art", eps, eps, 2, dev=dev)
        if prev is not None:
            assert (bu <= prev).all()
        prev = bu
    prev = None
    for p in (1, 2, 3, 5):
        _, bu, _, dev = run_gpu(w, "art", 0.05, 0.05, p, dev=dev)
        assert (bu >= np.minimum(w.visit_lengths(), p + 1)).all()
        if prev is not None:
            assert (bu >= prev).all()
        prev = bu


def test_one_statistic_disabled(small):
    w = small[2]
    for em, ed in ((np.inf, 1e-2), (1e-2, np.inf), (np.inf, np.inf)):
        out, bu, st, _ = run_gpu(w, "art", em, ed, 2)
        assert st == 0
        check_art(w, out, bu, em, ed, 2, what=f"eps ({em}, {ed})")


@pytest.mark.parametrize("order", ["natural", "reverse", "random", "sink_recent"])
def test_visit_orders(order):
    w = W.build(f"orders-{order}", seed=21, dtype="bf16", batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                page_size=16, block_size=64, seq_lens=[700, 1000, 333], paged="permuted", plant=True, order=order)
    for eps, p in ((0.0, 1), (2e-2, 1), (2e-2, 2)):
        out, bu, st, _ = run_gpu(w, "art", eps, eps, p)
        assert st == 0
        check_art(w, out, bu, eps, eps, p, what=f"order {order}")


SHAPES = [
    # dtype, d, Hq, Hkv, page, seq_lens, order
    ("bf16", 128, 8, 8, 16, [1, 63, 64, 65, 1000], "sink_recent"),       # G = 1
    ("bf16", 128, 8, 4, 32, [130, 77, 900], "random"),                  # G = 2
    ("bf16", 128, 16, 2, 8, [257, 640], "natural"),                     # G = 8, 8 pages per block
    ("bf16", 128, 14, 2, 64, [515, 2048], "sink_recent"),               # G = 7
    ("bf16", 128, 8, 2, 128, [300, 129, 1000], "sink_recent"),          # page larger than a block
    ("bf16", 128, 8, 2, 256, [1000, 17], None),                         # natural order via NULL list
    ("bf16", 64, 8, 2, 16, [333, 800], "sink_recent"),                  # 128-byte rows
    ("f32", 64, 4, 1, 64, [1024, 100], "natural"),                      # 256-byte rows
    ("f32", 128, 8, 2, 16, [500, 64], "random"),                        # 512-byte rows
    ("f32", 64, 2, 2, 16, [70], None),
]


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: f"{s[0]}-d{s[1]}-G{s[2] // s[3]}-ps{s[4]}")
def test_shapes(spec):
    dt, d, hq, hkv, ps, lens, order = spec
    w = W.build("shape", seed=31, dtype=dt, batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                page_size=ps, block_size=64, seq_lens=lens, paged="permuted", order=order)
    out, _, st, dev = run_gpu(w, "dense")
    assert st == 0
    check_dense(w, out, what=f"dense {spec}")
    for eps, p in ((0.0, 1), (1e-2, 1), (5e-2, 2)):
        out, bu, st, _ = run_gpu(w, "art", eps, eps, p, dev=dev)
        assert st == 0
        check_art(w, out, bu, eps, eps, p, what=f"art {spec} eps {eps}")


@pytest.mark.parametrize("p", [1, 2, 4, 16, 17])
def test_long_lists(p):
    """Lists of 141 and 235 blocks (9 to 30 units of 8 to 16 blocks on the unit
    path), stops anywhere in a unit, patience up to the longest unit and past it
    (where the unit path is not taken)."""
    w = W.build("long", seed=51, dtype="bf16", batch=2, num_q_heads=14, num_kv_heads=2, head_dim=128,
                page_size=16, block_size=64, seq_lens=[15000, 9000], paged="permuted", plant=True,
                order="sink_recent")
    for eps in (0.0, 1e-3, 1e-2, 5e-2):
        out, bu, st, _ = run_gpu(w, "art", eps, eps, p)
        assert st == 0
        check_art(w, out, bu, eps, eps, p, what=f"long lists eps {eps} p {p}")


def test_empty_and_zero_lengths():
    w = W.build("empty", seed=41, dtype="bf16", batch=4, num_q_heads=8, num_kv_heads=2, head_dim=128,
                page_size=16, block_size=64, seq_lens=[0, 200, 0, 64], paged="permuted", order="sink_recent")
    w.visit_order[1, 1, :] = -1  # an empty list for a non-empty sequence
    for mode in ("dense", "art"):
        out, bu, st, _ = run_gpu(w, mode, 1e-2, 1e-2, 1)
        assert st == 0
        if mode == "art":
            res = check_art(w, out, bu, 1e-2, 1e-2, 1)
            assert list(bu[[0, 1, 3, 4, 5]]) == [0, 0, 0, 0, 0]
        else:
            check_dense(w, out)
        assert np.abs(out[[0, 1, 3, 4, 5]]).max() == 0.0


def test_bad_device_data_is_reported_not_faulted():
    import kv_cache_early_gb300 as K
    w = W.build("bad", seed=51, dtype="bf16", batch=4, num_q_heads=8, num_kv_heads=2, head_dim=128,
                page_size=16, block_size=64, seq_lens=[300, 300, 300, 300], paged="permuted", order="sink_recent")
    T = 5
    w.visit_order[0, 0, 2] = T          # past the end
    w.visit_order[0, 1, 3] = w.visit_order[0, 1, 1]  # duplicate
    w.block_table[2, 1] = w.num_pages_total + 5      # page out of the pool (seq 2, both heads)
    w.seq_lens = w.seq_lens.copy()
    w.seq_lens[3] = w.max_pages_per_seq * w.page_size + 1  # longer than its table row
    out, bu, st, _ = run_gpu(w, "art", 1e-2, 1e-2, 1)
    bits = set(K.status_names(st))
    assert {"bad visit entry", "duplicate visit entry", "bad page id", "bad seq_len"} <= bits, bits
    assert list(bu) == [-1, -1, bu[2], bu[3], -1, -1, -1, -1]
    assert np.abs(out[[0, 1, 4, 5, 6, 7]]).max() == 0.0
    # the good items are still right
    check_art(w, out, bu, 1e-2, 1e-2, 1, items=[2, 3])
    # a repeated probe index poisons every item
    w2 = W.config(2, small=True)
    w2.probe_idx = w2.probe_idx.copy()
    w2.probe_idx[3] = w2.probe_idx[2]
    out, bu, st, _ = run_gpu(w2, "art", 1e-2, 1e-2, 1)
    assert "bad probe index" in K.status_names(st) and (bu == -1).all()


def test_repeated_calls_reuse_workspace(small):
    w = small[3]
    out1, bu1, st1, dev = run_gpu(w, "art", 1e-2, 1e-2, 2)
    out2, bu2, st2, _ = run_gpu(w, "art", 1e-2, 1e-2, 2, dev=dev)
    assert st1 == st2 == 0
    assert (bu1 == bu2).all()
    assert np.array_equal(out1, out2)


def test_side_stream(small):
    w = small[2]
    import kv_cache_early_gb300 as K
    dev = K.DeviceInputs(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dev.art(1e-2, 1e-2, 2, stream=s)
    s.synchronize()
    out = dev.out.float().cpu().numpy().reshape(w.num_items, w.group, w.head_dim)
    check_art(w, out, dev.blocks_used.cpu().numpy().reshape(-1), 1e-2, 1e-2, 2)


# ---------------------------------------------------------------------------
# full-size workloads, sampled items (the launch configuration bench.py times)
# ---------------------------------------------------------------------------
# the benchmark settings of every workload, and the ragged workload's whole threshold x
# patience grid; every item of the Llama-shaped and long-context workloads, 64 sampled
# items of the paged and ragged ones
FULL = [(2, 1e-3, 2), (3, 1e-3, 2)] + [(4, e, p) for e, p in W.CONFIG4_GRID] + [(5, 1e-3, 2), (1, 1e-3, 2)]
FULL_SAMPLE = {1: None, 2: None, 3: 64, 4: 64, 5: None}


@pytest.fixture(scope="module")
def full_cache():
    return {}


@pytest.mark.parametrize("k,eps,p", FULL, ids=lambda x: str(x))
def test_full_size_sampled(full_cache, k, eps, p):
    if k not in full_cache:
        full_cache.clear()
        full_cache[k] = W.config(k)
    w = full_cache[k]
    rng = np.random.default_rng(k)
    size = FULL_SAMPLE[k] or w.num_items
    items = np.sort(rng.choice(w.num_items, size=min(w.num_items, size), replace=False))
    out, bu, st, dev = run_gpu(w, "art", eps, eps, p)
    assert st == 0
    res = check_art(w, out, bu, eps, eps, p, items=items, what=f"full config {k}")
    print(f"config {k}: {res}")
    outd, _, st, _ = run_gpu(w, "dense", dev=dev)
    assert st == 0
    check_dense(w, outd, items=items, what=f"full dense config {k}")


@pytest.mark.parametrize("groups", ["1", "2", "3", "4"])
@pytest.mark.parametrize("k", [2, 3, 4, 5])
def test_consumer_group_variants(small, k, groups, monkeypatch):
    """Each bf16 kernel variant (one to four consumer groups per CTA; the
    library picks one from the item count, ART_GROUPS forces it) against the
    oracle, ART and dense."""
    monkeypatch.setenv("ART_GROUPS", groups)
    w = small[k]
    out, bu, st, dev = run_gpu(w, "art", 1e-2, 1e-2, 2)
    assert st == 0
    check_art(w, out, bu, 1e-2, 1e-2, 2, what=f"art config {k} groups {groups}")
    out, bu, st, _ = run_gpu(w, "art", 0.0, 0.0, 1, dev=dev)
    assert st == 0 and (bu == w.visit_lengths()).all()
    out, _, st, _ = run_gpu(w, "dense", dev=dev)
    assert st == 0
    check_dense(w, out, what=f"dense config {k} groups {groups}")


@pytest.mark.parametrize("groups,stages", [("3", "2"), ("3", "3"), ("3", "5"), ("4", "3"), ("2", "3")])
def test_ring_depths(small, groups, stages, monkeypatch):
    """Shallow and odd ring depths (ART_STAGES): the library raises the depth to
    one slot per consumer group (at an item's end every group merges while holding
    its first entry of the next item) and, with two copy warps (three groups),
    rounds it to an even count so that each slot's entries stay with one copy
    warp. Every depth must give the oracle's result, ART and dense, over repeated
    calls."""
    monkeypatch.setenv("ART_GROUPS", groups)
    monkeypatch.setenv("ART_STAGES", stages)
    monkeypatch.setenv("ART_UNITS", "0")
    w = small[4]
    dev = None
    for _ in range(2):
        out, bu, st, dev = run_gpu(w, "art", 1e-2, 1e-2, 2, dev=dev)
        assert st == 0
        check_art(w, out, bu, 1e-2, 1e-2, 2, what=f"ring depth {stages}, groups {groups}")
    out, _, st, _ = run_gpu(w, "dense", dev=dev)
    assert st == 0
    check_dense(w, out, what=f"dense, ring depth {stages}, groups {groups}")


@pytest.mark.parametrize("groups", ["2", "3", "4"])
def test_many_short_items_multi_group(groups, monkeypatch):
    """Hundreds of short items per call: with several consumer groups the ring
    slots change hands between groups at every item, and blocks of different
    groups land out of order. Repeated calls must all finish cleanly (status 0)
    and match the oracle."""
    monkeypatch.setenv("ART_GROUPS", groups)
    rs = np.random.default_rng(77)
    lens = rs.integers(1, 1500, size=64)
    w = W.build("short-items", seed=61, dtype="bf16", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
                page_size=16, block_size=64, seq_lens=list(lens), paged="permuted", plant=True,
                order="sink_recent")
    items = np.sort(rs.choice(w.num_items, size=48, replace=False))
    dev = None
    for call in range(3):
        out, bu, st, dev = run_gpu(w, "dense", dev=dev)
        assert st == 0, f"dense call {call}: status {st}"
        out, bu, st, dev = run_gpu(w, "art", 1e-2, 1e-2, 1, dev=dev)
        assert st == 0, f"art call {call}: status {st}"
    check_art(w, out, bu, 1e-2, 1e-2, 1, items=items, what=f"short items, groups {groups}")
    out, _, st, _ = run_gpu(w, "dense", dev=dev)
    check_dense(w, out, items=items, what=f"short items dense, groups {groups}")


@pytest.mark.parametrize("k", [2, 3, 4])
def test_two_d_copies(small, k, monkeypatch):
    """The bf16 kernels with one 2-D copy per 128-byte column half of each page
    (the fallback when the 3-D tensor view is not accepted; ART_TMA3D=0 forces
    it) against the oracle."""
    monkeypatch.setenv("ART_TMA3D", "0")
    w = small[k]
    out, bu, st, dev = run_gpu(w, "art", 1e-2, 1e-2, 2)
    assert st == 0
    check_art(w, out, bu, 1e-2, 1e-2, 2, what=f"2-D copies, config {k}")
    out, _, st, _ = run_gpu(w, "dense", dev=dev)
    assert st == 0
    check_dense(w, out, what=f"2-D copies dense, config {k}")


def _random_case(seed):
    rs = np.random.default_rng(np.random.SeedSequence([97, seed]))
    dt = "bf16" if rs.random() < 0.75 else "f32"
    d = int(rs.choice([64, 128]))
    G = int(rs.choice([1, 2, 4, 7, 8]))
    hkv = int(rs.integers(1, 4))
    B = int(rs.integers(1, 5))
    ps = int(rs.choice([8, 16, 32, 64, 128, 256]))
    lens = [int(x) for x in rs.integers(0, 2500, size=B)]
    order = rs.choice(["natural", "reverse", "random", "sink_recent", "none"])
    eps = float(rs.choice([0.0, 1e-3, 1e-2, 5e-2]))
    p = int(rs.integers(1, 5))
    groups = str(int(rs.integers(1, 5)))
    plant = bool(rs.random() < 0.5)
    w = W.build(f"random-{seed}", seed=1000 + seed, dtype=dt, batch=B, num_q_heads=G * hkv, num_kv_heads=hkv,
                head_dim=d, page_size=ps, block_size=64, seq_lens=lens, paged="permuted", plant=plant,
                order=None if order == "none" else str(order))
    return w, eps, p, groups


@pytest.mark.parametrize("seed", range(40))
def test_random_shapes(seed, monkeypatch):
    """Seeded random shapes, page sizes, lengths (empty included), orders,
    thresholds, patience and kernel variants against the oracle."""
    w, eps, p, groups = _random_case(seed)
    monkeypatch.setenv("ART_GROUPS", groups)
    out, bu, st, dev = run_gpu(w, "art", eps, eps, p)
    assert st == 0
    check_art(w, out, bu, eps, eps, p, what=f"random case {seed}")
    out, _, st, _ = run_gpu(w, "dense", dev=dev)
    assert st == 0
    check_dense(w, out, what=f"random case {seed} dense")


@pytest.mark.parametrize("k", [2, 3, 5])
def test_probe_heads_option(small, k, monkeypatch):
    """art_decode_ex with the probe formed by the first 1, 2 or G query heads of
    each group, against the oracle with the same option, for the kernel
    variants (one and three consumer groups)."""
    import kv_cache_early_gb300 as K
    w = small[k]
    for groups in ("1", "3"):
        monkeypatch.setenv("ART_GROUPS", groups)
        for ph in sorted({1, 2, w.group}):
            dev = K.DeviceInputs(w)
            dev.blocks_used.fill_(-7)
            dev.art(1e-2, 1e-2, 2, probe_heads=ph)
            torch.cuda.synchronize()
            assert dev.status() == 0
            out = dev.out.float().cpu().numpy().reshape(w.num_items, w.group, w.head_dim)
            bu = dev.blocks_used.cpu().numpy().reshape(-1)
            check_art(w, out, bu, 1e-2, 1e-2, 2, what=f"probe heads {ph}, groups {groups}", probe_heads=ph)


@pytest.mark.parametrize("k", [2, 4, 5])
def test_probe_every_head_dim(small, k):
    """A probe over every head dim (num_probe = head_dim, the full-d ablation): bf16
    calls run one CTA per item with the head dims split between the four warps of a
    group (one writer per probe column), against the oracle with the same probe."""
    import dataclasses
    w0 = small[k]
    w = dataclasses.replace(w0, probe_idx=np.arange(w0.head_dim, dtype=np.int32))
    for eps, p in ((1e-2, 2), (1e-3, 1), (0.0, 1)):
        out, bu, st, _ = run_gpu(w, "art", eps, eps, p)
        assert st == 0
        res = check_art(w, out, bu, eps, eps, p, what=f"full-d probe, config {k}, eps {eps}, p {p}")
        if eps == 0.0:
            assert (bu == w.visit_lengths()).all()
        print(res)


@pytest.mark.parametrize("d,G", [(64, 8), (128, 1), (64, 2)])
def test_probe_every_head_dim_shapes(d, G):
    """The full-d probe on other head dims and group sizes (permuted 16-token pages,
    ragged lengths)."""
    w = W.build(f"fullprobe-d{d}-g{G}", seed=55 + d + G, dtype="bf16", batch=2, num_q_heads=2 * G, num_kv_heads=2,
                head_dim=d, page_size=16, block_size=64, seq_lens=[1500, 777], paged="permuted", plant=True,
                order="sink_recent", probe_stride=1)
    assert w.num_probe == d
    for eps, p in ((1e-2, 2), (3e-2, 1)):
        out, bu, st, _ = run_gpu(w, "art", eps, eps, p)
        assert st == 0
        check_art(w, out, bu, eps, eps, p, what=f"full-d probe d {d} G {G}")
