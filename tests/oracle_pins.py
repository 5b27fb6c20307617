"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Every function takes an oracle build (`oracle.Oracle`) and raises
AssertionError when that build disagrees with a fact that does not come from
the oracle itself:

* Eq. (1) of the ART paper (sec. 3.1) evaluated directly -- a softmax over the
  gathered token rows -- on tiny inputs (brute force);
* a hand-derived closed-form case for the two statistics, the patience counter
  and the block-0 gate (tests/golden/stat_closed_form.json);
* closed forms of attention (constant value rows give that row; identical keys
  give the mean of the values);
* invariants: eps = 0 never terminates (strict comparison) and equals full
  attention; blocks_used is monotone in each threshold and in patience and is at
  least min(n, patience + 1); reordering blocks leaves full attention unchanged
  (gist.science explainer sec. 2.4, permutation invariance); scaling V leaves
  the statistics unchanged;
* the exact subset-error bound of the FlexPrefill appendix A (the difference
  between full attention and attention restricted to a subset S is bounded by
  sum_{j not in S} a_j |v_j| + (1/a_S - 1) sum_{j in S} a_j |v_j|).

The same functions run against deliberately broken builds of the oracle in
test_oracle_mutants.py, to show that each plausible mistake fails a pin.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# independent helpers (no oracle code)
# ----------------------------------------------------------------------------
def gathered_rows(w, b, g, blocks):
    """K and V rows (fp64) of the tokens of logical `blocks` of item (b, g), in list order."""
    N = int(w.seq_lens[b])
    Ks, Vs = [], []
    for c in blocks:
        for t in range(c * w.block_size, min((c + 1) * w.block_size, N)):
            page = int(w.block_table[b, t // w.page_size])
            Ks.append(W.as_f32(w.k_cache[page, g, t % w.page_size], w.dtype))
            Vs.append(W.as_f32(w.v_cache[page, g, t % w.page_size], w.dtype))
    d = w.head_dim
    K = np.array(Ks, dtype=np.float64).reshape(-1, d)
    V = np.array(Vs, dtype=np.float64).reshape(-1, d)
    return K, V


def softmax_weights(w, b, g, K):
    """Softmax weights a[h, t] of Eq. (1) for the q heads of group g."""
    G, d = w.group, w.head_dim
    A = []
    for h in range(G):
        qh = W.as_f32(w.q[b, g * G + h], w.dtype).astype(np.float64)
        s = K @ qh / np.sqrt(d)
        e = np.exp(s - s.max())
        A.append(e / e.sum())
    return np.array(A)


def brute_attention(w, b, g, blocks):
    K, V = gathered_rows(w, b, g, blocks)
    if K.shape[0] == 0:
        return np.zeros((w.group, w.head_dim))
    return softmax_weights(w, b, g, K) @ V


def listed(w, item):
    b, g = divmod(item, w.num_kv_heads)
    if w.visit_order is None:
        return list(range(-(-int(w.seq_lens[b]) // w.block_size)))
    row = w.visit_order[b, g]
    out = []
    for c in row:
        if c == -1:
            break
        out.append(int(c))
    return out


def tiny(dtype="f32", order="random", seed=11, **kw):
    args = dict(seed=seed, dtype=dtype, batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8,
                page_size=4, block_size=8, seq_lens=[37, 21], paged="permuted", order=order,
                threads=1)
    args.update(kw)
    return W.build("pin-tiny", **args)


def close(a, b, tol=1e-12, what=""):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    scale = max(1.0, float(np.abs(b).max(initial=0.0)))
    err = float(np.abs(a - b).max(initial=0.0))
    assert err <= tol * scale, f"{what}: max abs error {err:.3e} > {tol:.1e} * {scale:.3g}"


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------
def pin_brute_force_tiny(orc):
    """Dense output and forced prefixes equal direct softmax attention (Eq. 1),
    through a permuted page table, ragged tails and GQA (G = 2)."""
    for dtype in ("f32", "bf16"):
        w = tiny(dtype)
        r = O.run_workload(w, mode="dense", orc=orc)
        assert (r["status"] == 0).all()
        for it in range(w.num_items):
            b, g = divmod(it, w.num_kv_heads)
            L = listed(w, it)
            assert r["blocks_used"][it] == len(L)
            close(r["out"][it], brute_attention(w, b, g, L), what=f"dense item {it} {dtype}")
            for k in sorted({1, 2, len(L) - 1, len(L)}):
                if k < 1:
                    continue
                rf = O.run_workload(w, mode="forced", items=[it], forced=[k], orc=orc)
                assert rf["blocks_used"][0] == k
                close(rf["out"][0], brute_attention(w, b, g, L[:k]), what=f"prefix {k} item {it}")


def _closed_form_workload(fx, order_name, G):
    d, Ps, Bk = fx["head_dim"], fx["page_size"], fx["block_size"]
    L = fx["orders"][order_name]
    vals = fx["block_probe_values"]
    nblk = len(vals)
    N = nblk * Bk
    Hkv = 1
    k_cache = np.zeros((N // Ps, Hkv, Ps, d), np.float32)
    v_cache = np.zeros_like(k_cache)
    other = fx["other_columns"]
    for pos, c in enumerate(L):
        for t in range(c * Bk, (c + 1) * Bk):
            row = np.zeros(d, np.float32)
            row[fx["probe_idx"][0]], row[fx["probe_idx"][1]] = vals[pos]
            for col, v in other.items():
                row[int(col)] = t if v == "token index t" else v
            v_cache[t // Ps, 0, t % Ps] = row
    table = np.arange(N // Ps, dtype=np.int32)[None, :]
    vo = np.full((1, 1, nblk), -1, np.int32)
    vo[0, 0, : len(L)] = L
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, G, d)).astype(np.float32)
    w = W.Workload(name="closed-form", dtype="f32", batch=1, num_q_heads=G, num_kv_heads=Hkv,
                   head_dim=d, page_size=Ps, block_size=Bk, seq_lens=np.array([N], np.int32),
                   block_table=table, visit_order=vo, q=q, k_cache=k_cache, v_cache=v_cache,
                   probe_idx=np.array(fx["probe_idx"], np.int32))
    return w, L


def pin_closed_form_statistics(orc):
    """Hand-derived statistic values, patience and block-0 outcomes."""
    with open(os.path.join(GOLDEN, "stat_closed_form.json")) as f:
        fx = json.load(f)
    for G in (1, 2):
        w, L = _closed_form_workload(fx, "natural", G)
        r = O.run_workload(w, eps_mag=0.0, eps_dir=0.0, patience=1, trace=True, orc=orc)
        em = [np.nan if x is None else x for x in fx["expected_d_mag"]]
        ed = [np.nan if x is None else x for x in fx["expected_d_dir"]]
        np.testing.assert_allclose(r["trace_mag"][0], em, rtol=0, atol=1e-15, equal_nan=True)
        np.testing.assert_allclose(r["trace_dir"][0], ed, rtol=0, atol=1e-15, equal_nan=True)
        # partial outputs: uniform weights, so O^(k) is the mean of the first 2k rows
        for k in range(1, len(L) + 1):
            rf = O.run_workload(w, mode="forced", forced=[k], orc=orc)
            K, V = gathered_rows(w, 0, 0, L[:k])
            exp = np.repeat(V.mean(axis=0)[None, :], G, axis=0)
            close(rf["out"][0], exp, tol=1e-14, what=f"closed-form O^({k})")
            close(rf["out"][0][0, fx["probe_idx"]], fx["expected_probe"][k - 1], tol=1e-14,
                  what=f"closed-form probe x^({k})")
        for case in fx["expected_blocks_used"]:
            wc, _ = _closed_form_workload(fx, case["order"], G)
            rc = O.run_workload(wc, eps_mag=case["eps_mag"], eps_dir=case["eps_dir"],
                                patience=case["patience"], orc=orc)
            assert rc["blocks_used"][0] == case["blocks_used"], (case, int(rc["blocks_used"][0]))


def pin_constant_values(orc):
    """Constant V rows: every partial output equals that row, so the statistics
    vanish: eps > 0 stops at min(n, p + 1), eps = 0 never stops."""
    c = np.array([3.0, -1.0, 0.5, 2.0, 4.0, 1.0, -2.0, 0.25], np.float32)
    for dtype in ("f32", "bf16"):
        w = tiny(dtype, order="natural", seed=3)
        w.v_cache[...] = W.to_working(c, dtype)
        n = w.visit_lengths()
        for p in (1, 2, 3):
            r = O.run_workload(w, eps_mag=1e-3, eps_dir=1e-3, patience=p, orc=orc)
            assert (r["blocks_used"] == np.minimum(n, p + 1)).all(), (p, r["blocks_used"], n)
            close(r["out"], np.broadcast_to(c, r["out"].shape), tol=1e-14, what="constant V")
        r0 = O.run_workload(w, eps_mag=0.0, eps_dir=0.0, patience=1, orc=orc)
        assert (r0["blocks_used"] == n).all()


def pin_exact_constant_values_eps_zero(orc):
    """Zero keys and V rows whose probe entries are (1, 7): every partial output
    is exactly that row, the probe of the G = 2 heads has norm exactly 10, both
    statistics are exactly 0, and with thresholds 0 the strict comparison never
    passes."""
    w = tiny("f32", order="natural", seed=4, head_dim=8)
    w.k_cache[...] = 0.0
    row = np.array([1, 3, 3, 3, 7, 3, 3, 3], np.float32)
    w.v_cache[...] = row
    r = O.run_workload(w, eps_mag=0.0, eps_dir=0.0, patience=1, trace=True, orc=orc)
    assert (r["blocks_used"] == w.visit_lengths()).all(), r["blocks_used"]
    tm, td = r["trace_mag"], r["trace_dir"]
    assert np.nanmax(np.abs(tm)) == 0.0 and np.nanmax(np.abs(td)) == 0.0


def pin_identical_keys(orc):
    """Identical keys: uniform weights, so O^(k) is the mean of the listed rows."""
    w = tiny("bf16", order="random", seed=5)
    w.k_cache[...] = w.k_cache[0, 0, 0]
    for it in range(w.num_items):
        b, g = divmod(it, w.num_kv_heads)
        L = listed(w, it)
        for k in (1, len(L) // 2 + 1, len(L)):
            r = O.run_workload(w, mode="forced", items=[it], forced=[k], orc=orc)
            _, V = gathered_rows(w, b, g, L[:k])
            close(r["out"][0], np.repeat(V.mean(axis=0)[None], w.group, axis=0), what="mean of V")


def pin_eps_zero_is_dense(orc):
    w = W.config(2, small=True)
    r = O.run_workload(w, eps_mag=0.0, eps_dir=0.0, patience=1, orc=orc)
    rd = O.run_workload(w, mode="dense", orc=orc)
    assert (r["blocks_used"] == w.visit_lengths()).all()
    close(r["out"], rd["out"], tol=1e-15, what="eps=0 vs dense")
    # and dense equals direct attention on a few items
    for it in (0, w.num_items - 1):
        b, g = divmod(it, w.num_kv_heads)
        close(rd["out"][it], brute_attention(w, b, g, listed(w, it)), tol=1e-11, what="dense vs Eq.1")


def pin_monotone(orc):
    w = W.config(2, small=True)
    n = w.visit_lengths()
    prev = None
    for e in (1e-3, 3e-3, 1e-2, 3e-2, 0.1, 0.3, 1.0):
        bu = O.run_workload(w, eps_mag=e, eps_dir=e, patience=2, orc=orc)["blocks_used"]
        assert (bu >= np.minimum(n, 3)).all()
        if prev is not None:
            assert (bu <= prev).all(), ("not monotone in eps", e)
        prev = bu
    for which in ("mag", "dir"):
        prev = None
        for e in (1e-3, 1e-2, 0.1, 1.0, np.inf):
            kw = dict(eps_mag=e, eps_dir=0.05) if which == "mag" else dict(eps_mag=0.05, eps_dir=e)
            bu = O.run_workload(w, patience=1, orc=orc, **kw)["blocks_used"]
            if prev is not None:
                assert (bu <= prev).all(), ("not monotone in eps_" + which, e)
            prev = bu
    prev = None
    for p in (1, 2, 3, 4, 6):
        bu = O.run_workload(w, eps_mag=0.05, eps_dir=0.05, patience=p, orc=orc)["blocks_used"]
        assert (bu >= np.minimum(n, p + 1)).all()
        if prev is not None:
            assert (bu >= prev).all(), ("not monotone in patience", p)
        prev = bu


def pin_infinite_thresholds(orc):
    """eps = +inf: every step with finite statistics is stable, so the stop
    comes at p + 1 once block 0 (listed first) has been processed."""
    w = tiny("bf16", order="sink_recent", seed=6)
    n = w.visit_lengths()
    for p in (1, 2):
        r = O.run_workload(w, eps_mag=np.inf, eps_dir=np.inf, patience=p, orc=orc)
        assert (r["blocks_used"] == np.minimum(n, p + 1)).all()


def pin_block0_gate(orc):
    c = np.linspace(-1, 1, 8).astype(np.float32)
    w = tiny("f32", order="reverse", seed=7)
    w.v_cache[...] = c
    n = w.visit_lengths()
    r = O.run_workload(w, eps_mag=1e-3, eps_dir=1e-3, patience=1, orc=orc)
    assert (r["blocks_used"] == n).all(), "stopped before block 0 (listed last)"
    # remove block 0 from every list: the gate no longer applies
    vo = w.visit_order.copy()
    for b in range(w.batch):
        for g in range(w.num_kv_heads):
            row = [x for x in vo[b, g] if x not in (0, -1)]
            vo[b, g] = -1
            vo[b, g, : len(row)] = row
    r2 = O.run_workload(w, eps_mag=1e-3, eps_dir=1e-3, patience=1, visit_order=vo, orc=orc)
    assert (r2["blocks_used"] == np.minimum(n - 1, 2)).all()


def pin_permutation_invariance(orc):
    outs = []
    for order in ("natural", "reverse", "random", "sink_recent"):
        w = tiny("bf16", order=order, seed=8)
        outs.append(O.run_workload(w, eps_mag=0.0, eps_dir=0.0, patience=1, orc=orc)["out"])
    for o in outs[1:]:
        close(o, outs[0], tol=1e-12, what="permutation invariance")


def pin_subset_bound(orc):
    """Truncated outputs obey the exact subset bound of FlexPrefill appendix A."""
    w = W.config(4, small=True)
    rng = np.random.default_rng(9)
    items = list(range(0, w.num_items, 3))
    n = w.visit_lengths()
    forced = [int(rng.integers(1, n[i] + 1)) for i in items]
    r = O.run_workload(w, mode="forced", items=items, forced=forced, orc=orc)
    rd = O.run_workload(w, mode="dense", items=items, orc=orc)
    for k, it in enumerate(items):
        b, g = divmod(it, w.num_kv_heads)
        L = listed(w, it)
        K, V = gathered_rows(w, b, g, L)
        A = softmax_weights(w, b, g, K)
        nS = sum(w.block_tokens(b, c) for c in L[: forced[k]])
        aS = A[:, :nS].sum(axis=1, keepdims=True)
        bound = A[:, nS:] @ np.abs(V[nS:]) + (1.0 / aS - 1.0) * (A[:, :nS] @ np.abs(V[:nS]))
        diff = np.abs(rd["out"][k] - r["out"][k])
        assert (diff <= bound + 1e-12).all(), f"subset bound violated on item {it}"
        assert (bound <= (1 - aS) * np.abs(V).sum(axis=0) + 1e-9).all()


def pin_scale_invariance(orc):
    w = tiny("f32", order="sink_recent", seed=10)
    r1 = O.run_workload(w, eps_mag=1e-2, eps_dir=1e-2, patience=1, trace=True, orc=orc)
    w.v_cache *= 2.0
    r2 = O.run_workload(w, eps_mag=1e-2, eps_dir=1e-2, patience=1, trace=True, orc=orc)
    np.testing.assert_allclose(r2["trace_mag"], r1["trace_mag"], rtol=1e-12, atol=1e-15, equal_nan=True)
    np.testing.assert_allclose(r2["trace_dir"], r1["trace_dir"], rtol=1e-9, atol=1e-15, equal_nan=True)
    assert (r1["blocks_used"] == r2["blocks_used"]).all()
    close(r2["out"], 2 * r1["out"], what="V scaling")


def pin_bf16_equals_f32(orc):
    """bf16 inputs are read exactly: the same values given as fp32 give the same result."""
    wb = tiny("bf16", order="random", seed=12)
    wf = tiny("bf16", order="random", seed=12)
    wf.dtype = "f32"
    wf.q, wf.k_cache, wf.v_cache = (W.bf16_bits_to_f32(x) for x in (wb.q, wb.k_cache, wb.v_cache))
    a = O.run_workload(wb, eps_mag=1e-2, eps_dir=1e-2, trace=True, orc=orc)
    b = O.run_workload(wf, eps_mag=1e-2, eps_dir=1e-2, trace=True, orc=orc)
    assert (a["blocks_used"] == b["blocks_used"]).all()
    assert np.array_equal(a["out"], b["out"])


def pin_item_errors_and_empty(orc):
    w = tiny("f32", order="natural", seed=13)
    T0 = -(-int(w.seq_lens[0]) // w.block_size)
    vo = w.visit_order.copy()
    vo[0, 0, 1] = T0          # past the end
    vo[0, 1, 2] = vo[0, 1, 0]  # duplicate
    r = O.run_workload(w, visit_order=vo, orc=orc)
    assert r["status"][0] == 1 and r["blocks_used"][0] == -1
    assert r["status"][1] == 3 and r["blocks_used"][1] == -1
    assert (r["status"][2:] == 0).all()
    bt = w.block_table.copy()
    w.block_table = bt
    bt[1, 0] = w.num_pages_total  # out of the pool
    r = O.run_workload(w, orc=orc)
    assert (r["status"][2:] == 2).all() and (r["blocks_used"][2:] == -1).all()
    # empty: seq_len 0, and an empty list
    w2 = tiny("f32", order="natural", seed=14, seq_lens=[0, 21])
    vo2 = w2.visit_order.copy()
    vo2[1, 1] = -1
    r = O.run_workload(w2, visit_order=vo2, orc=orc)
    assert list(r["blocks_used"]) == [0, 0, r["blocks_used"][2], 0]
    assert np.abs(r["out"][[0, 1, 3]]).max() == 0.0


ALL_PINS = [pin_brute_force_tiny, pin_closed_form_statistics, pin_constant_values,
            pin_exact_constant_values_eps_zero, pin_identical_keys, pin_eps_zero_is_dense,
            pin_monotone, pin_infinite_thresholds, pin_block0_gate, pin_permutation_invariance,
            pin_subset_bound, pin_scale_invariance, pin_bf16_equals_f32, pin_item_errors_and_empty]
