"""Pins of the oracle's probe-heads option (the probe formed by the first
`probe_heads` query heads of each group instead of all G; the ART paper's
probe is a fragment of one head's output, sec. 3.2), CPU only.

* probe_heads = G is the default probe;
* a group whose G query vectors are all equal has G equal head outputs, so the
  probe over any number of them has the same relative magnitude change and
  the same cosine: identical decisions and statistics for every probe_heads;
* probe_heads = 1 on a G-head workload decides like the G = 1 workload built
  from each group's first query head with the same keys and values.
"""
import dataclasses

import numpy as np
import pytest

import oracle as O
import workloads as W


def _work(G=4):
    return W.build("probe-heads", seed=81, dtype="bf16", batch=3, num_q_heads=2 * G, num_kv_heads=2, head_dim=64,
                   page_size=16, block_size=64, seq_lens=[900, 1700, 333], paged="permuted", plant=True,
                   order="sink_recent")


@pytest.mark.parametrize("eps,p", [(1e-2, 1), (5e-2, 2), (2e-3, 2)])
def test_all_heads_is_the_default(eps, p):
    w = _work()
    a = O.run_workload(w, eps_mag=eps, eps_dir=eps, patience=p, trace=True)
    b = O.run_workload(w, eps_mag=eps, eps_dir=eps, patience=p, trace=True, probe_heads=w.group)
    assert np.array_equal(a["blocks_used"], b["blocks_used"])
    np.testing.assert_array_equal(a["trace_mag"], b["trace_mag"])


@pytest.mark.parametrize("eps,p", [(1e-2, 1), (5e-2, 2)])
def test_equal_heads_decide_alike(eps, p):
    w = _work()
    q = w.q.copy()
    G = w.group
    for g in range(w.num_kv_heads):
        q[:, g * G:(g + 1) * G] = q[:, g * G:g * G + 1]
    w = dataclasses.replace(w, q=q)
    ref = O.run_workload(w, eps_mag=eps, eps_dir=eps, patience=p, trace=True)
    for ph in range(1, G + 1):
        r = O.run_workload(w, eps_mag=eps, eps_dir=eps, patience=p, trace=True, probe_heads=ph)
        assert np.array_equal(r["blocks_used"], ref["blocks_used"]), ph
        np.testing.assert_allclose(r["trace_mag"], ref["trace_mag"], rtol=1e-9, atol=1e-15)
        np.testing.assert_allclose(r["trace_dir"], ref["trace_dir"], rtol=1e-6, atol=1e-12)


@pytest.mark.parametrize("eps,p", [(1e-2, 1), (5e-2, 2), (2e-3, 2)])
def test_first_head_equals_single_head_workload(eps, p):
    w = _work()
    G = w.group
    w1 = dataclasses.replace(w, q=np.ascontiguousarray(w.q[:, ::G]), num_q_heads=w.num_kv_heads)
    a = O.run_workload(w, eps_mag=eps, eps_dir=eps, patience=p, trace=True, probe_heads=1)
    b = O.run_workload(w1, eps_mag=eps, eps_dir=eps, patience=p, trace=True)
    assert np.array_equal(a["blocks_used"], b["blocks_used"])
    np.testing.assert_array_equal(a["trace_mag"], b["trace_mag"])
    np.testing.assert_array_equal(a["trace_dir"], b["trace_dir"])
    # and the option changes something on this workload
    c = O.run_workload(w, eps_mag=eps, eps_dir=eps, patience=p, trace=True)
    assert not np.array_equal(np.nan_to_num(a["trace_mag"]), np.nan_to_num(c["trace_mag"]))
