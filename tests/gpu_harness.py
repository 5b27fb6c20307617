"""Shared helpers of the GPU parity tests: run libart through the C ABI and
compare with the CPU oracle.

Tolerances (bf16 or fp32 inputs, fp32 accumulation on the device, fp64 in the
oracle): outputs within max-abs 2e-2 and relative L2 5e-3 of the oracle, the
relative L2 bound holding over all compared outputs together and for every
(sequence, query head) output vector on its own;
blocks_used identical except where a statistic at a step that decides the
stop lies within 1e-4 (relative) of its threshold (a tie, counted and
reported, not failed). When blocks_used differs in a tie, the output is
compared with the oracle forced to the device's blocks_used.
"""
from __future__ import annotations

import numpy as np

import kv_cache_early_gb300 as K
import oracle as O

MAX_ABS = 2e-2
REL_L2 = 5e-3
TIE_REL = 1e-4


def device_out(dev, w):
    import torch
    torch.cuda.synchronize()
    out = dev.out.float().cpu().numpy().reshape(w.num_items, w.group, w.head_dim)
    return out


def run_gpu(w, mode="art", eps_mag=None, eps_dir=None, patience=None, dev=None, visit_order="default"):
    import torch
    dev = dev or K.DeviceInputs(w)
    em = w.eps_mag if eps_mag is None else eps_mag
    ed = w.eps_dir if eps_dir is None else eps_dir
    p = w.patience if patience is None else patience
    if mode == "art":
        dev.blocks_used.fill_(-7)
        dev.art(em, ed, p, visit_order=visit_order)
    else:
        dev.dense(visit_order=visit_order)
    torch.cuda.synchronize()
    out = device_out(dev, w)
    bu = dev.blocks_used.cpu().numpy().reshape(-1) if mode == "art" else None
    return out, bu, dev.status(), dev


def compare(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if ref.size == 0:
        return 0.0, 0.0
    err = np.abs(gpu - ref)
    max_abs = float(err.max())
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(gpu - ref) / nref) if nref > 0 else float(np.linalg.norm(gpu - ref))
    assert np.isfinite(gpu).all(), f"{what}: non-finite device output"
    assert max_abs <= MAX_ABS, f"{what}: max abs error {max_abs:.3e} > {MAX_ABS}"
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2}"
    # every output vector (last axis) on its own: one wrong row cannot hide among many
    g2 = gpu.reshape(-1, gpu.shape[-1])
    r2 = ref.reshape(-1, ref.shape[-1])
    nr = np.linalg.norm(r2, axis=1)
    ne = np.linalg.norm(g2 - r2, axis=1)
    row_rel = np.where(nr > 0, ne / np.where(nr > 0, nr, 1.0), ne)
    worst = int(np.argmax(row_rel))
    assert row_rel[worst] <= REL_L2, (
        f"{what}: output vector {worst} (of {len(row_rel)}) relative L2 error {row_rel[worst]:.3e} > {REL_L2}")
    return max_abs, rel


def is_tie(trace_mag, trace_dir, lo, hi, eps_mag, eps_dir):
    """Any step in [lo, hi] (1-indexed, inclusive) with a statistic within
    TIE_REL (relative) of its threshold."""
    em, ed = float(np.float32(eps_mag)), float(np.float32(eps_dir))
    for i in range(max(lo, 2), hi + 1):
        for stat, eps in ((trace_mag[i - 1], em), (trace_dir[i - 1], ed)):
            if np.isfinite(stat) and np.isfinite(eps) and eps > 0 and abs(stat - eps) <= TIE_REL * eps:
                return True
    return False


def check_art(w, gpu_out, gpu_bu, eps_mag, eps_dir, patience, items=None, visit_order="default", what="",
              probe_heads=0):
    """blocks_used (exact up to ties) and outputs against the oracle.
    Returns dict(ties, mismatches, items, mean_bu)."""
    its = np.arange(w.num_items) if items is None else np.asarray(items)
    r = O.run_workload(w, items=None if items is None else its, eps_mag=eps_mag, eps_dir=eps_dir,
                       patience=patience, trace=True, visit_order=visit_order, probe_heads=probe_heads)
    ob = r["blocks_used"]
    gb = np.asarray(gpu_bu)[its]
    ties = 0
    for k in np.nonzero(ob != gb)[0]:
        assert ob[k] >= 0 and gb[k] >= 0, f"{what}: item {its[k]} blocks_used gpu {gb[k]} oracle {ob[k]}"
        lo = min(ob[k], gb[k]) - patience + 1
        hi = max(ob[k], gb[k])
        assert is_tie(r["trace_mag"][k], r["trace_dir"][k], lo, hi, eps_mag, eps_dir), (
            f"{what}: item {its[k]}: blocks_used gpu {gb[k]} != oracle {ob[k]} outside the tie zone "
            f"(d_mag {r['trace_mag'][k][max(lo, 2) - 1:hi]}, d_dir {r['trace_dir'][k][max(lo, 2) - 1:hi]})")
        ties += 1
    ok = gb >= 0
    rf = O.run_workload(w, mode="forced", items=its, forced=np.maximum(gb, 0), visit_order=visit_order)
    compare(np.asarray(gpu_out)[its][ok], rf["out"][ok], what)
    assert (np.abs(np.asarray(gpu_out)[its][~ok]).max(initial=0.0) == 0.0), f"{what}: bad items must be zero"
    return dict(ties=ties, mismatches=int((ob != gb).sum()), items=len(its), mean_bu=float(gb[ok].mean()) if ok.any() else 0.0)


def check_dense(w, gpu_out, items=None, visit_order="default", what=""):
    its = np.arange(w.num_items) if items is None else np.asarray(items)
    r = O.run_workload(w, mode="dense", items=None if items is None else its, visit_order=visit_order)
    ok = r["status"] == 0
    compare(np.asarray(gpu_out)[its][ok], r["out"][ok], what)
    return r
