"""Failure detection on the GPU without a fault.

Every wait in the kernels (mbarrier phases, flags written by other CTAs) is
bounded: when one runs out, the kernel sets ART_STATUS_TIMEOUT in the
workspace, each warp gives up at its own bounded wait, the warps that issued
copies wait for their own copies in flight, and the CTA returns, leaving the
context usable.

The test hook ART_TEST_STALL_NS=<ns> makes the consumer warps first wait on a
barrier that nothing completes, and sets every wait limit to <ns> (the final
drain of a warp's own copies keeps its 1 s limit). The call must
return, the stream synchronize without a CUDA error, the status word carry the
timeout bit, and the next call with the hook off, on the same buffers, must
match the oracle.
"""
import numpy as np
import pytest

import workloads as W
from gpu_harness import check_art, check_dense, run_gpu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 32  # ART_STATUS_TIMEOUT


@pytest.mark.parametrize("mode", ["art", "dense"])
@pytest.mark.parametrize("k,path,groups", [
    (2, "one-cta", None),  # four consumer groups and one copy warp (items fit one per SM)
    (2, "one-cta", "3"),   # three groups and two copy warps
    (2, "one-cta", "1"),   # one keys-split group, the producer issuing the copies
    (2, "units", None), (3, "units", None), (1, "one-cta", None)])
def test_bounded_wait_expires_and_next_call_is_clean(k, path, groups, mode, monkeypatch):
    import kv_cache_early_gb300 as K
    monkeypatch.setenv("ART_UNITS", "1" if path == "units" else "0")
    if groups is not None:
        monkeypatch.setenv("ART_GROUPS", groups)
    w = W.config(k, small=True)
    dev = K.DeviceInputs(w)
    assert K.art_decode_path(dev.shape, 2, dev.workspace.numel()) == (1 if path == "units" else 0)
    monkeypatch.setenv("ART_TEST_STALL_NS", "200000")
    if mode == "art":
        dev.art(1e-2, 1e-2, 2)
    else:
        dev.dense()
    torch.cuda.synchronize()  # raises on a CUDA error
    st = dev.status()
    assert st & TIMEOUT_BIT, K.status_names(st)
    monkeypatch.delenv("ART_TEST_STALL_NS")
    out, bu, st, _ = run_gpu(w, mode, 1e-2, 1e-2, 2, dev=dev)
    assert st == 0, K.status_names(st)
    if mode == "art":
        check_art(w, out, bu, 1e-2, 1e-2, 2, what=f"after a timeout, config {k} {path}")
    else:
        check_dense(w, out, what=f"after a timeout, config {k} {path}")
