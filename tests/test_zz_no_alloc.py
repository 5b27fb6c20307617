"""art_decode_static -- ART decode for callers that cannot allocate device memory.

The entry point keeps its scratch in a device array inside the library instead
of a caller-provided workspace. This test calls it through the C ABI twice in a
row on the same inputs and checks both results against art_decode (the entry
point with a caller workspace) within the parity tests' tolerances: identical
blocks_used, outputs within max-abs 2e-2 and relative L2 5e-3. It also checks
that batches beyond the array's capacity are refused before any device work.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import kv_cache_early_gb300 as K  # noqa: E402
import workloads as W  # noqa: E402
from gpu_harness import MAX_ABS, REL_L2  # noqa: E402

STATIC_MAX_ITEMS = 16384


def _static_fn():
    L = K.lib()
    f = L.art_decode_static
    P = ctypes.c_void_p
    f.argtypes = [P, P, P, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_int32, P, P, P,
                  ctypes.POINTER(K.ArtShape), P]
    f.restype = ctypes.c_int
    return f


def _call_static(f, dev, eps, p, out, bu):
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(ptr(dev.q), ptr(dev.k_cache), ptr(dev.v_cache), ptr(dev.block_table), ptr(dev.seq_lens),
             ptr(dev.visit_order), eps, eps, p, ptr(dev.probe_idx), ptr(out), ptr(bu), ctypes.byref(dev.shape),
             stream)


@pytest.mark.parametrize("k,eps,p", [(2, 1e-2, 2), (3, 5e-2, 1), (4, 1e-2, 2)])
def test_static_workspace_matches_caller_workspace(k, eps, p):
    w = W.config(k, small=True)
    dev = K.DeviceInputs(w)
    f = _static_fn()
    dev.art(eps, eps, p)
    torch.cuda.synchronize()
    ref_out = dev.out.float().cpu().numpy()
    ref_bu = dev.blocks_used.cpu().numpy()
    assert dev.status() == 0
    for call in range(2):
        out = torch.full_like(dev.out, float("nan"))
        bu = torch.full_like(dev.blocks_used, -7)
        rc = _call_static(f, dev, eps, p, out, bu)
        assert rc == K.ART_OK, (rc, K.lib().art_status_string(rc), K.lib().art_last_cuda_error())
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.array_equal(bu.cpu().numpy(), ref_bu), f"call {call}: blocks_used differ"
        err = np.abs(got - ref_out)
        assert np.isfinite(got).all()
        assert err.max() <= MAX_ABS, f"call {call}: max abs {err.max()}"
        rel = np.linalg.norm(got - ref_out) / max(np.linalg.norm(ref_out), 1e-30)
        assert rel <= REL_L2, f"call {call}: relative L2 {rel}"


def test_static_status_after_bad_page_then_good_call():
    """A call with one page id outside the pool (a bad host-side input that the
    kernels check): that sequence's items get blocks_used = -1 and the array's
    status word reports the bad page. The next call with good inputs on the same
    array matches art_decode again."""
    w = W.config(3, small=True)
    dev = K.DeviceInputs(w)
    f = _static_fn()
    eps, p = 1e-2, 2
    dev.art(eps, eps, p)
    torch.cuda.synchronize()
    ref_out = dev.out.float().cpu().numpy()
    ref_bu = dev.blocks_used.cpu().numpy()
    good_table = dev.block_table.clone()
    dev.block_table[1, 0] = w.k_cache.shape[0] + 5  # sequence 1's first page: outside the pool
    out = torch.zeros_like(dev.out)
    bu = torch.full_like(dev.blocks_used, -7)
    assert _call_static(f, dev, eps, p, out, bu) == K.ART_OK
    torch.cuda.synchronize()
    st = K.art_read_static_status()
    assert st & 4, K.status_names(st)  # bad page id
    got_bu = bu.cpu().numpy()
    assert (got_bu[1] == -1).all()
    assert np.array_equal(np.delete(got_bu, 1, axis=0), np.delete(ref_bu, 1, axis=0))
    dev.block_table.copy_(good_table)
    out = torch.full_like(dev.out, float("nan"))
    bu = torch.full_like(dev.blocks_used, -7)
    assert _call_static(f, dev, eps, p, out, bu) == K.ART_OK
    torch.cuda.synchronize()
    assert K.art_read_static_status() == 0
    assert np.array_equal(bu.cpu().numpy(), ref_bu)
    got = out.float().cpu().numpy()
    assert np.abs(got - ref_out).max() <= MAX_ABS
    assert np.linalg.norm(got - ref_out) / np.linalg.norm(ref_out) <= REL_L2


def test_static_workspace_refuses_too_many_items():
    w = W.config(2, small=True)
    dev = K.DeviceInputs(w)
    f = _static_fn()
    big = K.make_shape(**dict(w.shape_dict(), batch=STATIC_MAX_ITEMS // w.num_kv_heads + 1))
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = f(ptr(dev.q), ptr(dev.k_cache), ptr(dev.v_cache), ptr(dev.block_table), ptr(dev.seq_lens),
           ptr(dev.visit_order), 1e-2, 1e-2, 2, ptr(dev.probe_idx), ptr(dev.out), ptr(dev.blocks_used),
           ctypes.byref(big), None)
    assert rc == K.ART_ERR_UNSUPPORTED
