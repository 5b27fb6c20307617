"""Python binding of libart, the ART decode-attention library (include/art.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libart.so. The names follow the C ABI: `art_decode`,
`dense_decode`, `art_workspace_bytes`, `art_read_device_status`.
Tensors are torch CUDA tensors; PyTorch supplies device memory and streams.

The library must have been built (`kv_cache_early_gb300.build.build()`);
importing works without it, but the first call raises if it is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libart.so")

ART_DTYPE_BF16, ART_DTYPE_F32 = 0, 1
ART_OK, ART_ERR_INVALID_ARG, ART_ERR_UNSUPPORTED, ART_ERR_WORKSPACE, ART_ERR_LAUNCH = 0, -1, -2, -3, -4
STATUS_BITS = {1: "bad visit entry", 2: "duplicate visit entry", 4: "bad page id", 8: "bad seq_len",
               16: "bad probe index", 32: "wait timeout", 64: "internal check failed"}
EXPORTS = ("art_workspace_bytes", "art_decode_path", "dense_decode_path", "art_decode", "art_decode_ex",
           "dense_decode",
           "art_decode_static", "art_read_static_status", "art_read_device_status",
           "art_status_string", "art_last_cuda_error", "art_set_timing_events",
           "art_select_workspace_bytes", "art_select_blocks")


class ArtShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "block_size",
        "max_pages_per_seq", "max_visit", "num_probe", "num_pages_total", "dtype")]


class ArtOptions(ctypes.Structure):
    _fields_ = [("probe_heads", ctypes.c_int32), ("reserved", ctypes.c_int32 * 7)]


class ArtError(RuntimeError):
    pass


_lock = threading.Lock()
_lib = None


def lib(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libart.so; raises ArtError when it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise ArtError(f"{path} is missing: build the CUDA library first "
                               "(python -m kv_cache_early_gb300.build)")
            L = ctypes.CDLL(path)
            P, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            SP = ctypes.POINTER(ArtShape)
            L.art_workspace_bytes.argtypes = [SP]
            L.art_workspace_bytes.restype = SZ
            L.art_decode_path.argtypes = [SP, I32, SZ]
            L.art_decode_path.restype = ctypes.c_int
            L.dense_decode_path.argtypes = [SP, SZ]
            L.dense_decode_path.restype = ctypes.c_int
            L.art_decode.argtypes = [P, P, P, P, P, P, F32, F32, I32, P, P, P, SP, P, SZ, P]
            L.art_decode.restype = ctypes.c_int
            L.dense_decode.argtypes = [P, P, P, P, P, P, P, SP, P, SZ, P]
            L.dense_decode.restype = ctypes.c_int
            L.art_read_device_status.argtypes = [P, ctypes.POINTER(I32)]
            L.art_read_device_status.restype = ctypes.c_int
            L.art_status_string.argtypes = [ctypes.c_int]
            L.art_status_string.restype = ctypes.c_char_p
            L.art_last_cuda_error.argtypes = []
            L.art_last_cuda_error.restype = ctypes.c_char_p
            L.art_decode_ex.argtypes = [P, P, P, P, P, P, F32, F32, I32, P, P, P, SP, P, SZ, P,
                                        ctypes.POINTER(ArtOptions)]
            L.art_decode_ex.restype = ctypes.c_int
            L.art_decode_static.argtypes = [P, P, P, P, P, P, F32, F32, I32, P, P, P, SP, P]
            L.art_decode_static.restype = ctypes.c_int
            L.art_read_static_status.argtypes = [ctypes.POINTER(I32)]
            L.art_read_static_status.restype = ctypes.c_int
            L.art_set_timing_events.argtypes = [P, P]
            L.art_set_timing_events.restype = None
            L.art_select_workspace_bytes.argtypes = [SP]
            L.art_select_workspace_bytes.restype = SZ
            L.art_select_blocks.argtypes = [P, P, P, P, F32, I32, I32, P, SP, P, SZ, P]
            L.art_select_blocks.restype = ctypes.c_int
            _lib = L
    return _lib


def make_shape(**kw) -> ArtShape:
    return ArtShape(**{k: int(v) for k, v in kw.items()})


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int):
    if rc != ART_OK:
        L = lib()
        msg = L.art_status_string(rc).decode()
        if rc == ART_ERR_LAUNCH:
            msg += ": " + L.art_last_cuda_error().decode()
        raise ArtError(f"libart returned {rc} ({msg})")


def art_workspace_bytes(shape: ArtShape) -> int:
    return int(lib().art_workspace_bytes(ctypes.byref(shape)))


def art_decode_path(shape: ArtShape, patience: int, workspace_bytes: int) -> int:
    """0: one CTA per item; 1: the unit path (see include/art.h)."""
    return int(lib().art_decode_path(ctypes.byref(shape), int(patience), int(workspace_bytes)))


def dense_decode_path(shape: ArtShape, workspace_bytes: int) -> int:
    """The kernel path dense_decode takes: 0 one CTA per item, 1 the unit path."""
    return int(lib().dense_decode_path(ctypes.byref(shape), int(workspace_bytes)))


def art_decode(q, k_cache, v_cache, block_table, seq_lens, visit_order, eps_mag, eps_dir, patience,
               probe_idx, out, blocks_used, shape: ArtShape, workspace, stream=None, check: bool = True) -> int:
    """ART decode attention (see include/art.h). Tensors: torch CUDA tensors or raw
    device addresses (int). Returns the C return code (raises on error if check)."""
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else \
        art_workspace_bytes(shape)
    rc = lib().art_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
                          _ptr(visit_order), float(eps_mag), float(eps_dir), int(patience), _ptr(probe_idx),
                          _ptr(out), _ptr(blocks_used), ctypes.byref(shape), _ptr(workspace), ws_bytes,
                          _stream(stream))
    if check:
        _check(rc)
    return rc


def dense_decode(q, k_cache, v_cache, block_table, seq_lens, visit_order, out, shape: ArtShape, workspace,
                 stream=None, check: bool = True) -> int:
    """The full-scan twin of art_decode (no probe, no termination)."""
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else \
        art_workspace_bytes(shape)
    rc = lib().dense_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
                            _ptr(visit_order), _ptr(out), ctypes.byref(shape), _ptr(workspace), ws_bytes,
                            _stream(stream))
    if check:
        _check(rc)
    return rc


def art_decode_ex(q, k_cache, v_cache, block_table, seq_lens, visit_order, eps_mag, eps_dir, patience,
                  probe_idx, out, blocks_used, shape: ArtShape, workspace, stream=None, check: bool = True,
                  probe_heads: int = 0) -> int:
    """art_decode with options: probe_heads 1..G forms the probe from query heads
    0 .. probe_heads-1 of each group (0: all G)."""
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else \
        art_workspace_bytes(shape)
    opts = ArtOptions(probe_heads=int(probe_heads))
    rc = lib().art_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
                             _ptr(visit_order), float(eps_mag), float(eps_dir), int(patience), _ptr(probe_idx),
                             _ptr(out), _ptr(blocks_used), ctypes.byref(shape), _ptr(workspace), ws_bytes,
                             _stream(stream), ctypes.byref(opts))
    if check:
        _check(rc)
    return rc


def art_decode_static(q, k_cache, v_cache, block_table, seq_lens, visit_order, eps_mag, eps_dir, patience,
                      probe_idx, out, blocks_used, shape: ArtShape, stream=None, check: bool = True) -> int:
    """art_decode with the library's own fixed device scratch instead of a workspace."""
    rc = lib().art_decode_static(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
                                 _ptr(visit_order), float(eps_mag), float(eps_dir), int(patience),
                                 _ptr(probe_idx), _ptr(out), _ptr(blocks_used), ctypes.byref(shape),
                                 _stream(stream))
    if check:
        _check(rc)
    return rc


def art_select_workspace_bytes(shape: ArtShape) -> int:
    return int(lib().art_select_workspace_bytes(ctypes.byref(shape)))


def art_select_blocks(q, k_cache, block_table, seq_lens, top_frac, keep_last, visit_order, shape: ArtShape,
                      workspace, stream=None, check: bool = True, order: int = 0) -> int:
    """Key-based block selection writing an ART visit list (see include/art.h);
    order 0: most recent first, 1: highest score first."""
    ws_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else \
        art_select_workspace_bytes(shape)
    rc = lib().art_select_blocks(_ptr(q), _ptr(k_cache), _ptr(block_table), _ptr(seq_lens), float(top_frac),
                                 int(keep_last), int(order), _ptr(visit_order), ctypes.byref(shape),
                                 _ptr(workspace), ws_bytes,
                                 _stream(stream))
    if check:
        _check(rc)
    return rc


def set_timing_events(start=None, stop=None):
    """Have this thread's next calls record `start` / `stop` (torch.cuda.Event,
    already recorded once so that they exist) around the decode-kernel launch;
    no arguments clears."""
    h = lambda e: None if e is None else ctypes.c_void_p(int(e.cuda_event))
    lib().art_set_timing_events(h(start), h(stop))


def art_read_static_status() -> int:
    """Status word of art_decode_static's array on the current device (blocking)."""
    st = ctypes.c_int32(0)
    _check(lib().art_read_static_status(ctypes.byref(st)))
    return int(st.value)


def art_read_device_status(workspace) -> int:
    """Device status bits of the last call that used `workspace` (blocking copy)."""
    st = ctypes.c_int32(0)
    _check(lib().art_read_device_status(_ptr(workspace), ctypes.byref(st)))
    return int(st.value)


def status_names(bits: int) -> list:
    return [v for k, v in STATUS_BITS.items() if bits & k]


class DeviceInputs:
    """Device copies of one decode batch plus the matching ArtShape.

    `src` is any object with the attributes q, k_cache, v_cache, block_table,
    seq_lens, visit_order (or None), probe_idx and the size fields of ArtShape
    (numpy arrays; bf16 data as uint16 bits). Pure marshalling.
    """

    def __init__(self, src, device="cuda", pin: bool = False):
        import numpy as np
        import torch

        def dev(a, dtype=None):
            t = torch.from_numpy(np.ascontiguousarray(a))
            if dtype is not None:
                t = t.view(dtype)
            return t.to(device, non_blocking=False)

        bf16 = src.dtype == "bf16"
        tdt = torch.bfloat16 if bf16 else torch.float32
        self.torch_dtype = tdt
        self.q = dev(src.q, torch.bfloat16 if bf16 else None)
        self.k_cache = dev(src.k_cache, torch.bfloat16 if bf16 else None)
        self.v_cache = dev(src.v_cache, torch.bfloat16 if bf16 else None)
        self.block_table = dev(src.block_table.astype(np.int32))
        self.seq_lens = dev(src.seq_lens.astype(np.int32))
        self.visit_order = None if src.visit_order is None else dev(src.visit_order.astype(np.int32))
        self.probe_idx = dev(src.probe_idx.astype(np.int32))
        sd = src.shape_dict()
        self.shape = make_shape(**sd)
        self.num_items = sd["batch"] * sd["num_kv_heads"]
        self.out = torch.empty((sd["batch"], sd["num_q_heads"], sd["head_dim"]), dtype=tdt, device=device)
        self.blocks_used = torch.empty((sd["batch"], sd["num_kv_heads"]), dtype=torch.int32, device=device)
        nbytes = art_workspace_bytes(self.shape)
        self.workspace = torch.zeros((nbytes + 15) // 16 * 16, dtype=torch.uint8, device=device)

    def art(self, eps_mag, eps_dir, patience, stream=None, visit_order="default", out=None, blocks_used=None,
            probe_heads: int = 0):
        vo = self.visit_order if isinstance(visit_order, str) else visit_order
        args = (self.q, self.k_cache, self.v_cache, self.block_table, self.seq_lens, vo, eps_mag, eps_dir,
                patience, self.probe_idx, self.out if out is None else out,
                self.blocks_used if blocks_used is None else blocks_used, self.shape, self.workspace, stream)
        if probe_heads:
            art_decode_ex(*args, probe_heads=probe_heads)
        else:
            art_decode(*args)

    def dense(self, stream=None, visit_order="default", out=None):
        vo = self.visit_order if isinstance(visit_order, str) else visit_order
        dense_decode(self.q, self.k_cache, self.v_cache, self.block_table, self.seq_lens, vo,
                     self.out if out is None else out, self.shape, self.workspace, stream)

    def status(self) -> int:
        return art_read_device_status(self.workspace)
