"""CPU oracle for ART decode attention -- TEST INFRASTRUCTURE.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package. The CUDA product path never imports, links or calls it,
and it shares no code with that path (not even headers).

`art_oracle.c` holds the fp64 definition (exact softmax attention,
"ART: Attention Run-time Termination" sec. 3.1 Eq. (1), and the sequential
termination rule of sec. 3.2 / the gist.science explainer sec. 2.2-2.4).
This module builds it with gcc (no fast-math) and calls it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "art_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE_DENSE, MODE_ART, MODE_FORCED = 0, 1, 2
ITEM_STATUS = {0: "ok", 1: "visit entry out of range", 2: "page id out of range", 3: "duplicate visit entry"}


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "block_size",
        "max_pages_per_seq", "max_visit", "num_probe", "num_pages_total", "dtype")]


def build(force: bool = False, src: str = _SRC, lib: str = _LIB) -> str:
    """Compile the oracle shared library with gcc -O2 (IEEE fp64, no fast-math)."""
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        tmp = lib + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"])
        os.replace(tmp, lib)
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes front end of one build of the oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        lib.oracle_art.argtypes = [ctypes.POINTER(_Shape), P, P, P, P, P, P,
                                   ctypes.c_double, ctypes.c_double, ctypes.c_int32, P,
                                   ctypes.c_int32, P, ctypes.c_int32, P,
                                   P, P, P, P, P, ctypes.c_int32, ctypes.c_int32]
        lib.oracle_art.restype = ctypes.c_int
        self.lib = lib

    def run(self, shape: dict, q, k_cache, v_cache, block_table, seq_lens, visit_order, *,
            eps_mag: float = 0.0, eps_dir: float = 0.0, patience: int = 1, probe_idx=None,
            mode: str = "art", items=None, forced=None, trace: bool = False, threads: int = 0,
            probe_heads: int = 0) -> dict:
        """Run the oracle.

        shape: dict with the fields of the layout (batch, num_q_heads, num_kv_heads,
        head_dim, page_size, block_size, max_pages_per_seq, max_visit, num_probe,
        num_pages_total, dtype: 0 = bf16 bits as uint16, 1 = fp32).
        mode: "dense" (all listed blocks), "art" (the termination rule) or
        "forced" (out = O^(forced[k]) for each selected item).
        items: optional list of item ids b * num_kv_heads + g (default: all).
        eps values are compared in fp64 exactly as given (pass the float32 value
        used on the device to reproduce its thresholds).
        probe_heads: the probe is formed by query heads 0 .. probe_heads-1 of each
        group (0: all G heads).
        Returns dict(out [n_items, G, d] fp64, blocks_used, status, trace_mag,
        trace_dir (None unless trace), threads).
        """
        sh = _Shape(**{k: int(v) for k, v in shape.items()})
        G = sh.num_q_heads // sh.num_kv_heads
        dt = np.uint16 if sh.dtype == 0 else np.float32
        q = np.ascontiguousarray(q, dtype=dt)
        k_cache = np.ascontiguousarray(k_cache, dtype=dt)
        v_cache = np.ascontiguousarray(v_cache, dtype=dt)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        if visit_order is not None:
            visit_order = np.ascontiguousarray(visit_order, dtype=np.int32)
        probe = None if probe_idx is None else np.ascontiguousarray(probe_idx, dtype=np.int32)
        if items is None:
            its = None
            n_items = sh.batch * sh.num_kv_heads
        else:
            its = np.ascontiguousarray(items, dtype=np.int32)
            n_items = int(its.size)
        fz = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        m = {"dense": MODE_DENSE, "art": MODE_ART, "forced": MODE_FORCED}[mode]
        nn = max(n_items, 1)
        out = np.zeros((nn, G, sh.head_dim), dtype=np.float64)
        bu = np.zeros(nn, dtype=np.int32)
        st = np.zeros(nn, dtype=np.int32)
        tm = np.full((nn, sh.max_visit), np.nan) if trace else None
        td = np.full((nn, sh.max_visit), np.nan) if trace else None
        if n_items == 0:
            return dict(out=out[:0], blocks_used=bu[:0], status=st[:0], trace_mag=None,
                        trace_dir=None, threads=0)
        nt = self.lib.oracle_art(ctypes.byref(sh), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(block_table), _ptr(seq_lens), _ptr(visit_order),
                                 float(eps_mag), float(eps_dir), int(patience), _ptr(probe), m,
                                 _ptr(its), n_items if its is not None else 0, _ptr(fz),
                                 _ptr(out), _ptr(bu), _ptr(st), _ptr(tm), _ptr(td), int(threads),
                                 int(probe_heads))
        if nt < 0:
            raise ValueError(f"oracle rejected its arguments (code {nt})")
        return dict(out=out, blocks_used=bu, status=st, trace_mag=tm, trace_dir=td, threads=nt)


def default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def run(*args, **kw) -> dict:
    """Run the default build of the oracle; see Oracle.run."""
    return default().run(*args, **kw)


def run_workload(w, *, mode: str = "art", items=None, forced=None, trace: bool = False, threads: int = 0,
                 eps_mag=None, eps_dir=None, patience=None, visit_order="default", orc=None,
                 probe_heads: int = 0) -> dict:
    """Convenience wrapper taking a workload object with the usual attributes.
    Thresholds default to the workload's, rounded to float32 as the device sees them.
    `orc` selects another build of the oracle (default: the stock one)."""
    em = w.eps_mag if eps_mag is None else eps_mag
    ed = w.eps_dir if eps_dir is None else eps_dir
    vo = w.visit_order if isinstance(visit_order, str) else visit_order
    sh = w.shape_dict()
    if vo is not None:
        sh["max_visit"] = int(vo.shape[2])
    return (orc or default()).run(sh, w.q, w.k_cache, w.v_cache, w.block_table, w.seq_lens, vo,
        eps_mag=float(np.float32(em)), eps_dir=float(np.float32(ed)),
        patience=w.patience if patience is None else patience, probe_idx=w.probe_idx,
        mode=mode, items=items, forced=forced, trace=trace, threads=threads, probe_heads=probe_heads)
