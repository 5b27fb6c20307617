#!/usr/bin/env python3
"""Benchmark of ART decode attention on one decode workload.

One step = one art_decode call (memset of the workspace header, the plan
kernel, the persistent decode kernel) over the whole batch, inputs resident
in HBM. Prints one JSON line (rank 0) with queries/s, the HBM roofline of the
decode kernel, the dense twin, the CPU oracle baseline, clocks and an
end-to-end figure through the public API with host buffers.

Default workload: the ragged batch (64 sequences of 1k-64k tokens, 32 query /
8 KV heads, d=128, bf16, 16-token pages placed by a seeded permutation, 5 % of
the blocks with values x8, sink-first most-recent-first order, eps 1e-3,
patience 2), the largest of the five decode workloads (about 8.7 GB of listed
K and V).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 1..5] [--eps E] [--patience P] [--no-cpu-baseline]
                  [--shard sequences|replicas] [--diag]
Under torchrun (N > 1) the default (--shard sequences) partitions the one
seeded workload by sequence: rank r owns a contiguous slice of the sequences
with their block-table rows and the pages they name (strong scaling, no
collective on the data path; the step time is the max over ranks).
--shard replicas runs a full copy of the workload on every rank instead (weak
scaling). --diag prints the convergence and score-versus-contribution
diagnostics instead of the benchmark line.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--shard", default="sequences", choices=["sequences", "replicas"],
                    help="N > 1: partition the workload's sequences over the ranks, or run a replica per rank")
    ap.add_argument("--probe", default="stride4", choices=["stride4", "full"],
                    help="the probe columns: every 4th head dim (the workloads' own), or every head dim")
    ap.add_argument("--diag", action="store_true",
                    help="print the convergence (O^(t) vs O^(T)) and score-vs-contribution diagnostics")
    ap.add_argument("--eps", type=float, default=None)
    ap.add_argument("--patience", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None,
                    help="replace the workload's batch (smaller profiler captures of the same kernel)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over the ranks of the default process group
    (x itself without one). Used for the step time: the job is as slow as its
    slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# byte accounting (algorithmic bytes of one call)
# ---------------------------------------------------------------------------
def listed_blocks(w):
    """Per item: the listed logical blocks (list of arrays)."""
    lens = w.visit_lengths()
    out = []
    for it in range(w.num_items):
        b, g = divmod(it, w.num_kv_heads)
        if w.visit_order is None:
            out.append(np.arange(lens[it]))
        else:
            out.append(w.visit_order[b, g, : lens[it]].astype(np.int64))
    return out


def kv_bytes(w, blocks_used=None):
    """K+V bytes of the first blocks_used listed blocks of every item (all if None):
    tokens x 2 (K and V) x head_dim x element size."""
    per_tok = 2 * w.head_dim * w.elem_bytes
    tot = 0
    for it, lst in enumerate(listed_blocks(w)):
        b = it // w.num_kv_heads
        k = len(lst) if blocks_used is None else max(0, int(blocks_used[it]))
        c = lst[:k]
        toks = np.minimum(w.block_size, int(w.seq_lens[b]) - c * w.block_size).sum()
        tot += int(toks) * per_tok
    return tot


def side_bytes(w):
    """q, out, lists and table entries the call reads or writes besides K/V."""
    qo = 2 * w.batch * w.num_q_heads * w.head_dim * w.elem_bytes
    lists = 0 if w.visit_order is None else w.visit_order.nbytes
    pages = int(np.ceil(w.seq_lens / w.page_size).sum()) * 4
    return qo + lists + pages + w.seq_lens.nbytes + w.num_items * 8


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": float(np.median(power)) if power else None}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def _code_only(src: bytes) -> bytes:
    """Source text without comments and blank lines (comments do not change a kernel)."""
    t = re.sub(r"/\*.*?\*/", "", src.decode(), flags=re.S)
    t = re.sub(r"//[^\n]*", "", t)
    return "\n".join(line.rstrip() for line in t.splitlines() if line.strip()).encode()


def kernel_source_hash(path=None):
    """Hash of the code (comments stripped) of the CUDA sources a kernel path
    compiles from: "one CTA per item" (the decode kernel, its instantiations and
    the plan kernel), "units" (the unit and merge kernels, which also use the
    decode kernel's helpers), or every source when path is None."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_early_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh")):
            continue
        if path is not None and f == "art_select.cu":
            continue
        if path == "one CTA per item" and f.startswith("art_units"):
            continue
        if path == "units" and f.startswith("art_inst_"):
            continue
        h.update(_code_only(open(os.path.join(csrc, f), "rb").read()))
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_traffic(config_name, alg_bytes, path):
    """DRAM bytes (read + write) per decode call from the committed ncu summary
    of this workload, only if it was taken on the current kernel source and the
    same kernel path ("units" or "one CTA per item"). A capture of a smaller
    batch of the same workload is scaled by the algorithmic bytes of the two
    launches."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None, None
    d = json.load(open(p))
    e = d.get(config_name)
    if not e or e.get("kernel_hash") != kernel_source_hash(path) or e.get("path") != path:
        return None, None
    t = float(e["dram_bytes"]) * alg_bytes / float(e["algorithmic_bytes"])
    src = f"ncu capture of {e['captured_workload']}" + \
        ("" if e["captured_workload"] == config_name else ", scaled by algorithmic bytes")
    return t, src


def cpu_baseline(w, eps, p, budget_s=12.0):
    """The CPU oracle on the host cores: whole workload, repeated while under budget."""
    import oracle as O
    times = []
    t_all = time.time()
    nt = 0
    while True:
        t0 = time.time()
        r = O.run_workload(w, eps_mag=eps, eps_dir=eps, patience=p)
        times.append(time.time() - t0)
        nt = r["threads"]
        if time.time() - t_all > budget_s or len(times) >= 5:
            break
    t = float(np.median(times))
    q = w.batch * w.num_q_heads
    return {"value": q / t, "unit": "queries/s", "cores": int(nt), "kind": "oracle",
            "sample": f"whole workload ({w.num_items} items, fp64 C oracle, ART rule), median of {len(times)} runs",
            "seconds_per_run": t}


def config_dict(w, eps, p, ws, shard="sequences"):
    par = "single GPU" if ws == 1 else (f"partition by sequence over {ws} GPUs" if shard == "sequences"
                                        else f"{ws} independent replicas")
    return {"workload": w.name, "batch": w.batch, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "page_size": w.page_size, "block_size": w.block_size, "eps": eps,
            "patience": p, "probe_columns_per_head": int(w.num_probe),
            "l2": "flushed (256 MB write) before every timed call; inputs also exceed L2",
            "parallelism": par}


def load_workload(args):
    """The workload of the command line; --probe full replaces the probe by every head dim."""
    w = W.config(args.config, eps=args.eps, patience=args.patience, batch=args.batch)
    if args.probe == "full":  # a probe over every head dim (the full-d ablation)
        import dataclasses
        w = dataclasses.replace(w, name=w.name + "-probe-full", probe_idx=np.arange(w.head_dim, dtype=np.int32))
    return w


# ---------------------------------------------------------------------------
# reference arm: the oracle timed as it stands on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    w = load_workload(args)
    eps, p = w.eps_mag, w.patience
    import oracle as O
    # each step: the oracle over a bounded sample of items (at most ~10 s per step)
    n_items = w.num_items
    t0 = time.time()
    O.run_workload(w, items=np.arange(min(n_items, 8)), eps_mag=eps, eps_dir=eps, patience=p)
    per_item = max((time.time() - t0) / min(n_items, 8), 1e-6)
    k = int(max(1, min(n_items, 10.0 / per_item)))
    items = np.arange(k)
    for _ in range(args.warmup):
        O.run_workload(w, items=items[: max(1, k // 8)], eps_mag=eps, eps_dir=eps, patience=p)
    ts = []
    nt = 0
    for _ in range(args.steps):
        t0 = time.time()
        r = O.run_workload(w, items=items, eps_mag=eps, eps_dir=eps, patience=p)
        ts.append(time.time() - t0)
        nt = r["threads"]
    t = float(np.mean(ts))
    value = k * w.group / t
    line = {"metric": "decode-attention queries/s (ART)", "value": value, "unit": "queries/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": dict(config_dict(w, eps, p, ws=1), items_per_step=int(k)),
            "cpu_baseline": {"value": value, "unit": "queries/s", "cores": int(nt), "kind": "oracle",
                             "sample": f"{k} of {n_items} (sequence, KV head) items per step"},
            "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    import kv_cache_early_gb300 as K
    from kv_cache_early_gb300 import build as B

    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    B.build()
    w_all = load_workload(args)
    sharded = ws > 1 and args.shard == "sequences"
    # partition by sequence: this rank's slice of the one seeded workload; else a replica
    w = W.shard_sequences(w_all, rank, ws) if sharded else w_all
    eps, p = w.eps_mag, w.patience
    dev = K.DeviceInputs(w)
    queries = w.batch * w.num_q_heads  # this rank's
    queries_job = w_all.batch * w.num_q_heads if sharded else ws * queries
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")  # > L2 (126 MB)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    def events(steps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:  # record once so that the CUDA events exist
            a.record(stream)
            b.record(stream)
        return evs

    def time_calls(fn, steps, kernel=False):
        """Per-call times (ms) with CUDA events on the launching stream; with
        `kernel`, also the decode kernel alone (events recorded by libart right
        around its launch)."""
        evs, kev = events(steps), events(steps) if kernel else None
        barrier()
        for i in range(steps):
            flush.fill_(i & 255)
            evs[i][0].record(stream)
            if kernel:
                K.set_timing_events(*kev[i])
            fn()
            evs[i][1].record(stream)
        if kernel:
            K.set_timing_events()
        barrier()
        t = np.array([a.elapsed_time(b) for a, b in evs])
        if not kernel:
            return t
        return t, np.array([a.elapsed_time(b) for a, b in kev])

    art_call = lambda: dev.art(eps, eps, p, stream=stream)
    dense_call = lambda: dev.dense(stream=stream)

    for _ in range(max(3, args.warmup)):
        art_call()
    torch.cuda.synchronize()
    bu = dev.blocks_used.cpu().numpy().reshape(-1).copy()
    status = dev.status()

    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    time.sleep(0.3)
    t_art, t_kern = time_calls(art_call, args.steps, kernel=True)
    clocks = clk.stop()
    ms = max_over_ranks(float(t_art.mean()), device="cuda")
    ms_kernel = max_over_ranks(float(t_kern.mean()), device="cuda")
    value = queries_job / (ms * 1e-3)

    # dense twin on the same buffers
    dense = None
    if not args.no_dense:
        for _ in range(max(3, args.warmup)):
            dense_call()
        t_d, t_dk = time_calls(dense_call, args.steps, kernel=True)
        ms_d, ms_dk = float(t_d.mean()), float(t_dk.mean())
        dense = {"queries_per_s": queries / (ms_d * 1e-3), "ms_per_step": ms_d, "kernel_ms": ms_dk,
                 "path": "units" if K.dense_decode_path(dev.shape, dev.workspace.numel()) == 1
                 else "one CTA per item",
                 "kernel_gbs": (kv_bytes(w) + side_bytes(w)) / (ms_dk * 1e-3) / 1e9,
                 "speedup_art_over_dense": ms_d / ms}
        # the dense twin on the other kernel path too (the path env override is read at
        # each call): ART is also compared with the faster of the two full scans
        saved = os.environ.get("ART_UNITS")
        other = "0" if dense["path"] == "units" else "1"
        os.environ["ART_UNITS"] = other
        if K.dense_decode_path(dev.shape, dev.workspace.numel()) == int(other):
            for _ in range(3):
                dense_call()
            t_o, t_ok = time_calls(dense_call, args.steps, kernel=True)
            ms_o = float(t_o.mean())
            best = min(ms_d, ms_o)
            dense["other_path"] = {"path": "units" if other == "1" else "one CTA per item", "ms_per_step": ms_o,
                                   "kernel_ms": float(t_ok.mean())}
            dense["fastest_dense_ms_per_step"] = best
            dense["speedup_art_over_fastest_dense"] = best / ms
        if saved is None:
            os.environ.pop("ART_UNITS", None)
        else:
            os.environ["ART_UNITS"] = saved
        # the detector's own cost: ART with eps = 0 never stops
        zero = lambda: dev.art(0.0, 0.0, p, stream=stream)
        for _ in range(3):
            zero()
        ms_z = float(time_calls(zero, args.steps).mean())
        dense["art_eps0_ms_per_step"] = ms_z
        # against the full scan on ART's own kernel path, so that only the detector differs
        art_on_units = K.art_decode_path(dev.shape, p, dev.workspace.numel()) == 1
        same = ms_d if (dense["path"] == "units") == art_on_units else dense.get("other_path", {}).get("ms_per_step")
        if same is not None:
            dense["detector_overhead_frac"] = ms_z / same - 1.0
            dense["detector_overhead_basis"] = "ART at eps 0 against the dense twin on the same kernel path ({})".format(
                "units" if art_on_units else "one CTA per item")
        if "fastest_dense_ms_per_step" in dense:
            dense["art_eps0_over_fastest_dense"] = ms_z / dense["fastest_dense_ms_per_step"]
        # with selected lists shorter than the context (the long-context workload), the
        # full scan of the whole cache too: what key selection plus ART replaces
        if w.visit_order is not None and int(w.visit_lengths().sum()) < int(np.ceil(w.seq_lens / w.block_size).sum()) * w.num_kv_heads:
            full = lambda: dev.dense(stream=stream, visit_order=None)
            for _ in range(3):
                full()
            t_f, t_fk = time_calls(full, args.steps, kernel=True)
            ms_f, ms_fk = float(t_f.mean()), float(t_fk.mean())
            full_bytes = int(w.seq_lens.sum()) * w.num_kv_heads * 2 * w.head_dim * w.elem_bytes
            dense["full_cache"] = {
                "what": "the dense twin over every block of the cache in natural order (NULL lists)",
                "ms_per_step": ms_f, "kernel_ms": ms_fk,
                "path": "units" if K.dense_decode_path(dev.shape, dev.workspace.numel()) == 1 else "one CTA per item",
                "kv_bytes": full_bytes, "kernel_gbs": full_bytes / (ms_fk * 1e-3) / 1e9,
                "speedup_art_over_full_cache": ms_f / ms}

    # roofline of the decode kernel (bytes actually needed by the blocks processed)
    path = K.art_decode_path(dev.shape, p, dev.workspace.numel())
    kernels = "art_units_kernel + art_units_combine" if path == 1 else "art_decode_kernel"
    peak, peak_kind = load_peaks()
    alg = kv_bytes(w, bu) + side_bytes(w)
    achieved = alg / (ms_kernel * 1e-3) / 1e9
    traffic, traffic_src = load_traffic(w.name, alg, "units" if path == 1 else "one CTA per item")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "frac_of_8tbs": achieved / 8000.0,
                "traffic": traffic, "traffic_source": traffic_src, "peak_kind": peak_kind,
                "kernel": kernels, "path": "units" if path == 1 else "one CTA per item",
                "algorithmic_bytes_per_launch": alg,
                "kernel_ms_per_launch": ms_kernel,
                "kernel_ms_median_min_max": [float(np.median(t_kern)), float(t_kern.min()), float(t_kern.max())],
                "timed": "decode kernel(s) alone, CUDA events recorded by libart around the launch "
                         "(the unit path: the unit kernel and the merge kernel)",
                "call_achieved_gbs": alg / (ms * 1e-3) / 1e9}

    # end to end through the public API with host buffers: per step the step's
    # inputs (queries, lengths, page table, visit lists) go host->device and the
    # outputs (attention output, blocks_used) come back; the KV cache is the
    # device-resident state of the serving engine.
    e2e = None
    if not args.no_e2e:
        host = {}
        for name in ("q", "seq_lens", "block_table", "visit_order"):
            t = getattr(dev, name)
            if t is not None:
                host[name] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())
        out_h = torch.empty(dev.out.shape, dtype=dev.out.dtype, pin_memory=True)
        bu_h = torch.empty(dev.blocks_used.shape, dtype=torch.int32, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_h.numel() * out_h.element_size() + bu_h.numel() * 4

        def e2e_step():
            for name, t in host.items():
                getattr(dev, name).copy_(t, non_blocking=True)
            art_call()
            out_h.copy_(dev.out, non_blocking=True)
            bu_h.copy_(dev.blocks_used, non_blocking=True)

        for _ in range(3):
            e2e_step()
        t_e = time_calls(e2e_step, args.steps)
        ms_e = float(t_e.mean())
        ms_e = max_over_ranks(ms_e, device="cuda")
        e2e = {"value": queries_job / (ms_e * 1e-3), "unit": "queries/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e,
               "note": "KV cache resident on the device; per-step inputs and outputs copied"}

    # the key-based selection that builds this workload's lists, on the device
    selection = None
    sel = w.notes.get("selection")
    if sel is not None:
        T_max = -(-w.max_pages_per_seq * w.page_size // w.block_size)
        mv = min(T_max, int(np.ceil(sel["top_frac"] * T_max)) + 1 + sel["last"])
        sshape = K.make_shape(**dict(w.shape_dict(), max_visit=mv))
        vis = torch.empty((w.batch, w.num_kv_heads, mv), dtype=torch.int32, device="cuda")
        sws = torch.zeros(K.art_select_workspace_bytes(sshape), dtype=torch.uint8, device="cuda")
        sel_call = lambda: K.art_select_blocks(dev.q, dev.k_cache, dev.block_table, dev.seq_lens, sel["top_frac"],
                                               sel["last"], vis, sshape, sws, stream=stream)
        for _ in range(3):
            sel_call()
        ms_s = float(time_calls(sel_call, args.steps).mean())
        host = w.visit_order.reshape(w.num_items, -1)
        got = vis.cpu().numpy().reshape(w.num_items, -1)
        same = sum(int(np.array_equal(got[i][got[i] >= 0], host[i][host[i] >= 0])) for i in range(w.num_items))
        kbytes = int(w.seq_lens.sum()) * w.num_kv_heads * w.head_dim * w.elem_bytes
        selection = {"ms_per_call": ms_s, "k_bytes": kbytes, "gbs": kbytes / (ms_s * 1e-3) / 1e9,
                     "frac_of_peak": kbytes / (ms_s * 1e-3) / 1e9 / peak, "lists_equal_host": f"{same}/{w.num_items}",
                     "note": "art_select_blocks: pooled block scores over all K rows, top fraction + sink + last"}
        # the same kept blocks in importance order (highest score first): the blocks ART reads
        K.art_select_blocks(dev.q, dev.k_cache, dev.block_table, dev.seq_lens, sel["top_frac"], sel["last"], vis,
                            sshape, sws, stream=stream, order=1)
        ishape = K.make_shape(**dict(w.shape_dict(), max_visit=mv))
        iws = torch.zeros(K.art_workspace_bytes(ishape), dtype=torch.uint8, device="cuda")
        bu_imp = torch.empty_like(dev.blocks_used)
        K.art_decode(dev.q, dev.k_cache, dev.v_cache, dev.block_table, dev.seq_lens, vis, eps, eps, p, dev.probe_idx,
                     torch.empty_like(dev.out), bu_imp, ishape, iws, stream)
        torch.cuda.synchronize()
        bi = bu_imp.cpu().numpy().reshape(-1)
        n = w.visit_lengths()
        selection["blocks_used_fraction"] = {"recency_order": float(bu.sum() / max(1, n.sum())),
                                             "importance_order": float(bi.sum() / max(1, n.sum()))}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, eps, p)

    if rank == 0:
        n = w.visit_lengths()
        line = {"metric": "decode-attention queries/s (ART)", "value": value, "unit": "queries/s",
                "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "strong" if sharded else "weak", "vs_baseline": None,
                "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
                "config": config_dict(w_all, eps, p, ws, args.shard),
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks, "e2e": e2e,
                "gpu_launches": (3 if path == 1 else 2) * args.steps,
                "dense_twin": dense,
                "selection": selection,
                "blocks_used": {"mean": float(bu.mean()), "listed_mean": float(n.mean()),
                                "fraction": float(bu.sum() / max(1, n.sum()))},
                "status": status}
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# diagnostics: convergence of O^(t) and attention score vs value contribution
# ---------------------------------------------------------------------------
def _ranks(x):
    r = np.empty(x.size, dtype=np.float64)
    r[np.argsort(x, kind="stable")] = np.arange(x.size)
    return r


def score_vs_contribution(w, items, top=0.01):
    """Per sampled item, over its tokens t: the attention score a_t = max over the
    group's query heads of the softmax weight alpha_{h,t}, and the contribution
    c_t = max over those heads of |alpha_{h,t} v_t|_2 (the norm of token t's term in
    the head's output) -- the two rankings the ART paper compares (sec. 1, Fig. 1).
    Returns the Spearman rank correlation of a and c, the share of the top `top`
    tokens by contribution that are also in the top `top` by score, and the same
    share restricted to tokens of the value-boosted blocks."""
    G, d = w.group, w.head_dim
    rho, overlap, boosted_hit = [], [], []
    for it in items:
        b, g = divmod(int(it), w.num_kv_heads)
        N = int(w.seq_lens[b])
        toks = np.arange(N)
        pg, row = w.block_table[b, toks // w.page_size], toks % w.page_size
        kk = W.as_f32(w.k_cache[pg, g, row, :], w.dtype).astype(np.float64)
        vv = W.as_f32(w.v_cache[pg, g, row, :], w.dtype).astype(np.float64)
        qq = W.as_f32(w.q[b, g * G:(g + 1) * G], w.dtype).astype(np.float64)
        s = qq @ kk.T / np.sqrt(d)
        a = np.exp(s - s.max(axis=1, keepdims=True))
        a /= a.sum(axis=1, keepdims=True)
        vn = np.linalg.norm(vv, axis=1)
        score = a.max(axis=0)
        contrib = (a * vn[None, :]).max(axis=0)
        rs, rc = _ranks(score), _ranks(contrib)
        rho.append(float(np.corrcoef(rs, rc)[0, 1]))
        k = max(1, int(round(top * N)))
        ts, tc = set(np.argsort(-score)[:k].tolist()), np.argsort(-contrib)[:k]
        overlap.append(len(ts.intersection(tc.tolist())) / k)
        big = vn > 2.0 * np.median(vn)  # the x8 blocks
        tcb = [t for t in tc.tolist() if big[t]]
        if tcb:
            boosted_hit.append(sum(t in ts for t in tcb) / len(tcb))
    return {"items": [int(i) for i in items], "spearman_score_vs_contribution": float(np.mean(rho)),
            "top_frac": top, "top_overlap": float(np.mean(overlap)),
            "boosted_top_contrib_share_in_top_score": float(np.mean(boosted_hit)) if boosted_hit else None}


def run_diag(args):
    """The convergence curve: rel-L2(O^(t), O^(T)) against the loaded fraction t / n
    of the visit list (sink first, then most recent first), per item, binned; O^(t)
    from libart forced to stop after t blocks (eps = +inf, patience t - 1), O^(T)
    from the dense twin. Then the ART stop at eps 1e-3, patience 2, and the score
    versus contribution ranks on the ragged workload."""
    import torch

    import kv_cache_early_gb300 as K
    from kv_cache_early_gb300 import build as B
    B.build()
    torch.cuda.set_device(0)
    res = {"diag": "convergence of O^(t) and score vs contribution", "configs": {}}
    for cfg in (2, 4):
        w = W.config(cfg)
        dev = K.DeviceInputs(w)
        n = w.visit_lengths()
        shp = (w.num_items, w.group * w.head_dim)
        dev.dense()
        torch.cuda.synchronize()
        OT = dev.out.float().cpu().numpy().reshape(shp).astype(np.float64)
        nT = np.linalg.norm(OT, axis=1)
        fr, rel = [], []
        t = 2
        while t <= int(n.max()):
            dev.art(float("inf"), float("inf"), t - 1)
            torch.cuda.synchronize()
            bu = dev.blocks_used.cpu().numpy().reshape(-1)
            assert (bu == np.minimum(n, t)).all(), "forced stop"
            Ot = dev.out.float().cpu().numpy().reshape(shp).astype(np.float64)
            live = n >= t  # items whose list is not yet exhausted
            fr.append((t / n)[live])
            rel.append((np.linalg.norm(Ot - OT, axis=1) / nT)[live])
            t *= 2
        fr, rel = np.concatenate(fr), np.concatenate(rel)
        edges = [0.0, 1 / 64, 1 / 32, 1 / 16, 1 / 8, 1 / 4, 1 / 2, 1.0001]
        curve = []
        for lo, hi in zip(edges, edges[1:]):
            m = (fr > lo) & (fr <= hi)
            if m.any():
                curve.append({"loaded_frac": [lo, min(hi, 1.0)], "points": int(m.sum()),
                              "rel_l2_median": float(np.median(rel[m])), "rel_l2_p90": float(np.percentile(rel[m], 90))})
        dev.art(1e-3, 1e-3, 2)
        torch.cuda.synchronize()
        bu = dev.blocks_used.cpu().numpy().reshape(-1)
        Oa = dev.out.float().cpu().numpy().reshape(shp).astype(np.float64)
        ra = np.linalg.norm(Oa - OT, axis=1) / nT
        entry = {"workload": w.name, "curve": curve,
                 "art_eps1e-3_p2": {"loaded_frac_mean": float((bu / n).mean()),
                                    "rel_l2_median": float(np.median(ra)), "rel_l2_max": float(ra.max())}}
        if cfg == 4:
            rng = np.random.default_rng(0)
            entry["score_vs_contribution"] = score_vs_contribution(
                w, np.sort(rng.choice(w.num_items, size=8, replace=False)))
        res["configs"][str(cfg)] = entry
        del dev
        torch.cuda.empty_cache()
    print(json.dumps(res))


def main():
    args = parse()
    if args.diag:
        run_diag(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
