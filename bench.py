#!/usr/bin/env python3
"""Benchmark of ART decode attention on one decode workload.

One step = one art_decode call (memset of the workspace header, the plan
kernel, the persistent decode kernel) over the whole batch, inputs resident
in HBM. Prints one JSON line (rank 0) with queries/s, the HBM roofline of the
decode kernel, the dense twin, the CPU oracle baseline, clocks and an
end-to-end figure through the public API with host buffers.

Default workload: the Llama-3-8B-shaped decode layer (batch 16, 32 query /
8 KV heads, d=128, 32768-token context, bf16, KV block 64, planted keys,
sink-first most-recent-first order, eps 1e-3, patience 2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 1..5] [--eps E] [--patience P] [--no-cpu-baseline]
Under torchrun (N > 1) every rank runs its own independently seeded copy of
the workload (weak scaling, no collective on the data path); the timing is
the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
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
    ap.add_argument("--config", type=int, default=2)
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
def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_early_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(csrc, f), "rb").read())
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
    if not e or e.get("kernel_hash") != kernel_source_hash() or e.get("path") != path:
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


def config_dict(w, eps, p, ws):
    return {"workload": w.name, "batch": w.batch, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "page_size": w.page_size, "block_size": w.block_size, "eps": eps,
            "patience": p, "l2": "flushed (256 MB write) before every timed call; inputs also exceed L2",
            "parallelism": f"{ws} independent replicas" if ws > 1 else "single GPU"}


# ---------------------------------------------------------------------------
# reference arm: the oracle timed as it stands on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    w = W.config(args.config, eps=args.eps, patience=args.patience, batch=args.batch)
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
    w = W.config(args.config, eps=args.eps, patience=args.patience, batch=args.batch)  # one replica per rank
    eps, p = w.eps_mag, w.patience
    dev = K.DeviceInputs(w)
    queries = w.batch * w.num_q_heads
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
    value = ws * queries / (ms * 1e-3)

    # dense twin on the same buffers
    dense = None
    if not args.no_dense:
        for _ in range(max(3, args.warmup)):
            dense_call()
        t_d, t_dk = time_calls(dense_call, args.steps, kernel=True)
        ms_d, ms_dk = float(t_d.mean()), float(t_dk.mean())
        dense = {"queries_per_s": queries / (ms_d * 1e-3), "ms_per_step": ms_d, "kernel_ms": ms_dk,
                 "path": "units" if K.art_decode_path(dev.shape, 1, dev.workspace.numel()) == 1
                 else "one CTA per item",
                 "kernel_gbs": (kv_bytes(w) + side_bytes(w)) / (ms_dk * 1e-3) / 1e9,
                 "speedup_art_over_dense": ms_d / ms}
        # the detector's own cost: ART with eps = 0 never stops
        zero = lambda: dev.art(0.0, 0.0, p, stream=stream)
        for _ in range(3):
            zero()
        ms_z = float(time_calls(zero, args.steps).mean())
        dense["art_eps0_ms_per_step"] = ms_z
        dense["detector_overhead_frac"] = ms_z / ms_d - 1.0

    # roofline of the decode kernel (bytes actually needed by the blocks processed)
    path = K.art_decode_path(dev.shape, p, dev.workspace.numel())
    kernels = "art_units_kernel + art_units_combine" if path == 1 else "art_decode_kernel"
    peak, peak_kind = load_peaks()
    alg = kv_bytes(w, bu) + side_bytes(w)
    achieved = alg / (ms_kernel * 1e-3) / 1e9
    traffic, traffic_src = load_traffic(w.name, alg, "units" if path == 1 else "one CTA per item")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
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
        e2e = {"value": ws * queries / (ms_e * 1e-3), "unit": "queries/s", "h2d_bytes_per_step": int(h2d),
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
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
                "config": config_dict(w, eps, p, ws),
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


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
