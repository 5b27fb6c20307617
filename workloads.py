"""Seeded synthetic inputs for ART decode attention.

This module only draws and lays out inputs: queries, a paged K/V cache, block
tables, sequence lengths, visit lists and probe indices. It holds none of the
attention or termination arithmetic, and both the CUDA path and the CPU oracle
read the arrays it returns.

Values are drawn in float32 with numpy's PCG64 and rounded once to the working
dtype (bf16 round-to-nearest-even, kept as raw uint16 bits, or fp32); both
sides read exactly those values. Large arrays are drawn in fixed-size chunks,
each from its own child seed, so the result does not depend on the number of
threads used to draw them.

The five named workloads follow the decode configurations of the ART pages
(batch serving of Llama-3-8B / Mistral-7B / Llama-3.1-70B style layers on a
paged KV cache) with synthetic data standing in for LongBench prompts and
trained weights, which are not available here.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

CHUNK = 1 << 22  # elements per independently seeded draw


# ----------------------------------------------------------------------------
# dtype helpers
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_working(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    return np.ascontiguousarray(x, dtype=np.float32)


def as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


def _fill_normal(out: np.ndarray, seed_seq: np.random.SeedSequence, dtype: str, threads: int) -> None:
    """Fill `out` (flat view, working dtype) with N(0,1) drawn chunk by chunk."""
    flat = out.reshape(-1)
    n = flat.size
    nchunks = (n + CHUNK - 1) // CHUNK
    kids = seed_seq.spawn(nchunks)

    def work(i):
        lo, hi = i * CHUNK, min(n, (i + 1) * CHUNK)
        r = np.random.default_rng(kids[i])
        v = r.standard_normal(hi - lo, dtype=np.float32)
        flat[lo:hi] = to_working(v, dtype)

    if threads <= 1 or nchunks == 1:
        for i in range(nchunks):
            work(i)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(nchunks)))


# ----------------------------------------------------------------------------
# the workload container
# ----------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    dtype: str  # "bf16" or "f32"
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    block_size: int
    seq_lens: np.ndarray  # int32 [B]
    block_table: np.ndarray  # int32 [B, max_pages_per_seq]
    visit_order: Optional[np.ndarray]  # int32 [B, Hkv, max_visit], -1 terminated; None = natural
    q: np.ndarray  # [B, Hq, d]
    k_cache: np.ndarray  # [num_pages, Hkv, page_size, d]
    v_cache: np.ndarray
    probe_idx: np.ndarray  # int32 [m]
    eps_mag: float = 1e-3
    eps_dir: float = 1e-3
    patience: int = 2
    notes: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def num_items(self) -> int:
        return self.batch * self.num_kv_heads

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_visit(self) -> int:
        if self.visit_order is None:
            return int(max(1, -(-int(self.seq_lens.max(initial=0)) // self.block_size)))
        return int(self.visit_order.shape[2])

    @property
    def num_probe(self) -> int:
        return int(self.probe_idx.shape[0])

    @property
    def num_pages_total(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def shape_dict(self) -> dict:
        return dict(batch=self.batch, num_q_heads=self.num_q_heads, num_kv_heads=self.num_kv_heads,
                    head_dim=self.head_dim, page_size=self.page_size, block_size=self.block_size,
                    max_pages_per_seq=self.max_pages_per_seq, max_visit=self.max_visit,
                    num_probe=self.num_probe, num_pages_total=self.num_pages_total,
                    dtype=0 if self.dtype == "bf16" else 1)

    def visit_lengths(self) -> np.ndarray:
        """Number of listed blocks per item (b * Hkv + g)."""
        T = -(-self.seq_lens.astype(np.int64) // self.block_size)
        if self.visit_order is None:
            return np.repeat(T, self.num_kv_heads).astype(np.int64)
        vo = self.visit_order.reshape(self.num_items, -1)
        neg = vo == -1
        first = np.where(neg.any(axis=1), neg.argmax(axis=1), vo.shape[1])
        return first.astype(np.int64)

    def block_tokens(self, b: int, c: int) -> int:
        return int(max(0, min(self.block_size, int(self.seq_lens[b]) - c * self.block_size)))


# ----------------------------------------------------------------------------
# builders
# ----------------------------------------------------------------------------
def _orders(kind: str, T: int, rng: np.random.Generator) -> np.ndarray:
    if kind == "natural":
        return np.arange(T, dtype=np.int32)
    if kind == "sink_recent":  # block 0 (the sink) first, then most recent first
        return np.concatenate([[0], np.arange(T - 1, 0, -1)]).astype(np.int32) if T > 0 else np.zeros(0, np.int32)
    if kind == "reverse":  # most recent first, block 0 last
        return np.arange(T - 1, -1, -1, dtype=np.int32)
    if kind == "random":
        return rng.permutation(T).astype(np.int32)
    raise ValueError(kind)


def build(name: str, *, seed: int, dtype: str, batch: int, num_q_heads: int, num_kv_heads: int,
          head_dim: int, page_size: int, block_size: int, seq_lens, paged: str = "identity",
          plant: bool = False, v_boost_frac: float = 0.0, v_boost: float = 8.0,
          order: Optional[str] = "sink_recent", selection: Optional[dict] = None,
          eps_mag: float = 1e-3, eps_dir: float = 1e-3, patience: int = 2, probe_stride: int = 4,
          kv_const_v: Optional[float] = None, identical_keys: bool = False,
          threads: Optional[int] = None) -> Workload:
    """Draw one workload. Generation order: q, K, V, page permutation, planting,
    value boosts, visit lists."""
    threads = threads if threads is not None else min(16, os.cpu_count() or 1)
    ss = np.random.SeedSequence(seed)
    s_q, s_k, s_v, s_rest = ss.spawn(4)
    seq_lens = np.asarray(seq_lens, dtype=np.int32).reshape(batch)
    G = num_q_heads // num_kv_heads
    d = head_dim
    pages_per_seq = -(-seq_lens.astype(np.int64) // page_size)
    max_pages = int(max(1, pages_per_seq.max(initial=1)))

    # physical pool
    if paged == "identity":
        num_pages = batch * max_pages
    elif paged == "permuted":
        num_pages = int(pages_per_seq.sum())
    else:
        raise ValueError(paged)
    num_pages = max(num_pages, 1)
    np_dtype = np.uint16 if dtype == "bf16" else np.float32

    q = np.empty((batch, num_q_heads, d), dtype=np_dtype)
    _fill_normal(q, s_q, dtype, 1)
    k_cache = np.empty((num_pages, num_kv_heads, page_size, d), dtype=np_dtype)
    v_cache = np.empty_like(k_cache)
    if identical_keys:
        k_cache[...] = 0
    else:
        _fill_normal(k_cache, s_k, dtype, threads)
    if kv_const_v is not None:
        v_cache[...] = to_working(np.full(d, kv_const_v, np.float32), dtype)
    else:
        _fill_normal(v_cache, s_v, dtype, threads)

    rng = np.random.default_rng(s_rest)

    # logical page -> physical page
    block_table = np.full((batch, max_pages), -1, dtype=np.int32)
    if paged == "identity":
        for b in range(batch):
            block_table[b, : pages_per_seq[b]] = b * max_pages + np.arange(pages_per_seq[b])
    # (permuted tables are filled after planting, see below)

    def phys_rows(b: int, toks: np.ndarray, table: np.ndarray):
        return table[b, toks // page_size], toks % page_size

    # planting is done against the final table, so draw the permutation first when paged
    if paged == "permuted":
        perm = rng.permutation(num_pages).astype(np.int32)
        off = 0
        for b in range(batch):
            block_table[b, : pages_per_seq[b]] = perm[off: off + pages_per_seq[b]]
            off += int(pages_per_seq[b])

    qf = as_f32(q, dtype).astype(np.float64)
    if plant:
        for b in range(batch):
            N = int(seq_lens[b])
            if N <= 0:
                continue
            for g in range(num_kv_heads):
                qbar = qf[b, g * G:(g + 1) * G].mean(axis=0)
                u = qbar / np.linalg.norm(qbar)
                toks = [np.arange(min(4, N))]
                toks.append(np.arange(max(0, N - 256), N))
                starts = rng.integers(0, max(0, N - 32), size=16, endpoint=True)
                for s0 in starts:
                    toks.append(np.arange(s0, min(N, s0 + 32)))
                toks = np.unique(np.concatenate(toks))
                noise = rng.normal(0.0, 0.5, size=(toks.size, d)).astype(np.float32)
                kk = (3.0 * u[None, :]).astype(np.float32) + noise
                pg, row = phys_rows(b, toks, block_table)
                k_cache[pg, g, row, :] = to_working(kk, dtype)

    if v_boost_frac > 0.0:
        Tmax = int(-(-int(seq_lens.max()) // block_size))
        sel = rng.random((batch, num_kv_heads, Tmax)) < v_boost_frac
        for b, g, c in zip(*np.nonzero(sel)):
            N = int(seq_lens[b])
            lo, hi = c * block_size, min(N, (c + 1) * block_size)
            if lo >= hi:
                continue
            toks = np.arange(lo, hi)
            pg, row = phys_rows(b, toks, block_table)
            vv = as_f32(v_cache[pg, g, row, :], dtype) * np.float32(v_boost)
            v_cache[pg, g, row, :] = to_working(vv, dtype)

    # visit lists
    T_b = -(-seq_lens.astype(np.int64) // block_size)
    visit_order = None
    notes = {}
    if selection is not None:
        # key-based selection of kept blocks (the KV manager's job, upstream of ART):
        # pooled score mean_h(q_h) . mean_{t in block}(k_t), top fraction, plus the
        # sink block and the last `last` blocks; visit order: 0 first, then by
        # descending block index (most recent first).
        frac, last = selection.get("top_frac", 0.25), selection.get("last", 8)
        lists = []
        for b in range(batch):
            T = int(T_b[b])
            N = int(seq_lens[b])
            for g in range(num_kv_heads):
                qbar = qf[b, g * G:(g + 1) * G].mean(axis=0)
                toks = np.arange(N)
                pg, row = phys_rows(b, toks, block_table)
                kk = as_f32(k_cache[pg, g, row, :], dtype).astype(np.float64)
                sums = np.add.reduceat(kk, np.arange(0, N, block_size), axis=0)
                cnt = np.minimum(block_size, N - np.arange(T) * block_size)[:, None]
                score = (sums / cnt) @ qbar
                kth = int(np.ceil(frac * T))
                top = np.lexsort((np.arange(T), -score))[:kth]  # ties by lower index
                keep = set(top.tolist()) | {0} | set(range(max(0, T - last), T))
                rest = sorted((c for c in keep if c != 0), reverse=True)
                lists.append([0] + rest if 0 in keep else rest)
        mv = max(len(x) for x in lists)
        visit_order = np.full((batch, num_kv_heads, mv), -1, dtype=np.int32)
        for i, lst in enumerate(lists):
            visit_order[i // num_kv_heads, i % num_kv_heads, : len(lst)] = lst
        notes["selection"] = dict(top_frac=frac, last=last)
    elif order is not None:
        mv = int(max(1, T_b.max(initial=1)))
        visit_order = np.full((batch, num_kv_heads, mv), -1, dtype=np.int32)
        for b in range(batch):
            for g in range(num_kv_heads):
                lst = _orders(order, int(T_b[b]), rng)
                visit_order[b, g, : lst.size] = lst

    probe_idx = np.arange(0, d, probe_stride, dtype=np.int32)
    return Workload(name=name, dtype=dtype, batch=batch, num_q_heads=num_q_heads,
                    num_kv_heads=num_kv_heads, head_dim=d, page_size=page_size,
                    block_size=block_size, seq_lens=seq_lens, block_table=block_table,
                    visit_order=visit_order, q=q, k_cache=k_cache, v_cache=v_cache,
                    probe_idx=probe_idx, eps_mag=eps_mag, eps_dir=eps_dir, patience=patience,
                    notes=notes)


# ----------------------------------------------------------------------------
# the five decode workloads (full size) and their scaled-down parity versions
# ----------------------------------------------------------------------------
CONFIG_NAMES = {
    1: "tiny-fp32-b1-h1-d64-n1024",
    2: "llama3-8b-layer-bf16-b16-gqa32x8-d128-ctx32768",
    3: "paged-bf16-b128-gqa32x8-d128-ctx8192-page16",
    4: "ragged-bf16-b64-gqa32x8-d128-ctx1k-64k-page16",
    5: "longctx-select-bf16-b4-gqa28x4-d128-ctx131072",
}


def config(k: int, *, small: bool = False, eps: Optional[float] = None, patience: Optional[int] = None,
           threads: Optional[int] = None, batch: Optional[int] = None) -> Workload:
    """Workload k (1..5). `small=True` keeps the structure at a size the oracle
    finishes in seconds (several ART blocks, ragged tails, paged tables).
    `batch` replaces the batch of a full-size config 2..5 (same shapes and
    seeds otherwise; for smaller profiler captures of the same kernel); the
    workload name then carries the new batch."""
    e = 1e-3 if eps is None else eps
    p = 2 if patience is None else patience
    if batch is not None and (small or k == 1 or batch < 1):
        raise ValueError("a batch override applies to the full-size configs 2..5")

    def name(B0, B):
        n = CONFIG_NAMES[k] + ("-small" if small else "")
        return n if batch is None else n.replace(f"-b{B0}-", f"-b{B}-")

    if k == 1:
        return build(CONFIG_NAMES[1], seed=1, dtype="f32", batch=1, num_q_heads=1, num_kv_heads=1,
                     head_dim=64, page_size=64, block_size=64, seq_lens=[1024], paged="identity",
                     order=None, eps_mag=e, eps_dir=e, patience=p, threads=threads)
    if k == 2:
        B, N = (2, 2000) if small else (batch or 16, 32768)
        return build(name(16, B), seed=2, dtype="bf16", batch=B,
                     num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64, block_size=64,
                     seq_lens=[N] * B, paged="identity", plant=True, order="sink_recent",
                     eps_mag=e, eps_dir=e, patience=p, threads=threads)
    if k == 3:
        B, N = (3, 1000) if small else (batch or 128, 8192)
        return build(name(128, B), seed=3, dtype="bf16", batch=B,
                     num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, block_size=64,
                     seq_lens=[N] * B, paged="permuted", plant=True, order="sink_recent",
                     eps_mag=e, eps_dir=e, patience=p, threads=threads)
    if k == 4:
        rs = np.random.default_rng(np.random.SeedSequence([4, 1]))
        if small:
            B = 4
            lens = rs.integers(64, 3000, size=B, endpoint=True)
        else:
            B = batch or 64
            lens = rs.integers(1024, 65536, size=B, endpoint=True)
        return build(name(64, B), seed=4, dtype="bf16", batch=B,
                     num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, block_size=64,
                     seq_lens=lens, paged="permuted", v_boost_frac=0.05, v_boost=8.0,
                     order="sink_recent", eps_mag=e, eps_dir=e, patience=p, threads=threads)
    if k == 5:
        B, N = (2, 4096) if small else (batch or 4, 131072)
        return build(name(4, B), seed=5, dtype="bf16", batch=B,
                     num_q_heads=28, num_kv_heads=4, head_dim=128, page_size=64, block_size=64,
                     seq_lens=[N] * B, paged="identity", plant=True,
                     selection=dict(top_frac=0.25, last=8), eps_mag=e, eps_dir=e, patience=p,
                     threads=threads)
    raise ValueError(k)


CONFIG4_GRID = [(e, p) for e in (0.0, 1e-3, 1e-2) for p in (1, 2, 4)]


# ----------------------------------------------------------------------------
# partition by sequence (one GPU per shard; no exchange between shards)
# ----------------------------------------------------------------------------
def shard_range(batch: int, rank: int, world: int) -> tuple:
    """Sequences [lo, hi) of shard `rank` of `world`: contiguous, sizes differing by
    at most one, every sequence in exactly one shard."""
    if not (1 <= world <= batch and 0 <= rank < world):
        raise ValueError(f"{world} shards of a batch of {batch}")
    return rank * batch // world, (rank + 1) * batch // world


def shard_sequences(w: Workload, rank: int, world: int) -> Workload:
    """The shard of `w` that owns sequences [lo, hi) (shard_range): their queries,
    lengths, visit lists and block-table rows, and the pages those rows name,
    gathered into a pool of their own (table entries renumbered in order of first
    use). Items (b, g) of the shard are items (lo + b, g) of `w`."""
    lo, hi = shard_range(w.batch, rank, world)
    table = w.block_table[lo:hi]
    pages_per_seq = -(-w.seq_lens[lo:hi].astype(np.int64) // w.page_size)
    used = np.concatenate([table[i, : pages_per_seq[i]] for i in range(hi - lo)]) if hi > lo else \
        np.zeros(0, np.int32)
    phys, first = np.unique(used, return_index=True)
    phys = phys[np.argsort(first, kind="stable")]  # order of first use
    remap = {int(pg): i for i, pg in enumerate(phys)}
    new_table = np.full_like(table, -1)
    for i in range(hi - lo):
        new_table[i, : pages_per_seq[i]] = [remap[int(x)] for x in table[i, : pages_per_seq[i]]]
    k_cache = np.ascontiguousarray(w.k_cache[phys]) if phys.size else w.k_cache[:1].copy()
    v_cache = np.ascontiguousarray(w.v_cache[phys]) if phys.size else w.v_cache[:1].copy()
    notes = dict(w.notes, shard=dict(rank=rank, world=world, lo=lo, hi=hi))
    return Workload(name=f"{w.name}-shard{rank}of{world}", dtype=w.dtype, batch=hi - lo,
                    num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                    page_size=w.page_size, block_size=w.block_size,
                    seq_lens=np.ascontiguousarray(w.seq_lens[lo:hi]), block_table=new_table,
                    visit_order=None if w.visit_order is None else np.ascontiguousarray(w.visit_order[lo:hi]),
                    q=np.ascontiguousarray(w.q[lo:hi]), k_cache=k_cache, v_cache=v_cache,
                    probe_idx=w.probe_idx, eps_mag=w.eps_mag, eps_dir=w.eps_dir, patience=w.patience,
                    notes=notes)
