"""CPU oracle of key-based block selection -- TEST INFRASTRUCTURE.

Only the test suite and the benchmark may import this module; the CUDA path
never does, and the two share no code.

Definition (the pooled block estimate of the FlexPrefill summary, used as
the key-centric KV selection that ART is composed with in the ART paper,
sec. 4), in fp64 on the exact bf16 / fp32 input values, for every item
(sequence b, KV head g) with T = ceil(seq_len / block_size) blocks:

    qbar    = the mean of the G query vectors of KV head g
    kbar_c  = the mean of the key rows t < seq_len of block c (through the
              block table)
    score_c = qbar . kbar_c
    kept    = the ceil(top_frac * T) highest scores (equal scores: lower
              block index first), block 0, the last keep_last blocks
    list    = [0] + the other kept blocks in descending index order (recency),
              or by descending score, equal scores lower index first (importance)

Each step is written out with plain loops over blocks and rows.
"""
from __future__ import annotations

import math

import numpy as np


def _as_f64(a, dtype):
    if dtype == "bf16":
        bits = np.asarray(a).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def block_scores(q, k_cache, block_table, seq_len, b, g, *, num_q_heads, num_kv_heads, page_size, block_size,
                 dtype):
    """score_c for c < T of item (b, g), fp64."""
    G = num_q_heads // num_kv_heads
    qbar = np.zeros(q.shape[-1], np.float64)
    for h in range(G):
        qbar += _as_f64(q[b, g * G + h], dtype)
    qbar /= G
    T = (int(seq_len) + block_size - 1) // block_size
    scores = np.zeros(T, np.float64)
    for c in range(T):
        lo, hi = c * block_size, min((c + 1) * block_size, int(seq_len))
        ksum = np.zeros(q.shape[-1], np.float64)
        for t in range(lo, hi):
            page = int(block_table[b, t // page_size])
            ksum += _as_f64(k_cache[page, g, t % page_size], dtype)
        scores[c] = float(np.dot(qbar, ksum / (hi - lo)))
    return scores


def kept_list(scores, top_frac: float, keep_last: int, order: str = "recency"):
    """The visit list from one item's scores."""
    T = len(scores)
    if T == 0:
        return []
    k = min(T, math.ceil(top_frac * T))
    ranked = sorted(range(T), key=lambda c: (-scores[c], c))
    kept = set(ranked[:k]) | {0} | set(range(max(0, T - keep_last), T))
    if order == "importance":
        return [0] + [c for c in ranked if c in kept and c != 0]
    return [0] + sorted((c for c in kept if c != 0), reverse=True)


def select_blocks(w, top_frac: float, keep_last: int, items=None, order: str = "recency"):
    """Lists and scores for a workloads.Workload (all items, or `items`)."""
    items = range(w.num_items) if items is None else items
    out = {}
    for it in items:
        b, g = divmod(int(it), w.num_kv_heads)
        sc = block_scores(w.q, w.k_cache, w.block_table, w.seq_lens[b], b, g, num_q_heads=w.num_q_heads,
                          num_kv_heads=w.num_kv_heads, page_size=w.page_size, block_size=w.block_size,
                          dtype=w.dtype)
        out[int(it)] = (kept_list(sc, top_frac, keep_last, order), sc)
    return out
