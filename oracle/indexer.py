"""Hierarchical sparse indexer: Full (scan + shared candidate pool + Top-k),
Reindex (re-score the pool) and Reuse (no indexer).

Test infrastructure (see oracle/__init__.py).

[deep-dive §3.1] Indexer Q x Indexer K -> score -> Top-K.
[deep-dive §3.2] Full: fresh Main KV / Indexer K, fresh Top-K.  Reindex: reuse the
                 earlier Main KV and Indexer K, score with this layer's own Indexer Q.
                 Reuse: reuse Main KV and Top-K; no indexer runs.
[deep-dive §3.3] The first Full indexer scans the whole causally visible range and
                 keeps the best positions of every block; 2,048 blocks x 8 positions
                 = a 16,384-entry shared candidate pool; Reindex layers score only the
                 pool and each picks its own Top-512; Reuse layers take the most recent
                 Top-512.  The search range stays 16,384 whatever the context length.
[paper-reading §4.2] mode table (same three modes).
"""
import numpy as np


def scores(q, w, K, relu=True):
    """s(e) = sum_h w_h * ReLU(q_h . K_e)  (float64).

    READING: the pages only say "Indexer Q x Indexer K -> score" [deep-dive §3.1].
    With several indexer heads (32 x 128 in [deep-dive §6.3]) a plain sum of q_h . k
    would collapse to one head, so the score is the per-query head-weighted sum of
    ReLU'd head dot products (the form of DeepSeek's earlier sparse indexer); the
    weights w are a per-query input.  relu=False gives the literal weighted dot sum.

    q: [H, dk], w: [H], K: [n, dk]  ->  [n]
    """
    q = np.asarray(q, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    dots = K @ q.T                        # [n, H]
    if relu:
        dots = np.maximum(dots, 0.0)
    return dots @ w


def block_bounds(n, num_blocks):
    """Block b of the visible range [0, n) is [floor(b*n/NB), floor((b+1)*n/NB)).

    READING: the block size is not printed; NB balanced blocks is the one partition
    under which the pool is exactly NB*per_block entries for every n >= NB*per_block
    ("search range fixed at 16,384", [deep-dive §3.3]) and covers the whole range when
    n is smaller."""
    b = np.arange(num_blocks + 1, dtype=np.int64)
    return (b * n) // num_blocks


def top_positions(s, k):
    """Positions of the k best values of s, best = larger score, equal scores going
    to the lower position (ties break to the lower index).  Returned in ascending
    position order (the canonical order of every index set here)."""
    s = np.asarray(s, dtype=np.float64)
    k = min(int(k), len(s))
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    pos = np.arange(len(s))
    order = np.lexsort((pos, -s))         # primary: score descending; then position
    return np.sort(order[:k])


def full(q, w, K, num_blocks, per_block, k, relu=True):
    """Full mode over the visible entries K[0:n] [deep-dive §3.3 step 1-2]:
    score every entry, keep the top min(per_block, len) of each block, the union in
    ascending entry order is the pool, and Top-k is taken from the pool (READING,
    as stated for this build: Full's Top-k comes from its own pool).

    Returns (pool int64[pool_len] ascending, topk int64[<=k] ascending, s float64[n]).
    """
    n = len(K)
    s = scores(q, w, K, relu) if n else np.zeros(0)
    bb = block_bounds(n, num_blocks)
    parts = []
    for b in range(num_blocks):
        lo, hi = bb[b], bb[b + 1]
        if hi > lo:
            parts.append(lo + top_positions(s[lo:hi], min(per_block, hi - lo)))
    pool = np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)
    topk = pool[top_positions(s[pool], k)] if len(pool) else pool
    return pool, topk, s


def reindex(q, w, K, pool, k, relu=True):
    """Reindex mode [deep-dive §3.3 step 3]: this layer's own indexer Q scores only the
    shared pool (entries of the Main KV / Indexer K cache built by the Full layer) and
    picks its own Top-k.  Returns (topk ascending, pool scores)."""
    pool = np.asarray(pool, dtype=np.int64)
    if len(pool) == 0:
        return pool, np.zeros(0)
    s = scores(q, w, np.asarray(K)[pool], relu)
    return pool[top_positions(s, k)], s


def reuse(previous_topk):
    """Reuse mode [deep-dive §3.2]: no indexer; the most recent Top-k is used as is."""
    return np.asarray(previous_topk).copy()


def fp8_form(q, K8, Ks):
    """The compressed (FP8) indexer: the values it scores.

    READING (not on the pages; the pages keep indexer K in the form Main KV implies): each
    entry's bf16 indexer K row is stored as E4M3 bytes K8 with one float32 scale Ks =
    amax / 448 (formats.fp8_rows_quantize), and each query head's bf16 indexer Q row is
    quantised the same way at scoring time, as FP8 indexers do.  The scores are then those
    of scores() / full() / reindex() over the dequantised values of both.

    q: [H, dk] float values of the bf16 indexer Q; K8: [n, dk] uint8; Ks: [n] float32.
    Returns (q_hat [H, dk], K_hat [n, dk]) in float64, both exact.
    """
    from . import formats
    q8, qs = formats.fp8_rows_quantize(np.asarray(q, dtype=np.float32))
    return formats.fp8_rows_dequantize(q8, qs), formats.fp8_rows_dequantize(K8, Ks)
