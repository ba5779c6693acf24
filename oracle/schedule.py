"""Static layer schedules and a whole decode step over them.

Test infrastructure (see oracle/__init__.py).

[deep-dive §3.2] Encoder (20 layers): layers 1-2 SWA only, then 3 groups of
                 [Full x1 + Reuse x5] at ratio 2.  Decoder (20 layers): group 1 is
                 [Full x1 + Reuse x3], groups 2-5 are [Reindex x1 + Reuse x3], ratio 1.
[deep-dive §3.3] the pool is created by the decoder's first Full layer and shared by
                 the Reindex layers; Reuse layers use the most recent Top-512.
"""
import numpy as np

from . import attention, indexer

FULL, REINDEX, REUSE = "full", "reindex", "reuse"


def decoder_schedule():
    return [FULL, REUSE, REUSE, REUSE] + [REINDEX, REUSE, REUSE, REUSE] * 4


def encoder_schedule():
    """Layers 3..20 of the encoder (layers 1-2 are SWA-only)."""
    return ([FULL] + [REUSE] * 5) * 3


def decode_step(layers, K_idx, codes, scales, num_blocks, per_block, k, tau, relu=True):
    """One decode query through a schedule.

    layers[l] = dict(q_idx [H_i, dk] (Full/Reindex), w [H_i], q [Hq, d],
                     swa_rows, swa_scale, swa_start, swa_len)
    K_idx / codes / scales: the query's sequence, entries [0, n) in entry order.
    Returns list of (mode, topk, out, lse) per layer.
    """
    sched = [L["mode"] for L in layers]
    pool = None
    topk = None
    res = []
    for L, mode in zip(layers, sched):
        if mode == FULL:
            pool, topk, _ = indexer.full(L["q_idx"], L["w"], K_idx, num_blocks, per_block, k, relu)
        elif mode == REINDEX:
            topk, _ = indexer.reindex(L["q_idx"], L["w"], K_idx, pool, k, relu)
        else:
            topk = indexer.reuse(topk)
        out, lse = attention.sparse_attention(L["q"], codes, scales, topk, L["swa_rows"],
                                              L["swa_scale"], L["swa_start"], L["swa_len"], tau)
        res.append((mode, np.asarray(topk), out, lse))
    return res
