"""Sparse MQA attention of one query over the selected FP4 Main KV entries plus the
layer-local FP8 SWA window, in one softmax.

Test infrastructure (see oracle/__init__.py).

[deep-dive §3.1] Main Q attends to (selected Main KV + layer-local SWA KV) -> output;
                 every layer keeps its own Main Q and SWA KV.
[leak-digest]    the selected entries and the windowed KV are concatenated and enter
                 one attention.
[deep-dive §6.3] 64 query heads x 512 dims, SWA window n_win = 128, Top-K = 512.
"""
import math

import numpy as np

from . import formats


def gather_rows(codes_cache, scales_cache, topk, swa_rows, swa_scale, swa_start, swa_len):
    """Key/value rows of one query: every topk entry >= 0 (FP4, dequantised exactly)
    followed by SWA rows [swa_start, swa_start + swa_len) (E4M3 x row scale).

    codes_cache / scales_cache are the entries of the query's sequence in entry order
    (already resolved through the page table).  READING: no de-duplication between
    the two sources -- the selected entries come from the encoder state H_20 and the
    window from the layer's own hidden states [deep-dive §2]."""
    sel = np.asarray([t for t in np.asarray(topk).tolist() if t >= 0], dtype=np.int64)
    parts = []
    if len(sel):
        parts.append(formats.fp4_dequantize(codes_cache[sel], scales_cache[sel]))
    if swa_len > 0:
        parts.append(formats.fp8_rows_dequantize(swa_rows[swa_start:swa_start + swa_len],
                                                 swa_scale[swa_start:swa_start + swa_len]))
    if not parts:
        d = codes_cache.shape[-1] * 2
        return np.zeros((0, d))
    return np.concatenate(parts, axis=0)


def attend(q, kv, tau):
    """One softmax over all rows of kv, per head (float64).

    READING: the entry vector serves as both key and value (one 512-d vector per
    entry, and the head dim 512 equals the entry width, [deep-dive §6.3]); logits are
    tau * q_h . kv_s; no sink, no extra mask.  An empty row set gives out = 0 and
    lse = -inf.

    q: [Hq, d], kv: [S, d]  ->  (out [Hq, d], lse [Hq])
    """
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    Hq, d = q.shape
    if kv.shape[0] == 0:
        return np.zeros((Hq, d)), np.full(Hq, -np.inf)
    logits = tau * (q @ kv.T)                     # [Hq, S]
    mx = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - mx)
    den = p.sum(axis=1, keepdims=True)
    out = (p @ kv) / den
    lse = (mx + np.log(den))[:, 0]
    return out, lse


def sparse_attention(q, codes_cache, scales_cache, topk, swa_rows, swa_scale,
                     swa_start, swa_len, tau):
    """One decode query of one layer: gather_rows then attend."""
    kv = gather_rows(codes_cache, scales_cache, topk, swa_rows, swa_scale, swa_start, swa_len)
    return attend(q, kv, tau)


def dense_attention_loops(q, kv, tau):
    """Dense attention written with scalar loops (math.exp), used only to pin the
    sparse path: with Top-k covering every visible entry the sparse result must equal
    dense attention over all entries plus the window."""
    Hq = len(q)
    S = len(kv)
    d = len(q[0])
    out = np.zeros((Hq, d))
    lse = np.zeros(Hq)
    for h in range(Hq):
        lg = []
        for s in range(S):
            acc = 0.0
            for c in range(d):
                acc += float(q[h][c]) * float(kv[s][c])
            lg.append(tau * acc)
        m = max(lg)
        ws = [math.exp(v - m) for v in lg]
        tot = math.fsum(ws)
        for s in range(S):
            for c in range(d):
                out[h, c] += ws[s] / tot * float(kv[s][c])
        lse[h] = m + math.log(tot)
    return out, lse
