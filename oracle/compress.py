"""Non-overlapping compressor, RoPE, FP4 quantisation and the indexer-K projection.

Test infrastructure (see oracle/__init__.py).

[deep-dive §2]   C = H . W_KV (Global KV entries), Z = H . W_Z (compression weights),
                 both layer-dependent linear projections of the hidden states.
[deep-dive §3.1] Hidden states -> non-overlapping compressor -> Main KV -> (projection)
                 -> Indexer K.  Every m tokens become one entry, with no overlap between
                 adjacent windows and no absolute position encoding in the compression.
                 Encoder m = 2, decoder m = 1.
[deep-dive §3.4] RoPE is applied to the entry before it is quantised to FP4.
"""
import numpy as np

from . import formats


def project(H, W):
    """C = H . W (or Z = H . W_Z) in float64 from the stored input values
    [deep-dive §2]."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(W, dtype=np.float64)


def pool_groups(C, Z, m):
    """Group g covers tokens [g*m, g*m + m) (non-overlapping, [deep-dive §3.1]).
    Per channel c: e[g, c] = sum_j softmax_j(Z[g*m + j, c]) * C[g*m + j, c]
    (the per-channel softmax weighting of Z; READING: softmax over the m tokens of
    the group, no positional bias since the compressor has no absolute PE).
    A trailing partial group is not emitted (READING: an entry exists once all m
    tokens exist); callers pass T divisible by m."""
    C = np.asarray(C, dtype=np.float64)
    T, d = C.shape
    assert T % m == 0
    G = T // m
    Cg = C.reshape(G, m, d)
    if m == 1:
        return Cg[:, 0, :].copy()
    Zg = np.asarray(Z, dtype=np.float64).reshape(G, m, d)
    zmax = Zg.max(axis=1, keepdims=True)
    ez = np.exp(Zg - zmax)
    wts = ez / ez.sum(axis=1, keepdims=True)
    return (wts * Cg).sum(axis=1)


def rope_f32(y, pos, cos_tab, sin_tab, d_rope):
    """Rotary embedding on the last ``d_rope`` channels of float32 rows
    [deep-dive §3.4: RoPE before quantisation].

    READING: channel pairs (b + 2i, b + 2i + 1), b = d - d_rope, are rotated by the
    angle whose cosine / sine are cos_tab[pos, i] / sin_tab[pos, i] (float32 tables
    supplied by the caller, like the projection weights).  The arithmetic is float32
    with every product and sum rounded on its own (no fused multiply-add):
        y0' = x0*c - x1*s,   y1' = x0*s + x1*c.
    """
    y = np.asarray(y, dtype=np.float32)
    if d_rope == 0:
        return y.copy()
    out = y.copy()
    d = y.shape[-1]
    b = d - d_rope
    x0 = y[:, b::2]
    x1 = y[:, b + 1::2]
    c = np.asarray(cos_tab, dtype=np.float32)[pos]
    s = np.asarray(sin_tab, dtype=np.float32)[pos]
    p00 = (x0 * c).astype(np.float32)
    p11 = (x1 * s).astype(np.float32)
    p01 = (x0 * s).astype(np.float32)
    p10 = (x1 * c).astype(np.float32)
    out[:, b::2] = (p00 - p11).astype(np.float32)
    out[:, b + 1::2] = (p01 + p10).astype(np.float32)
    return out


def project_index_k(codes, scales, W_ik):
    """Indexer K of an entry: bf16_RNE( dequant(FP4 entry) . W_IK ) in float64
    [deep-dive §3.1: "Indexer K directly projected from Main KV"].  READING: the
    projection reads the dequantised FP4 entry (the only form of Main KV kept in the
    cache) and the result is stored as bf16 (the pages quantise only Main KV and
    SWA KV).  Returns uint16 bf16 bits [G, d_ik]."""
    deq = formats.fp4_dequantize(codes, scales)
    return formats.bf16_round(deq @ np.asarray(W_ik, dtype=np.float64))


def compress_quant(C, Z, m, pos, cos_tab, sin_tab, d_rope, W_ik=None):
    """Given C (and Z when m > 1) per token, produce the FP4 entries.

    Steps, in the order of [deep-dive §3.1, §3.4]: per-channel softmax pooling of
    each group of m tokens (float64) -> round to float32 (the precision the
    quantiser reads) -> RoPE (float32) -> FP4 E2M1 + E4M3/16 -> optional indexer K.

    pos[g]: RoPE position of group g (READING: the position of the group's last
    token, g*m + m - 1 plus the chunk offset; the caller supplies it).
    Returns dict(y=float32 pre-quant rows, codes, scales, idx_k or None).
    """
    e = pool_groups(C, Z, m)
    y = e.astype(np.float32)
    y = rope_f32(y, np.asarray(pos), cos_tab, sin_tab, d_rope)
    codes, scales = formats.fp4_quantize(y)
    idx_k = project_index_k(codes, scales, W_ik) if W_ik is not None else None
    return dict(y=y, codes=codes, scales=scales, idx_k=idx_k)


def compress_quant_from_hidden(H, W_kv, W_z, m, pos, cos_tab, sin_tab, d_rope, W_ik=None):
    """The full compressor from hidden states: C = H.W_KV, Z = H.W_Z [deep-dive §2],
    then compress_quant."""
    C = project(H, W_kv)
    Z = project(H, W_z) if (m > 1 and W_z is not None) else None
    return compress_quant(C, Z, m, pos, cos_tab, sin_tab, d_rope, W_ik)


def append_token(pending, h, t, W_kv, W_z, m, cos_tab, sin_tab, d_rope, W_ik=None):
    """The decode-time append of one new token of a sequence at compression ratio m.

    [deep-dive §3.1] every m tokens become one entry (encoder m = 2).  READING (C2): an
    entry exists once all m of its tokens exist, so a token that does not complete its
    group waits in the sequence's pending list; the token at position t with t % m == m - 1
    completes group g = t // m, which is then compressed exactly as compress_quant does
    for the m tokens together, at the RoPE position of the group's last token, t.

    pending: the sequence's list of (C, Z) rows of its waiting tokens (updated in place).
    h: the token's hidden state [d_model].  Returns None while the group is incomplete,
    else (g, the compress_quant result of that one entry).
    """
    C = project(np.asarray(h)[None, :], W_kv)[0]
    Z = project(np.asarray(h)[None, :], W_z)[0] if (m > 1 and W_z is not None) else None
    assert len(pending) == t % m, "tokens of a sequence must arrive in order"
    pending.append((C, Z))
    if t % m != m - 1:
        return None
    Cg = np.stack([c for c, _ in pending])
    Zg = np.stack([z for _, z in pending]) if m > 1 else None
    pending.clear()
    return t // m, compress_quant(Cg, Zg, m, np.array([t]), cos_tab, sin_tab, d_rope, W_ik)


def index_k_fp8(idx_k_bits):
    """The compressed form of indexer K (READING, see indexer.fp8_form): each bf16 row
    quantised to E4M3 with one float32 scale amax / 448.  Returns (bytes, scales)."""
    return formats.fp8_rows_quantize(formats.bf16_value(idx_k_bits).astype(np.float32))
