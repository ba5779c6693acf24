"""Comparison rules for GPU-vs-oracle parity.

  * FP4 codes / scales, given identical float32 rows: bit-exact.
  * FP4 codes / scales from a float32 GPU pipeline vs the float64 oracle: equal except
    where the oracle's a/6 or y/s lies within 1e-5 (relative), or within the float32
    computation's error bound when the test supplies one, of a rounding decision (an
    E4M3 / E2M1 midpoint, or 0 for the sign of a code that rounds to zero).
  * Index sets: equal except for swaps at a selection boundary between entries whose
    oracle scores differ by <= 1e-5 relative (to the larger magnitude, with a floor of
    1e-5 x the largest |score| among the candidates for scores near zero).
  * Attention: relative L2 <= 2e-3 and max-abs <= 1e-2 against the float64 oracle.
"""
import numpy as np
import torch

from oracle import formats

REL_TIE = 1e-5
ATTN_REL_L2 = 2e-3
ATTN_MAX_ABS = 1e-2


def to_dev(a, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def bf16_dev(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def paged_to_logical(plane, page_table, seq, n):
    """Entries [0, n) of sequence seq from a paged plane [pages, 64, w] (numpy)."""
    e = np.arange(n)
    pages = page_table[seq, e // 64]
    return plane[pages, e % 64]


def logical_to_paged(rows_per_seq, page_table, num_pages, width, dtype):
    plane = np.zeros((num_pages, 64, width), dtype=dtype)
    for s, rows in enumerate(rows_per_seq):
        e = np.arange(len(rows))
        plane[page_table[s, e // 64], e % 64] = rows
    return plane


def check_index_set(gpu, ref, score_of, what=""):
    """gpu, ref: ascending entry arrays (no -1).  score_of: dict-like entry -> oracle
    score.  Returns the number of tolerated swaps; raises on any other difference."""
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    assert len(gpu) == len(ref), f"{what}: size {len(gpu)} vs {len(ref)}"
    assert len(np.unique(gpu)) == len(gpu), f"{what}: duplicate entries"
    assert (np.diff(gpu) > 0).all(), f"{what}: not ascending"
    only_g = np.setdiff1d(gpu, ref)
    only_r = np.setdiff1d(ref, gpu)
    if len(only_g) == 0:
        return 0
    sg = np.sort(np.array([score_of(e) for e in only_g]))[::-1]
    sr = np.sort(np.array([score_of(e) for e in only_r]))[::-1]
    floor = REL_TIE * max(1e-30, max(np.abs(sg).max(), np.abs(sr).max()))
    for a, b in zip(sg, sr):
        tol = REL_TIE * max(abs(a), abs(b)) + floor
        assert abs(a - b) <= tol, f"{what}: swap of scores {a!r} vs {b!r} exceeds the near-tie rule"
    return len(only_g)


def near_midpoint(x, grid, rel=REL_TIE):
    """True where |x| lies within rel of a midpoint of the ascending magnitude grid."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    mids = (grid[1:] + grid[:-1]) / 2
    i = np.clip(np.searchsorted(mids, x), 1, len(mids) - 1)
    near = np.minimum(np.abs(x - mids[i - 1]), np.abs(x - mids[np.minimum(i, len(mids) - 1)]))
    return near <= rel * np.maximum(x, 1e-30)


def near_midpoint_abs(x, grid, err):
    """True where |x| lies within the absolute distance err (or REL_TIE relative) of a
    midpoint of the ascending magnitude grid."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    mids = (grid[1:] + grid[:-1]) / 2
    i = np.clip(np.searchsorted(mids, x), 1, len(mids) - 1)
    near = np.minimum(np.abs(x - mids[i - 1]), np.abs(x - mids[np.minimum(i, len(mids) - 1)]))
    return near <= np.maximum(REL_TIE * np.maximum(x, 1e-30), np.asarray(err, dtype=np.float64))


def fp4_mismatch_is_tolerated(y_oracle, codes_g, scales_g, codes_o, scales_o, y_err=None):
    """Per 16-channel group: a mismatching group is tolerated only if the oracle's a/6 is
    near an E4M3 midpoint, or (same scale) every mismatching code's y/s is near an E2M1
    midpoint.  "Near" is REL_TIE relative, or, when y_err (a bound on |y_gpu - y_oracle|
    per element) is given, within that bound carried through the division.
    Returns (n_mismatched_groups, n_tolerated)."""
    y = np.asarray(y_oracle, dtype=np.float32)
    G, d = y.shape
    cg = formats.fp4_unpack(codes_g).reshape(G, d // 16, 16)
    co = formats.fp4_unpack(codes_o).reshape(G, d // 16, 16)
    bad = (scales_g != scales_o) | (cg != co).any(-1)
    e4 = formats.e4m3_value(np.arange(0x7F))
    e2 = formats.e2m1_value(np.arange(8))
    yg = y.reshape(G, d // 16, 16)
    eg = np.zeros_like(yg, dtype=np.float64) if y_err is None else np.asarray(y_err, np.float64).reshape(G, d // 16, 16)
    tol = 0
    for gi, qi in zip(*np.nonzero(bad)):
        a = np.abs(yg[gi, qi]).max()
        if scales_g[gi, qi] != scales_o[gi, qi]:
            ok = near_midpoint_abs(np.float32(a) / np.float32(6.0), e4, eg[gi, qi].max() / 6.0).item()
        else:
            s = np.float32(formats.e4m3_value(scales_o[gi, qi]))
            diff = cg[gi, qi] != co[gi, qi]
            yd, ed = yg[gi, qi][diff], eg[gi, qi][diff]
            near = near_midpoint_abs(yd / s, e2, ed / s)
            # E2M1 keeps the sign of a value that rounds to zero: +0 vs -0 is the decision
            # at the boundary 0, tolerated when |y| is within the error bound of 0
            zero = ((cg[gi, qi][diff] & 7) == 0) & ((co[gi, qi][diff] & 7) == 0) & (
                np.abs(yd) <= np.maximum(ed, REL_TIE * s))
            ok = bool((near | zero).all())
        tol += int(ok)
    return int(bad.sum()), tol


def projection_error_bound(H, W_kv, W_z, m, d_rope, C, Z):
    """Bound on |y_gpu - y_oracle| for the compressor from hidden states, per (group,
    channel).  The projection sums K bf16 x bf16 products (exact in fp32) in fp32 in some
    order: |error| <= gamma_K * sum_k |h_k w_k|, gamma_K = K u / (1 - K u), u = 2^-24
    (the standard bound for recursive summation in any order).  The m-token softmax
    pooling e = sum_j w_j C_j, w = softmax(Z), moves by at most max_j eC_j from the C
    errors and, to first order, max_j eZ_j * (max_j C_j - min_j C_j) from the Z errors
    (doubled here); the RoPE rotation of a pair adds the two errors of the pair."""
    H = np.abs(np.asarray(H, dtype=np.float64))
    K = H.shape[1]
    u = 2.0 ** -24
    gamma = K * u / (1 - K * u)
    eC = gamma * (H @ np.abs(np.asarray(W_kv, dtype=np.float64)))
    T, d = eC.shape
    if m == 1:
        e = eC
    else:
        eZ = gamma * (H @ np.abs(np.asarray(W_z, dtype=np.float64)))
        Cg = np.asarray(C, dtype=np.float64).reshape(T // m, m, d)
        e = eC.reshape(T // m, m, d).max(1) + 2.0 * eZ.reshape(T // m, m, d).max(1) * (Cg.max(1) - Cg.min(1))
    if d_rope:
        b = d - d_rope
        pair = e[:, b::2] + e[:, b + 1::2]
        e = e.copy()
        e[:, b::2] = pair
        e[:, b + 1::2] = pair
    return e


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def check_index_k(got_bits, ref_bits, codes, scales, Wik):
    """GPU indexer K (float32 sum of d products, then bf16) vs the oracle (float64 sum,
    then bf16): within one bf16 ulp of the oracle value plus the float32 recursive-sum
    error bound d * 2^-24 * sum_c |deq_c * W_c| (which dominates when the sum cancels)."""
    a = formats.bf16_value(got_bits)
    b = formats.bf16_value(ref_bits)
    ulp = np.abs(formats.bf16_value(ref_bits.astype(np.uint32) + 1) - b)
    deq = formats.fp4_dequantize(codes, scales)
    mag = np.abs(deq) @ np.abs(formats.bf16_value(Wik))
    d = deq.shape[-1]
    bound = ulp + d * 2.0 ** -24 * mag
    assert (np.abs(a - b) <= bound).all(), float(np.max(np.abs(a - b) - bound))
