"""Seeded synthetic inputs for the CSA2 hot path.

This module is shared by the tests, the benchmark and the CPU oracle's callers.  It
only draws random numbers and arranges them in the documented layouts: it contains
none of the method's arithmetic (no quantisation, no scoring, no softmax).  Every
array is numpy on the host; callers copy to the device themselves.

Recipes (all from ``numpy.random.default_rng(seed)``):
  * bf16 tensors (hidden states, indexer Q/K, main Q, weights): float32 draws
    ~ N(0, sigma^2), narrowed to their upper 16 bits with round-half-even on the bit
    pattern (a plain dtype narrowing, not part of the method).
  * FP4 Main KV entries (when given directly rather than produced by the compressor):
    uniformly random bytes for the packed E2M1 codes and E4M3 scale bytes drawn
    uniformly from [0x20, 0x3F] (scales 2^-3 .. 1.875).
  * SWA rows: E4M3 bytes with a random sign, exponent field uniform in [3, 13] and
    a uniform 3-bit mantissa (never the NaN pattern), one positive float32 scale per
    row drawn uniformly from [0.005, 0.02].
  * page tables: a random permutation of page ids.
"""
import numpy as np


def rng(seed):
    return np.random.default_rng(seed)


def bf16_bits_from_f32(x):
    """Narrow float32 to bf16 bit patterns (round-half-even on the bit pattern)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_normal(r, shape, sigma=1.0):
    return bf16_bits_from_f32(r.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def f32_normal(r, shape, sigma=1.0):
    return (r.standard_normal(shape, dtype=np.float32) * np.float32(sigma)).astype(np.float32)


def fp4_codes(r, shape_entries, d):
    """Random packed E2M1 bytes [*shape_entries, d/2]."""
    return r.integers(0, 256, size=tuple(shape_entries) + (d // 2,), dtype=np.uint8)


def fp4_scales(r, shape_entries, d):
    """Random E4M3 scale bytes [*shape_entries, d/16] in [0x20, 0x3F]."""
    return r.integers(0x20, 0x40, size=tuple(shape_entries) + (d // 16,), dtype=np.uint8)


def fp8_rows(r, rows, d):
    sign = r.integers(0, 2, size=(rows, d), dtype=np.uint8) << 7
    expo = r.integers(3, 14, size=(rows, d), dtype=np.uint8) << 3
    man = r.integers(0, 8, size=(rows, d), dtype=np.uint8)
    return (sign | expo | man).astype(np.uint8)


def fp8_row_scales(r, rows):
    return r.uniform(0.005, 0.02, size=rows).astype(np.float32)


def page_table(r, num_seqs, pages_per_seq, shuffle=True):
    """int32 [num_seqs, pages_per_seq]: sequence s, page p -> physical page id.
    With shuffle the physical pages are a random permutation of all pages."""
    total = num_seqs * pages_per_seq
    ids = r.permutation(total) if shuffle else np.arange(total)
    return ids.astype(np.int32).reshape(num_seqs, pages_per_seq)


def rope_tables(max_pos, d_rope, theta=10000.0):
    """Frequency tables cos/sin [max_pos, d_rope/2] float32 for angle p * theta^(-2i/d_rope),
    computed in float64 and narrowed to float32.  These are model buffers handed to
    the compressor like its weights."""
    if d_rope == 0:
        z = np.zeros((max_pos, 0), dtype=np.float32)
        return z, z
    i = np.arange(d_rope // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / d_rope)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def sorted_distinct(r, n, k):
    """k distinct ascending integers from [0, n)."""
    k = min(k, n)
    return np.sort(r.choice(n, size=k, replace=False)).astype(np.int32)


# ---------------------------------------------------------------------------
# Workload shapes (the five configurations of the hot path)
# ---------------------------------------------------------------------------

TINY = dict(name="tiny_full_layer", N=4096, m=1, d=128, d_model=256, Hq=8, H_i=4, d_ik=64,
            NB=64, P=8, k=64, W=32, B=16, d_rope=32)
DEC128K = dict(name="decoder_N131072_B32", N=131072, m=1, d=512, d_model=5120, Hq=64, H_i=8,
               d_ik=128, NB=2048, P=8, k=512, W=128, B=32, d_rope=64)
# the pages' 32-head indexer (4x the scoring FLOPs of DEC128K for the same bytes)
DEC128K_HI32 = dict(name="decoder_N131072_B32_Hi32", N=131072, m=1, d=512, d_model=5120, Hq=64, H_i=32,
                    d_ik=128, NB=2048, P=8, k=512, W=128, B=32, d_rope=64)
# a speculative-decoding verification step: 32 sequences x 6 consecutive positions
DEC128K_V6 = dict(name="decoder_N131072_B32x6", N=131072, m=1, d=512, d_model=5120, Hq=64, H_i=8,
                  d_ik=128, NB=2048, P=8, k=512, W=128, B=32, G=6, d_rope=64)
DEC1M = dict(name="decoder_N1048576_B64", N=1048576, m=1, d=512, d_model=5120, Hq=64, H_i=8,
             d_ik=128, NB=2048, P=8, k=512, W=128, B=64, d_rope=64)
# the same decode workloads with the compressed (FP8) indexer-K form
DEC128K_IK8 = dict(DEC128K, name="decoder_N131072_B32_ik8", ik8=True)
DEC1M_IK8 = dict(DEC1M, name="decoder_N1048576_B64_ik8", ik8=True)
PREFILL = dict(name="encoder_prefill_T65536", T=65536, m=2, d=512, d_model=5120, Hq=64, H_i=8,
               d_ik=128, NB=2048, P=8, k=512, W=128, Q=8192, d_rope=64)
PAGE = 64
