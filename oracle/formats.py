"""Number formats of the CSA2 cache: FP4 E2M1 codes with one FP8 E4M3 scale per 16
channels (Main KV), FP8 E4M3 rows (SWA KV) and bf16 (indexer K).

Test infrastructure (see oracle/__init__.py).

[deep-dive §3.4] Main KV is stored as E2M1 values sharing one E4M3 scale per 16
channels, quantised after RoPE; SWA KV stays FP8.  [daily-report] states the same
E2M1 + E4M3-per-16 format.  The bit layouts below are the OCP E2M1 / E4M3 (FN)
definitions that those names denote.

Everything here is written from the definitions: decoders build values from the
sign / exponent / mantissa fields, encoders pick the nearest representable value
by comparing exact distances (float64 holds every float32 and every grid value
exactly, so the comparison is exact), ties going to the even code.
"""
import numpy as np

# ---------------------------------------------------------------------------
# E2M1: 1 sign bit (bit 3), 2 exponent bits (bits 2..1), 1 mantissa bit (bit 0),
# exponent bias 1, no infinities or NaN.
# ---------------------------------------------------------------------------


def e2m1_value(code):
    """Decode 4-bit E2M1 codes (0..15) to float64."""
    code = np.asarray(code, dtype=np.int64)
    sign = np.where(code & 8, -1.0, 1.0)
    e = (code >> 1) & 3
    man = code & 1
    mag = np.where(e == 0, man * 0.5, (1.0 + man / 2.0) * np.exp2(e - 1.0))
    return sign * mag


_E2M1_MAG = e2m1_value(np.arange(8))          # 0, .5, 1, 1.5, 2, 3, 4, 6 ascending


def _nearest_code(x_abs, grid):
    """Index into ascending ``grid`` nearest to each x_abs (float64, >= 0, within
    [grid[0], grid[-1]]); exact ties go to the even index.  Because the codes of
    non-negative values are ascending in value, "even index" is "even code",
    i.e. round-half-to-even on the mantissa LSB."""
    x_abs = np.asarray(x_abs, dtype=np.float64)
    i = np.searchsorted(grid, x_abs, side="right") - 1
    i = np.clip(i, 0, len(grid) - 2)
    lo = grid[i]
    hi = grid[i + 1]
    dlo = x_abs - lo
    dhi = hi - x_abs
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (i % 2 == 1))
    out = np.where(pick_hi, i + 1, i)
    # x exactly on the top grid value
    out = np.where(x_abs >= grid[-1], len(grid) - 1, out)
    return out.astype(np.int64)


def e2m1_encode(x):
    """Round float32 values to E2M1 codes, round-to-nearest-even, saturating to
    +-6.  The sign bit is the sign bit of x (a negative value that rounds to zero
    keeps its sign, as IEEE rounding does).  NaN is outside the contract."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x).astype(np.float64)
    mag = np.minimum(mag, _E2M1_MAG[-1])                 # satfinite
    code = _nearest_code(mag, _E2M1_MAG)
    neg = np.signbit(x)
    return (code | np.where(neg, 8, 0)).astype(np.uint8)


# ---------------------------------------------------------------------------
# E4M3 (FN variant): 1 sign bit (7), 4 exponent bits (6..3), 3 mantissa bits
# (2..0), bias 7.  Exponent field 0 is subnormal (man * 2^-9).  S.1111.111 is NaN;
# there is no infinity.  Largest finite magnitude 448.
# ---------------------------------------------------------------------------


def e4m3_value(byte):
    """Decode E4M3 bytes to float64 (NaN for the two NaN encodings)."""
    b = np.asarray(byte, dtype=np.int64) & 0xFF
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    man = b & 7
    mag = np.where(e == 0, man * np.exp2(-9.0), (1.0 + man / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (man == 7), np.nan, mag)
    return sign * mag


_E4M3_MAG = e4m3_value(np.arange(0x7F))      # codes 0..126: every finite magnitude, ascending


def e4m3_encode(x):
    """Round float32 values to E4M3 bytes: round-to-nearest-even, saturating to
    +-448 (the "satfinite" behaviour: NaN is never produced from finite input)."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.minimum(np.abs(x).astype(np.float64), _E4M3_MAG[-1])
    code = _nearest_code(mag, _E4M3_MAG)
    neg = np.signbit(x)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


# ---------------------------------------------------------------------------
# bf16: the upper half of a float32, same exponent range, 8 significant bits.
# ---------------------------------------------------------------------------


def bf16_value(bits):
    """Decode bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_round(x):
    """Round float64 values to bf16, round-to-nearest-even, directly from the
    float64 value (no intermediate float32 rounding).  Returns uint16 bits."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.float64)
    nz = (x != 0) & np.isfinite(x)
    _, E = np.frexp(np.where(nz, x, 1.0))        # |x| = f * 2^E, f in [0.5, 1)
    lead = np.maximum(E - 1, -126)               # exponent of the leading bit (normals)
    ulp = np.exp2(lead - 7.0)                    # 8 significant bits
    r = np.round(x / ulp) * ulp                  # np.round: ties to even; /ulp is exact
    out = np.where(nz, r, x)
    big = np.abs(out) > 3.3895313892515355e38    # largest finite bf16
    out = np.where(big, np.copysign(np.inf, x), out)
    return (out.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# FP4 Main KV rows: E2M1 codes, one E4M3 scale per 16 channels.
# ---------------------------------------------------------------------------

GROUP = 16   # channels per scale [deep-dive §3.4], [daily-report]


def fp4_quantize(y):
    """Quantise float32 rows ``y[..., d]`` (d % 16 == 0) to packed FP4.

    Per group of 16 channels [deep-dive §3.4]:
      a   = max |y_i|                       (exact, float32)
      s   = E4M3_RNE_satfinite(a / 6)       (a/6 is the float32 division, correctly
                                             rounded; 6 is the largest E2M1 value)
      s == 0  -> scale byte 0, every code 0 (+0)
      else    -> code_i = E2M1_RNE_sat(y_i / s)  (float32 division, correctly rounded)
    Packing (READING): two codes per byte, the even channel in the low nibble.

    Returns (codes uint8[..., d/2], scales uint8[..., d/16]).
    """
    y = np.asarray(y, dtype=np.float32)
    d = y.shape[-1]
    assert d % GROUP == 0
    g = y.reshape(y.shape[:-1] + (d // GROUP, GROUP))
    a = np.max(np.abs(g), axis=-1)                          # float32
    s32 = (a / np.float32(6.0)).astype(np.float32)          # float32 division
    sbyte = e4m3_encode(s32)
    s = e4m3_value(sbyte).astype(np.float32)                # exact
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (g / s[..., None]).astype(np.float32)           # float32 division
    code = e2m1_encode(np.where(s[..., None] > 0, q, np.float32(0.0)))
    code = np.where(s[..., None] > 0, code, 0).astype(np.uint8)
    code = code.reshape(y.shape[:-1] + (d,))
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, sbyte


def fp4_unpack(codes):
    """uint8[..., d/2] packed codes -> uint8[..., d] 4-bit codes (even channel =
    low nibble)."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


def fp4_dequantize(codes, scales):
    """Packed FP4 rows -> float64 values code_value * scale.  The product of a
    2-significant-bit E2M1 value and a 4-significant-bit E4M3 scale is exact in
    float64 (and in float32, bf16 and fp16)."""
    c = fp4_unpack(codes)
    v = e2m1_value(c)
    s = e4m3_value(scales)
    d = v.shape[-1]
    return v * np.repeat(s, GROUP, axis=-1).reshape(v.shape[:-1] + (d,))


def fp8_rows_dequantize(rows, row_scale):
    """SWA rows: E4M3 bytes times a per-row float32 scale (READING: one scale per
    row), exact in float64."""
    return e4m3_value(rows) * np.asarray(row_scale, dtype=np.float64)[..., None]


# ---------------------------------------------------------------------------
# FP8 rows with one float32 scale per row: the SWA window rows, rebuilt here when a
# window is replayed [deep-dive §3.4, "SWA Bounded Replay"], and the optional compressed
# indexer-K plane.
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0      # the largest finite E4M3 magnitude


def fp8_rows_quantize(x):
    """Quantise rows ``x[..., d]`` (float32 values; bf16 values are exact in float32) to
    E4M3 bytes with one float32 scale per row.

    READING (the pages say only that SWA KV stays FP8 [deep-dive §3.4]): the row's scale
    maps its largest magnitude onto the largest E4M3 value, as the FP4 scale maps a
    group's onto the largest E2M1 value:
      a = max_i |x_i|                              (exact)
      s = a / 448                                  (float32 division, correctly rounded)
      s == 0 -> every byte 0
      else   -> byte_i = E4M3_RNE_satfinite(x_i / s)   (float32 division)

    Returns (bytes uint8[..., d], scales float32[...]).
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.max(np.abs(x), axis=-1)
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)          # float32 division
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (x / s[..., None]).astype(np.float32)              # float32 division
    b = e4m3_encode(np.where(s[..., None] > 0, q, np.float32(0.0)))
    b = np.where(s[..., None] > 0, b, 0).astype(np.uint8)
    return b, s
