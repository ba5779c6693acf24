"""Pins for oracle.formats: the E2M1 / E4M3 / bf16 definitions and the FP4 group
quantiser, checked against golden tables, brute force and torch's own casts."""
import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import formats


def test_e2m1_grid_matches_definition_table():
    rows = read_golden("e2m1_grid.txt")
    for code, val in rows:
        code = int(code)
        assert formats.e2m1_value(code) == float(val)
        assert formats.e2m1_value(code | 8) == -float(val)


def test_e2m1_rounding_golden_midpoints():
    for x, code in read_golden("e2m1_rounding.txt"):
        got = int(formats.e2m1_encode(np.float32(float(x))))
        assert got == int(code), (x, got, code)


def _e2m1_bruteforce(x):
    """Nearest of the 8 magnitudes by exhaustive comparison; tie -> even code."""
    mag = min(abs(float(x)), 6.0)
    best = None
    for c in range(8):
        v = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0][c]
        dist = abs(mag - v)
        if best is None or dist < best[0] or (dist == best[0] and c % 2 == 0):
            best = (dist, c)
    return best[1] | (8 if np.signbit(np.float32(x)) else 0)


def test_e2m1_encode_matches_bruteforce_sweep():
    r = np.random.default_rng(1)
    xs = np.concatenate([
        np.linspace(-7.5, 7.5, 6001, dtype=np.float32),
        r.uniform(-8, 8, 4000).astype(np.float32),
        np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]) * np.float32(-1),
    ])
    got = formats.e2m1_encode(xs)
    want = np.array([_e2m1_bruteforce(x) for x in xs], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


def test_e4m3_decode_golden_and_torch():
    for b, v in read_golden("e4m3_points.txt"):
        got = formats.e4m3_value(int(b, 16))
        if v == "nan":
            assert np.isnan(got)
        else:
            assert got == float(v) and np.signbit(got) == np.signbit(float(v))
    allb = np.arange(256, dtype=np.uint8)
    tv = torch.from_numpy(allb).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    ov = formats.e4m3_value(allb)
    nan = np.isnan(tv)
    np.testing.assert_array_equal(np.isnan(ov), nan)
    np.testing.assert_array_equal(ov[~nan], tv[~nan])


def test_e4m3_encode_matches_torch_on_every_f32_in_a_dense_sweep():
    # every float32 bit pattern with a stride, from 2^-14 up to 448, plus exact
    # midpoints between neighbouring E4M3 values
    lo = np.float32(2.0 ** -14).view(np.uint32)
    hi = np.float32(448.0).view(np.uint32)
    bits = np.arange(lo, hi + 1, 97, dtype=np.uint32)
    xs = bits.view(np.float32)
    grid = formats.e4m3_value(np.arange(0x7F))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([xs, mids, -mids, np.float32([0.0, 448.0])])
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = formats.e4m3_encode(xs)
    np.testing.assert_array_equal(got, want)


def test_e4m3_encode_saturates():
    xs = np.float32([448.0, 449.0, 464.0, 480.0, 1e6, 3e38])
    assert (formats.e4m3_encode(xs) == 0x7E).all()
    assert (formats.e4m3_encode(-xs) == 0xFE).all()


def test_bf16_round_matches_torch_for_float32_inputs():
    r = np.random.default_rng(2)
    xs = np.concatenate([r.standard_normal(20000).astype(np.float32) * 100,
                         r.uniform(-1e-30, 1e-30, 1000).astype(np.float32)])
    want = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = formats.bf16_round(xs.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_round_from_float64_has_no_double_rounding():
    # 1 + 2^-8 is the midpoint between bf16 1.0 and 1.0078125; a hair above it must
    # round up, even though the same value narrowed to float32 first would sit on
    # the midpoint and round to even (down).
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert formats.bf16_value(formats.bf16_round(x)) == 1.0078125
    assert formats.bf16_value(formats.bf16_round(1.0 + 2.0 ** -8)) == 1.0
    assert formats.bf16_value(formats.bf16_round(1.0 + 3 * 2.0 ** -8)) == 1.015625


def test_fp4_nibble_order_and_scale():
    y = np.zeros(32, dtype=np.float32)
    y[0] = 6.0       # group 0: amax 6 -> scale 1.0 (0x38); channel 0 -> code 7 (low nibble)
    y[1] = -0.5      # channel 1 -> code 9 (high nibble)
    y[16] = 0.0      # group 1 all zero -> scale byte 0, codes 0
    codes, scales = formats.fp4_quantize(y)
    assert scales.tolist() == [0x38, 0x00]
    assert codes[0] == (7 | (9 << 4))
    assert (codes[8:] == 0).all()


def test_fp4_roundtrip_of_representable_groups_is_identity():
    r = np.random.default_rng(3)
    for _ in range(200):
        sb = int(r.integers(0x08, 0x70))                 # a normal E4M3 scale
        s = formats.e4m3_value(sb)
        c = r.integers(0, 16, size=16)
        c[r.integers(0, 16)] = 7 | (8 * int(r.integers(0, 2)))   # amax = 6 s exactly
        y = (formats.e2m1_value(c) * s).astype(np.float32)
        codes, scales = formats.fp4_quantize(y)
        assert scales[0] == sb
        back = formats.fp4_dequantize(codes, scales)
        np.testing.assert_array_equal(back, y.astype(np.float64))


def test_fp4_error_bound():
    # |y - deq| <= s: half the widest grid gap (4 -> 6) times the scale, once the
    # scale covers amax (s >= a/6 up to E4M3 rounding, which the bound absorbs for
    # values that do not saturate; saturated values sit within a - 6 s of 6 s).
    r = np.random.default_rng(4)
    y = r.standard_normal((500, 64)).astype(np.float32)
    codes, scales = formats.fp4_quantize(y)
    deq = formats.fp4_dequantize(codes, scales)
    s = np.repeat(formats.e4m3_value(scales), 16, axis=-1)
    a = np.repeat(np.abs(y).reshape(500, 4, 16).max(-1), 16, axis=-1)
    bound = np.maximum(s, a - 6 * s + 1e-12)
    assert (np.abs(deq - y) <= bound + 1e-12).all()


def test_fp4_tiny_group_gets_zero_scale():
    y = np.full(16, 1e-4, dtype=np.float32)          # a/6 < 2^-10 -> scale rounds to 0
    codes, scales = formats.fp4_quantize(y)
    assert scales[0] == 0 and (codes == 0).all()


def test_fp8_rows_dequantize():
    rows = np.array([[0x38, 0xB8, 0x7E, 0x00]], dtype=np.uint8)
    out = formats.fp8_rows_dequantize(rows, np.float32([0.5]))
    np.testing.assert_array_equal(out, [[0.5, -0.5, 224.0, 0.0]])


@pytest.mark.parametrize("bad", [np.float32(0.2), np.float32(-3.3)])
def test_fp4_quantize_uses_float32_division(bad):
    # y / s is the float32 quotient: check against the brute-force rounding of
    # that float32 quotient.
    y = np.zeros(16, dtype=np.float32)
    y[0] = np.float32(5.9)
    y[1] = bad
    codes, scales = formats.fp4_quantize(y)
    s = np.float32(formats.e4m3_value(scales[0]))
    q = np.float32(bad) / s
    assert formats.fp4_unpack(codes)[1] == _e2m1_bruteforce(q)


# ---- FP8 rows with one float32 scale per row -------------------------------------------

def _fp8_rows_by_torch(x):
    """The same row quantiser written with torch's own float32 arithmetic and its E4M3 cast
    (torch rounds to nearest even; the quotients are clamped to the finite range first,
    which is what satfinite does)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    a = t.abs().amax(dim=-1)
    s = a / torch.tensor(448.0, dtype=torch.float32)
    q = torch.where(s[..., None] > 0, t / s[..., None], torch.zeros_like(t)).clamp(-448.0, 448.0)
    return q.to(torch.float8_e4m3fn).view(torch.uint8).numpy(), s.numpy()


def test_fp8_rows_quantize_matches_torch_on_wide_rows():
    r = np.random.default_rng(11)
    x = r.standard_normal((300, 512)).astype(np.float32)
    x *= np.exp2(r.integers(-30, 30, size=(300, 1))).astype(np.float32)     # rows over 60 octaves
    x[::7] *= np.exp2(r.uniform(-20, 0, size=(43, 512))).astype(np.float32)  # within-row spread
    got_b, got_s = formats.fp8_rows_quantize(x)
    want_b, want_s = _fp8_rows_by_torch(x)
    np.testing.assert_array_equal(got_s.view(np.uint32), want_s.view(np.uint32))
    np.testing.assert_array_equal(got_b, want_b)


def test_fp8_rows_largest_magnitude_maps_to_448():
    r = np.random.default_rng(12)
    x = (r.standard_normal((200, 128)) * np.exp2(r.integers(-40, 40, size=(200, 1)))).astype(np.float32)
    b, s = formats.fp8_rows_quantize(x)
    i = np.argmax(np.abs(x), axis=1)
    top = b[np.arange(200), i]
    assert ((top & 0x7F) == 0x7E).all()                          # +-448
    assert (np.signbit(x[np.arange(200), i]) == ((top & 0x80) != 0)).all()


def test_fp8_rows_roundtrip_of_representable_rows_is_identity():
    # rows that are E4M3 values times a power of two, with a +-448 element: quantising
    # gives back the same bytes and exactly that scale
    r = np.random.default_rng(13)
    finite = np.array([v for v in range(256) if (v & 0x7F) != 0x7F], dtype=np.uint8)
    b0 = r.choice(finite, size=(64, 512))
    b0[:, 5] = np.where(r.random(64) < 0.5, 0x7E, 0xFE)
    s0 = np.exp2(r.integers(-20, 10, size=64)).astype(np.float32)
    x = (formats.e4m3_value(b0) * s0[:, None]).astype(np.float32)
    b, s = formats.fp8_rows_quantize(x)
    np.testing.assert_array_equal(s, s0)
    np.testing.assert_array_equal(formats.e4m3_value(b), formats.e4m3_value(b0))   # +-0 may swap sign bytes only


def test_fp8_rows_error_bound_and_zero_rows():
    r = np.random.default_rng(14)
    x = r.standard_normal((50, 512)).astype(np.float32)
    x[3] = 0.0
    x[4] = -0.0
    b, s = formats.fp8_rows_quantize(x)
    assert s[3] == 0 and s[4] == 0 and (b[3] == 0).all() and (b[4] == 0).all()
    deq = formats.fp8_rows_dequantize(b, s)
    # |x - deq| <= s * (half the E4M3 gap at |x|/s): gap 2^(e-3) in [2^e, 2^(e+1)), 2^-9 below 2^-6
    q = np.abs(x.astype(np.float64)) / np.where(s > 0, s, 1)[:, None]
    e = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
    half_gap = np.where(q < 2.0 ** -6, 2.0 ** -10, np.exp2(e - 4))
    assert (np.abs(deq - x) <= s[:, None] * half_gap * (1 + 1e-6) + 1e-30).all()
