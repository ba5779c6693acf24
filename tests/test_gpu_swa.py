"""GPU parity of csa2_swa_quant -- the FP8 window rows that a bounded replay rebuilds --
against the oracle's FP8 row quantiser, and of attention over a rebuilt window."""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import csa2, synth
from oracle import attention, formats
from parity_utils import ATTN_MAX_ABS, ATTN_REL_L2, bf16_dev, logical_to_paged, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _rows(r, R, d):
    """Rows over 60 octaves, some spread inside the row, plus zero / -0 / one-element /
    subnormal-scale / near-float32-max rows."""
    x = r.standard_normal((R, d)).astype(np.float32) * np.exp2(r.integers(-30, 30, size=(R, 1))).astype(np.float32)
    x[::5] *= np.exp2(r.uniform(-24, 0, size=(len(x[::5]), d))).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2] = 0.0
    x[2, 7] = -3.0
    x[3] = (r.standard_normal(d) * 1e-41).astype(np.float32)       # a / 448 underflows toward 0
    x[4] = (r.standard_normal(d) * 1e37).astype(np.float32)
    return x


def _device_rows(x, dtype):
    if dtype == "bf16":
        bits = synth.bf16_bits_from_f32(x)
        return bf16_dev(bits), formats.bf16_value(bits).astype(np.float32)
    return to_dev(x), x


@pytest.mark.parametrize("d,dtype", [(512, "f32"), (512, "bf16"), (128, "f32"), (128, "bf16")])
def test_swa_quant_bit_exact(d, dtype):
    r = np.random.default_rng(900 + d + len(dtype))
    R, rows = 1000, 1500
    x = _rows(r, R, d)
    xd, xv = _device_rows(x, dtype)
    dst = r.permutation(rows)[:R].astype(np.int32)
    swa = torch.full((rows, d), 0xAB, dtype=torch.uint8, device="cuda")
    sc = torch.full((rows,), -1.0, dtype=torch.float32, device="cuda")
    csa2.swa_quant(xd, swa, sc, to_dev(dst))
    assert csa2.device_error() == 0
    want_b, want_s = formats.fp8_rows_quantize(xv)
    got_b, got_s = swa.cpu().numpy(), sc.cpu().numpy()
    np.testing.assert_array_equal(got_s[dst].view(np.uint32), want_s.view(np.uint32))
    np.testing.assert_array_equal(got_b[dst], want_b)
    untouched = np.setdiff1d(np.arange(rows), dst)
    assert (got_b[untouched] == 0xAB).all() and (got_s[untouched] == -1.0).all()


def test_swa_quant_without_row_index_and_bad_rows_flagged():
    r = np.random.default_rng(950)
    d, R = 512, 40
    x = _rows(r, R, d)
    swa = torch.zeros((R, d), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((R,), dtype=torch.float32, device="cuda")
    csa2.swa_quant(to_dev(x), swa, sc)                      # row r -> row r
    assert csa2.device_error() == 0
    want_b, want_s = formats.fp8_rows_quantize(x)
    np.testing.assert_array_equal(swa.cpu().numpy(), want_b)
    np.testing.assert_array_equal(sc.cpu().numpy(), want_s)
    dst = np.arange(R, dtype=np.int32)
    dst[3], dst[9] = R + 5, -1                               # outside the window array: flagged, skipped
    swa.fill_(0x11)
    csa2.swa_quant(to_dev(x), swa, sc, to_dev(dst))
    assert csa2.device_error() & 0x20
    got = swa.cpu().numpy()
    ok = np.setdiff1d(np.arange(R), [3, 9])
    np.testing.assert_array_equal(got[ok], want_b[ok])
    assert (got[[3, 9]] == 0x11).all()


@pytest.mark.parametrize("k", [0, 512])
def test_bounded_replay_window_attention(k):
    # a bounded replay: the window rows of each query's last W tokens are recomputed (random
    # float32 rows stand in for the layer's projections of the replayed tokens), rebuilt as
    # FP8 into a fresh window array, and attended over -- alone (k = 0, as the encoder's
    # window-only layers) or with the selected FP4 entries in one softmax
    r = np.random.default_rng(960 + k)
    B, Hq, d, W, n = 4, 64, 512, 128, 3000
    x = (r.standard_normal((B * W, d)) * 0.7).astype(np.float32)
    swa = torch.zeros((B * W, d), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((B * W,), dtype=torch.float32, device="cuda")
    csa2.swa_quant(to_dev(x), swa, sc)
    mp = (n + 63) // 64
    pt = synth.page_table(r, 1, mp)
    codes = synth.fp4_codes(r, (n,), d)
    scales = synth.fp4_scales(r, (n,), d)
    cache = csa2.PagedCache.allocate(1, n, d, 0, "cuda", torch.from_numpy(pt))
    cache.codes.copy_(to_dev(logical_to_paged([codes], pt, mp, d // 2, np.uint8)))
    cache.scales.copy_(to_dev(logical_to_paged([scales], pt, mp, d // 16, np.uint8)))
    topk = np.full((B, max(k, 1)), -1, np.int32)
    for b in range(B):
        if k:
            topk[b] = synth.sorted_distinct(r, n, k)
    q = synth.bf16_normal(r, (B, Hq, d))
    seq = np.zeros(B, np.int32)
    starts = (np.arange(B) * W).astype(np.int32)
    tk = to_dev(topk) if k else torch.empty((B, 0), dtype=torch.int32, device="cuda")
    out, lse = csa2.sparse_attn(cache, bf16_dev(q), to_dev(seq), tk, None, swa, sc, to_dev(starts),
                                to_dev(np.full(B, W, np.int32)), W, out_dtype=torch.float32)
    assert csa2.device_error() == 0
    wb, ws = formats.fp8_rows_quantize(x)
    np.testing.assert_array_equal(swa.cpu().numpy(), wb)
    for b in range(B):
        o, l = attention.sparse_attention(formats.bf16_value(q[b]), codes, scales, topk[b] if k else [], wb, ws,
                                          int(starts[b]), W, 1 / np.sqrt(d))
        got = out[b].cpu().numpy()
        assert rel_l2(got, o) <= ATTN_REL_L2 and np.abs(got - o).max() <= ATTN_MAX_ABS
        np.testing.assert_allclose(lse[b].cpu().numpy(), l, rtol=1e-4, atol=1e-4)
