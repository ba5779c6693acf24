"""GPU parity of csa2_compress_quant against the oracle compressor."""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import csa2, synth
from oracle import compress, formats
from parity_utils import (bf16_dev, check_index_k, projection_error_bound, bf16_host_bits, fp4_mismatch_is_tolerated, paged_to_logical, to_dev)

pytestmark = pytest.mark.gpu


_check_index_k = check_index_k


def _check_fp4_of_own_rows(y_gpu, codes, scales):
    """The quantiser rule: the GPU's FP4 codes and scales are exactly the FP4 of the
    float32 rows it quantised (its own y_out), bit for bit."""
    c_own, s_own = formats.fp4_quantize(np.asarray(y_gpu, dtype=np.float32))
    np.testing.assert_array_equal(scales, s_own)
    np.testing.assert_array_equal(codes, c_own)


def _special_rows(r, G, d):
    """N(0,1) rows with groups scaled over many decades, plus zero / -0 / tiny / huge
    groups (scale 0, satfinite E4M3, saturated E2M1)."""
    C = r.standard_normal((G, d)).astype(np.float32)
    gs = np.exp2(r.integers(-14, 12, size=(G, d // 16))).astype(np.float32)
    C *= np.repeat(gs, 16, axis=1)
    C[0] = 0.0
    C[1] = -0.0
    C[2, :16] = 1e-4                       # a/6 < 2^-10 -> zero scale
    C[3, :16] = 5000.0                     # a/6 > 448 -> scale saturates, codes saturate
    C[4, 16:32] = -np.float32(6.0) * np.float32(0.25)
    C[5] = np.where(r.random(d) < 0.5, -0.0, 0.0).astype(np.float32)
    C[5, 3] = 1.0
    return C


def _layout(r, G, num_seqs=3):
    seq = (np.arange(G) % num_seqs).astype(np.int32)
    entry = (np.arange(G) // num_seqs).astype(np.int32)
    per = int(entry.max()) + 1
    mp = (per + 63) // 64
    pt = synth.page_table(r, num_seqs, mp)
    return seq, entry, pt


def _read_back(cache, pt, seq, entry):
    codes = cache.codes.cpu().numpy()
    scales = cache.scales.cpu().numpy()
    pages = pt[seq, entry // 64]
    return codes[pages, entry % 64], scales[pages, entry % 64]


@pytest.mark.parametrize("d,d_rope", [(128, 32), (512, 64), (512, 0)])
def test_quant_given_rows_bit_exact(d, d_rope):
    r = np.random.default_rng(100 + d + d_rope)
    G = 1000
    C = _special_rows(r, G, d)
    seq, entry, pt = _layout(r, G)
    cos, sin = synth.rope_tables(4096, d_rope)
    pos = r.integers(0, 4096, size=G).astype(np.int32)
    cache = csa2.PagedCache.allocate(3, int(entry.max()) + 1, d, 0, "cuda", torch.from_numpy(pt))
    y = torch.empty((G, d), dtype=torch.float32, device="cuda")
    csa2.compress_quant(cache, to_dev(seq), to_dev(entry), m=1, C=to_dev(C), pos=to_dev(pos),
                        rope_cos=to_dev(cos) if d_rope else None, rope_sin=to_dev(sin) if d_rope else None,
                        y_out=y)
    assert csa2.device_error() == 0
    ref = compress.compress_quant(C, None, 1, pos, cos, sin, d_rope)
    np.testing.assert_array_equal(y.cpu().numpy().view(np.uint32), ref["y"].view(np.uint32))
    codes, scales = _read_back(cache, pt, seq, entry)
    np.testing.assert_array_equal(scales, ref["scales"])
    np.testing.assert_array_equal(codes, ref["codes"])


def test_quant_every_e4m3_scale_and_e2m1_midpoint():
    # rows built so that a/6 walks every E4M3 value and its midpoints, and y/s hits every
    # E2M1 midpoint exactly: the hardware conversions must round exactly like the oracle.
    d = 512
    e4 = formats.e4m3_value(np.arange(1, 0x7F)).astype(np.float32)
    mids = np.concatenate([e4, ((e4[1:] + e4[:-1]) / 2).astype(np.float32)])
    e2mid = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    G = (len(mids) * 16 + d - 1) // d
    C = np.zeros((G * (d // 16), 16), dtype=np.float32)
    for i, s6 in enumerate(mids):
        a = np.float32(s6) * np.float32(6.0)
        s = np.float32(formats.e4m3_value(formats.e4m3_encode(np.float32(a) / np.float32(6.0))))
        row = np.concatenate([[a], -e2mid * s, e2mid * s, [0.0]]).astype(np.float32)
        C[i] = row
    C = C.reshape(G, d)
    r = np.random.default_rng(7)
    seq, entry, pt = _layout(r, G, 1)
    cache = csa2.PagedCache.allocate(1, G, d, 0, "cuda", torch.from_numpy(pt))
    csa2.compress_quant(cache, to_dev(seq), to_dev(entry), m=1, C=to_dev(C))
    ref = compress.compress_quant(C, None, 1, np.zeros(G, np.int32), None, None, 0)
    codes, scales = _read_back(cache, pt, seq, entry)
    np.testing.assert_array_equal(scales, ref["scales"])
    np.testing.assert_array_equal(codes, ref["codes"])


@pytest.mark.parametrize("m", [2, 4])
def test_quant_given_rows_pooled(m):
    r = np.random.default_rng(200 + m)
    d, G = 512, 600
    C = r.standard_normal((G * m, d)).astype(np.float32)
    Z = (2 * r.standard_normal((G * m, d))).astype(np.float32)
    seq, entry, pt = _layout(r, G, 2)
    cos, sin = synth.rope_tables(8192, 64)
    pos = (np.arange(G) * m + m - 1).astype(np.int32)
    cache = csa2.PagedCache.allocate(2, int(entry.max()) + 1, d, 0, "cuda", torch.from_numpy(pt))
    y = torch.empty((G, d), dtype=torch.float32, device="cuda")
    csa2.compress_quant(cache, to_dev(seq), to_dev(entry), m=m, C=to_dev(C), Z=to_dev(Z), pos=to_dev(pos),
                        rope_cos=to_dev(cos), rope_sin=to_dev(sin), y_out=y)
    ref = compress.compress_quant(C, Z, m, pos, cos, sin, 64)
    yg = y.cpu().numpy()
    np.testing.assert_allclose(yg, ref["y"], rtol=2e-6, atol=1e-6)
    codes, scales = _read_back(cache, pt, seq, entry)
    _check_fp4_of_own_rows(yg, codes, scales)
    bad, tol = fp4_mismatch_is_tolerated(ref["y"], codes, scales, ref["codes"], ref["scales"],
                                         np.abs(yg.astype(np.float64) - ref["y"]))
    assert bad == tol, f"{bad - tol} FP4 groups differ where the measured row error crosses no rounding decision"
    assert bad <= 5


@pytest.mark.parametrize("h_dtype,m,T,d_model", [("bf16", 1, 512, 256), ("f32", 1, 512, 256), ("bf16", 2, 512, 256),
                                               ("bf16", 1, 200, 5120), ("bf16", 2, 384, 1024),
                                               ("bf16", 1, 32, 5120), ("f32", 1, 64, 1024), ("bf16", 2, 64, 512),
                                               ("bf16", 1, 1, 5120), ("bf16", 4, 512, 1024),
                                               ("bf16", 2, 24576, 512), ("bf16", 4, 24576, 256)])
def test_compress_projection(h_dtype, m, T, d_model):
    # T <= 64 takes the few-row projection (decode append); larger bf16 T the tensor-core
    # GEMM (ragged last tile at T = 200, an 80-deep K loop at d_model = 5120, W_KV and W_Z
    # column tiles at m = 2, pooling/RoPE/FP4 in its epilogue at m <= 2, several tiles per
    # CTA of the persistent grid through both accumulator buffers at T = 24576); f32 H the
    # tiled SIMT one
    r = np.random.default_rng(300 + m + T)
    d, d_ik = 512, 128
    if h_dtype == "bf16":
        Hb = synth.bf16_normal(r, (T, d_model))
        H_host, H_dev = formats.bf16_value(Hb), bf16_dev(Hb)
    else:
        H_host = synth.f32_normal(r, (T, d_model))
        H_dev = to_dev(H_host)
    Wkv = synth.bf16_normal(r, (d_model, d), 1 / np.sqrt(d_model))
    Wz = synth.bf16_normal(r, (d_model, d), 1 / np.sqrt(d_model))
    Wik = synth.bf16_normal(r, (d, d_ik), 1 / np.sqrt(d))
    G = T // m
    seq = np.zeros(G, np.int32)
    entry = np.arange(G, dtype=np.int32)
    pt = synth.page_table(r, 1, (G + 63) // 64)
    cos, sin = synth.rope_tables(T, 64)
    pos = (np.arange(G) * m + m - 1).astype(np.int32)
    cache = csa2.PagedCache.allocate(1, G, d, d_ik, "cuda", torch.from_numpy(pt))
    y = torch.empty((G, d), dtype=torch.float32, device="cuda")
    csa2.compress_quant(cache, to_dev(seq), to_dev(entry), m=m, H=H_dev, W_kv=bf16_dev(Wkv), W_z=bf16_dev(Wz),
                        pos=to_dev(pos), rope_cos=to_dev(cos), rope_sin=to_dev(sin), W_ik=bf16_dev(Wik), y_out=y)
    assert csa2.device_error() == 0
    ref = compress.compress_quant_from_hidden(H_host, formats.bf16_value(Wkv), formats.bf16_value(Wz), m, pos,
                                              cos, sin, 64, formats.bf16_value(Wik))
    yg = y.cpu().numpy()
    err = np.abs(yg.astype(np.float64) - ref["y"])
    assert err.max() <= 1e-5 * np.abs(ref["y"]).max(), err.max()
    # the measured error lies within the float32 summation bound of the projection (plus
    # a few float32 ulps of the pooling and RoPE roundings)
    C = compress.project(H_host, formats.bf16_value(Wkv))
    Z = compress.project(H_host, formats.bf16_value(Wz)) if m > 1 else None
    bound = projection_error_bound(H_host, formats.bf16_value(Wkv), formats.bf16_value(Wz), m, 64, C, Z)
    assert (err <= bound + 4 * np.spacing(np.abs(ref["y"]).astype(np.float32))).all()
    codes, scales = _read_back(cache, pt, seq, entry)
    _check_fp4_of_own_rows(yg, codes, scales)
    # against the oracle's rows, a group may differ only where the measured row error
    # reaches a rounding decision
    bad, tol = fp4_mismatch_is_tolerated(ref["y"], codes, scales, ref["codes"], ref["scales"], err)
    assert bad == tol and bad <= max(2, 0.002 * G * d / 16)
    # indexer K: compare entries whose FP4 bytes agree, within one bf16 ulp
    ik = bf16_host_bits(cache.idx_k).reshape(-1, 64, d_ik)
    ikg = ik[pt[seq, entry // 64], entry % 64]
    same = (codes == ref["codes"]).all(1) & (scales == ref["scales"]).all(1)
    _check_index_k(ikg[same], ref["idx_k"][same], ref["codes"][same], ref["scales"][same], Wik)


@pytest.mark.parametrize("G,d,d_ik", [(1, 512, 128), (37, 512, 128), (200, 128, 64), (777, 512, 128),
                                      (2100, 512, 128)])
def test_index_k_of_bit_exact_entries(G, d, d_ik):
    # a few entries (the decode append) quantise and project in one launch; 777 and 2100 take
    # the tensor-core projection
    r = np.random.default_rng(400 + G)
    C = r.standard_normal((G, d)).astype(np.float32)
    Wik = synth.bf16_normal(r, (d, d_ik), 1 / np.sqrt(d))
    seq, entry, pt = _layout(r, G, 2)
    cache = csa2.PagedCache.allocate(2, int(entry.max()) + 1, d, d_ik, "cuda", torch.from_numpy(pt))
    csa2.compress_quant(cache, to_dev(seq), to_dev(entry), m=1, C=to_dev(C), W_ik=bf16_dev(Wik))
    ref = compress.compress_quant(C, None, 1, np.zeros(G, np.int32), None, None, 0, formats.bf16_value(Wik))
    codes, scales = _read_back(cache, pt, seq, entry)
    np.testing.assert_array_equal(codes, ref["codes"])
    ik = bf16_host_bits(cache.idx_k)[pt[seq, entry // 64], entry % 64]
    _check_index_k(ik, ref["idx_k"], ref["codes"], ref["scales"], Wik)
    assert (ik == ref["idx_k"]).mean() > (0.99 if G >= 100 else 0.95)


def test_bad_page_id_sets_error_word_and_skips():
    r = np.random.default_rng(500)
    d = 128
    C = r.standard_normal((64, d)).astype(np.float32)
    pt = np.array([[0, 7]], dtype=np.int32)           # page 7 does not exist (1 page... see below)
    cache = csa2.PagedCache.allocate(1, 64, d, 0, "cuda", torch.zeros((1, 1), dtype=torch.int32))
    cache.page_table = torch.from_numpy(pt).cuda()    # 2 pages in the table, only 1 allocated
    entry = np.arange(64, dtype=np.int32) + 32          # entries 64..95 fall on the bad page
    csa2.compress_quant(cache, to_dev(np.zeros(64, np.int32)), to_dev(entry), m=1, C=to_dev(C))
    err = csa2.device_error()
    assert err & 0x1
    ref = compress.compress_quant(C, None, 1, np.zeros(64, np.int32), None, None, 0)
    np.testing.assert_array_equal(cache.codes.cpu().numpy()[0, 32:], ref["codes"][:32])
    assert csa2.device_error() == 0
