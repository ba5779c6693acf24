"""Pins for oracle.attention and oracle.schedule: dense equality when Top-k covers
every entry, closed forms, permutation invariance and the pages' layer schedules."""
import numpy as np

from conftest import read_golden
from fp4_compressed_sparse_02_gb300 import synth
from oracle import attention, formats, indexer, schedule


def _cache(r, n, d):
    return synth.fp4_codes(r, (n,), d), synth.fp4_scales(r, (n,), d)


def test_sparse_with_everything_selected_equals_dense_loops():
    r = np.random.default_rng(0)
    n, d, W, Hq = 10, 32, 3, 2
    codes, scales = _cache(r, n, d)
    swa = synth.fp8_rows(r, 8, d)
    sc = synth.fp8_row_scales(r, 8)
    q = formats.bf16_value(synth.bf16_normal(r, (Hq, d)))
    tau = 1 / np.sqrt(d)
    out, lse = attention.sparse_attention(q, codes, scales, np.arange(n), swa, sc, 4, W, tau)
    kv = np.concatenate([formats.fp4_dequantize(codes, scales),
                         formats.fp8_rows_dequantize(swa[4:4 + W], sc[4:4 + W])])
    dout, dlse = attention.dense_attention_loops(q.tolist(), kv.tolist(), tau)
    np.testing.assert_allclose(out, dout, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, dlse, rtol=1e-12)


def test_single_key_returns_its_row():
    r = np.random.default_rng(1)
    codes, scales = _cache(r, 5, 32)
    q = r.standard_normal((3, 32))
    out, lse = attention.sparse_attention(q, codes, scales, np.array([-1, 2, -1]),
                                          np.zeros((1, 32), np.uint8), np.ones(1, np.float32),
                                          0, 0, 0.3)
    row = formats.fp4_dequantize(codes[2], scales[2])
    np.testing.assert_allclose(out, np.tile(row, (3, 1)), rtol=1e-14)
    np.testing.assert_allclose(lse, 0.3 * (q @ row), rtol=1e-14)


def test_zero_query_is_mean_of_rows():
    r = np.random.default_rng(2)
    codes, scales = _cache(r, 20, 64)
    sel = np.array([1, 4, 7, 19])
    out, lse = attention.sparse_attention(np.zeros((2, 64)), codes, scales, sel,
                                          np.zeros((1, 64), np.uint8), np.ones(1, np.float32),
                                          0, 0, 1.0)
    np.testing.assert_allclose(out[0], formats.fp4_dequantize(codes[sel], scales[sel]).mean(0),
                               rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(4.0))


def test_permutation_invariance():
    r = np.random.default_rng(3)
    codes, scales = _cache(r, 50, 64)
    swa = synth.fp8_rows(r, 10, 64)
    sc = synth.fp8_row_scales(r, 10)
    q = r.standard_normal((4, 64))
    sel = np.array([3, 8, 11, 20, 42])
    a = attention.sparse_attention(q, codes, scales, sel, swa, sc, 2, 5, 0.125)
    b = attention.sparse_attention(q, codes, scales, sel[::-1], swa, sc, 2, 5, 0.125)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13, atol=1e-13)


def test_empty_selection_and_window():
    r = np.random.default_rng(4)
    codes, scales = _cache(r, 5, 32)
    out, lse = attention.sparse_attention(np.ones((2, 32)), codes, scales, np.array([-1, -1]),
                                          np.zeros((1, 32), np.uint8), np.ones(1, np.float32),
                                          0, 0, 1.0)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_softmax_scale_enters_logits():
    kv = np.array([[1.0, 0.0], [0.0, 1.0]])
    q = np.array([[2.0, 0.0]])
    out, lse = attention.attend(q, kv, 0.5)
    p0 = np.exp(1.0) / (np.exp(1.0) + 1.0)
    np.testing.assert_allclose(out[0], [p0, 1 - p0], rtol=1e-14)


def test_schedules_match_pages():
    g = {r[0]: r[1:] for r in read_golden("pages_numbers.txt")}
    assert schedule.decoder_schedule() == g["decoder_schedule"]
    assert schedule.encoder_schedule() == g["encoder_schedule"]


def test_decode_step_reuse_gives_recomputed_result():
    r = np.random.default_rng(5)
    n, d, dk = 400, 64, 16
    codes, scales = _cache(r, n, d)
    K = r.standard_normal((n, dk))
    swa = synth.fp8_rows(r, 8, d)
    sc = synth.fp8_row_scales(r, 8)
    layers = []
    for mode in schedule.decoder_schedule():
        layers.append(dict(mode=mode, q_idx=r.standard_normal((2, dk)), w=np.ones(2),
                           q=r.standard_normal((2, d)), swa_rows=swa, swa_scale=sc,
                           swa_start=0, swa_len=8))
    res = schedule.decode_step(layers, K, codes, scales, 16, 8, 20, 0.125)
    assert len(res) == 20
    for l, (mode, topk, out, lse) in enumerate(res):
        if mode == "reuse":
            np.testing.assert_array_equal(topk, res[l - 1][1])
            o2, _ = attention.sparse_attention(layers[l]["q"], codes, scales, res[l - 1][1], swa, sc,
                                               0, 8, 0.125)
            np.testing.assert_array_equal(out, o2)
        if mode == "reindex":
            pool, _, _ = indexer.full(layers[0]["q_idx"], layers[0]["w"], K, 16, 8, 20)
            assert set(topk.tolist()) <= set(pool.tolist())
