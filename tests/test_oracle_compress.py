"""Pins for oracle.compress: projections, per-channel softmax pooling of m tokens,
RoPE and the indexer-K projection, against closed forms and scalar loops."""
import math

import numpy as np
import pytest

from fp4_compressed_sparse_02_gb300 import synth
from oracle import compress, formats


def test_project_matches_scalar_loops():
    r = np.random.default_rng(0)
    H = synth.bf16_normal(r, (5, 7))
    W = synth.bf16_normal(r, (7, 3))
    Hv = formats.bf16_value(H)
    Wv = formats.bf16_value(W)
    got = compress.project(Hv, Wv)
    for t in range(5):
        for c in range(3):
            assert math.isclose(got[t, c], math.fsum(Hv[t, j] * Wv[j, c] for j in range(7)),
                                rel_tol=1e-15, abs_tol=1e-15)


def test_m1_pooling_is_identity():
    r = np.random.default_rng(1)
    C = r.standard_normal((6, 32))
    np.testing.assert_array_equal(compress.pool_groups(C, None, 1), C)


def test_constant_z_gives_group_mean():
    r = np.random.default_rng(2)
    C = r.standard_normal((8, 16))
    Z = np.ones((8, 16)) * 3.7
    e = compress.pool_groups(C, Z, 4)
    np.testing.assert_allclose(e, C.reshape(2, 4, 16).mean(1), rtol=1e-14, atol=1e-14)


def test_two_token_softmax_closed_form():
    C = np.array([[1.0, 2.0], [5.0, -1.0]])
    Z = np.array([[0.3, -2.0], [1.1, 0.5]])
    e = compress.pool_groups(C, Z, 2)[0]
    for c in range(2):
        w0 = 1.0 / (1.0 + math.exp(Z[1, c] - Z[0, c]))
        assert math.isclose(e[c], w0 * C[0, c] + (1 - w0) * C[1, c], rel_tol=1e-14)


def test_dominant_z_selects_token_and_groups_do_not_overlap():
    r = np.random.default_rng(3)
    C = r.standard_normal((6, 8))
    Z = np.zeros((6, 8))
    Z[1] = 800.0          # group 0 -> token 1
    Z[4] = 800.0          # group 1 -> token 4; token 2/3 never leak into group 0
    e = compress.pool_groups(C, Z, 3)
    np.testing.assert_allclose(e[0], C[1], rtol=0, atol=1e-300)
    np.testing.assert_allclose(e[1], C[4], rtol=0, atol=1e-300)


def test_rope_identity_and_quarter_turn():
    r = np.random.default_rng(4)
    y = r.standard_normal((3, 64)).astype(np.float32)
    cos = np.zeros((4, 8), dtype=np.float32)
    sin = np.zeros((4, 8), dtype=np.float32)
    cos[0] = 1.0          # position 0: identity
    sin[1] = 1.0          # position 1: quarter turn (x0, x1) -> (-x1, x0)
    cos[2] = -1.0         # position 2: half turn
    out = compress.rope_f32(y, np.array([0, 1, 2]), cos, sin, 16)
    np.testing.assert_array_equal(out[0], y[0])
    np.testing.assert_array_equal(out[:, :48], y[:, :48])           # untouched channels
    np.testing.assert_array_equal(out[1, 48::2], -y[1, 49::2])
    np.testing.assert_array_equal(out[1, 49::2], y[1, 48::2])
    np.testing.assert_array_equal(out[2, 48:], -y[2, 48:])


def test_rope_preserves_pair_norm():
    r = np.random.default_rng(5)
    cos, sin = synth.rope_tables(4096, 64)
    y = r.standard_normal((200, 512)).astype(np.float32)
    pos = r.integers(0, 4096, 200)
    out = compress.rope_f32(y, pos, cos, sin, 64).astype(np.float64)
    yn = y.astype(np.float64)
    n0 = np.hypot(yn[:, 448::2], yn[:, 449::2])
    n1 = np.hypot(out[:, 448::2], out[:, 449::2])
    assert (np.abs(n1 - n0) <= 4 * np.spacing(n0.astype(np.float32)).astype(np.float64)).all()


def test_rope_tables_closed_form():
    cos, sin = synth.rope_tables(16, 8)
    assert (cos[0] == 1).all() and (sin[0] == 0).all()
    np.testing.assert_allclose(cos ** 2 + sin ** 2, 1.0, atol=1e-6)
    assert np.isclose(cos[1, 0], np.float32(math.cos(1.0)))


def test_index_k_projection_matches_loops():
    r = np.random.default_rng(6)
    codes = synth.fp4_codes(r, (3,), 32)
    scales = synth.fp4_scales(r, (3,), 32)
    W = synth.bf16_normal(r, (32, 4), 0.2)
    Wv = formats.bf16_value(W)
    got = compress.project_index_k(codes, scales, Wv)
    deq = formats.fp4_dequantize(codes, scales)
    for g in range(3):
        for j in range(4):
            ref = math.fsum(deq[g, c] * Wv[c, j] for c in range(32))
            assert got[g, j] == formats.bf16_round(ref)


def test_compress_pipeline_order_rope_before_quant():
    # a group whose RoPE'd value differs from the raw one must quantise the RoPE'd
    # value: compare with quantising the rotated rows directly.
    r = np.random.default_rng(7)
    C = r.standard_normal((4, 128))
    cos, sin = synth.rope_tables(8, 32)
    pos = np.array([1, 3, 5, 7])
    res = compress.compress_quant(C, None, 1, pos, cos, sin, 32)
    rot = compress.rope_f32(C.astype(np.float32), pos, cos, sin, 32)
    codes, scales = formats.fp4_quantize(rot)
    np.testing.assert_array_equal(res["codes"], codes)
    np.testing.assert_array_equal(res["scales"], scales)
    unrot, _ = formats.fp4_quantize(C.astype(np.float32))
    assert not np.array_equal(unrot, codes)


@pytest.mark.parametrize("m", [1, 2, 4])
def test_append_token_by_token_equals_compressing_the_whole_sequence(m):
    # buffering each token until its group completes, then compressing the group, must
    # give the entries of compressing all tokens at once (entries of complete groups only)
    r = np.random.default_rng(70 + m)
    d_model, d, d_ik, T = 64, 128, 64, 11
    H = r.standard_normal((T, d_model))
    Wkv = r.standard_normal((d_model, d)) / 8
    Wz = r.standard_normal((d_model, d)) / 8
    Wik = r.standard_normal((d, d_ik)) / 11
    cos, sin = synth.rope_tables(64, 32)
    pending, got = [], {}
    for t in range(T):
        res = compress.append_token(pending, H[t], t, Wkv, Wz, m, cos, sin, 32, Wik)
        if t % m != m - 1:
            assert res is None
        else:
            got[res[0]] = res[1]
    G = T // m
    assert sorted(got) == list(range(G)) and len(pending) == T % m
    pos = np.arange(G) * m + m - 1
    ref = compress.compress_quant_from_hidden(H[:G * m], Wkv, Wz, m, pos, cos, sin, 32, Wik)
    for g in range(G):
        np.testing.assert_array_equal(got[g]["y"][0], ref["y"][g])
        np.testing.assert_array_equal(got[g]["codes"][0], ref["codes"][g])
        np.testing.assert_array_equal(got[g]["scales"][0], ref["scales"][g])
        np.testing.assert_array_equal(got[g]["idx_k"][0], ref["idx_k"][g])
