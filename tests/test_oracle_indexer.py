"""Pins for oracle.indexer: scoring, the balanced block partition, the shared pool
and Top-k, against scalar loops, a counting definition of top-k and the pages'
pool-size invariant."""
import math

import numpy as np
import pytest

from conftest import read_golden
from fp4_compressed_sparse_02_gb300 import synth
from oracle import formats, indexer


def _golden():
    return {r[0]: r[1:] for r in read_golden("pages_numbers.txt")}


def test_scores_match_scalar_loops():
    r = np.random.default_rng(0)
    q = r.standard_normal((3, 5))
    w = r.standard_normal(3)
    K = r.standard_normal((7, 5))
    s = indexer.scores(q, w, K)
    for e in range(7):
        want = math.fsum(w[h] * max(0.0, math.fsum(q[h, c] * K[e, c] for c in range(5)))
                         for h in range(3))
        assert math.isclose(s[e], want, rel_tol=1e-13, abs_tol=1e-13)


def test_literal_single_head_is_plain_dot():
    r = np.random.default_rng(1)
    q = r.standard_normal((1, 8))
    K = r.standard_normal((9, 8))
    np.testing.assert_allclose(indexer.scores(q, np.ones(1), K, relu=False), K @ q[0], rtol=1e-14)


def _top_by_counting(s, k):
    """i is selected iff fewer than k entries beat it (higher score, or equal score
    at a lower position)."""
    out = []
    for i in range(len(s)):
        beaten = sum(1 for j in range(len(s)) if s[j] > s[i] or (s[j] == s[i] and j < i))
        if beaten < k:
            out.append(i)
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("k", [0, 1, 5, 17, 40, 60])
def test_top_positions_matches_counting_definition_with_ties(k):
    r = np.random.default_rng(k)
    s = r.integers(-3, 4, size=50).astype(np.float64)     # many exact ties
    np.testing.assert_array_equal(indexer.top_positions(s, k), _top_by_counting(s, k))


def test_negative_zero_ties_with_zero():
    s = np.array([0.0, -0.0, 0.0, -0.0])
    np.testing.assert_array_equal(indexer.top_positions(s, 2), [0, 1])


@pytest.mark.parametrize("n,nb", [(0, 8), (5, 8), (8, 8), (100, 8), (101, 7), (4097, 64)])
def test_block_bounds_balanced(n, nb):
    bb = indexer.block_bounds(n, nb)
    assert bb[0] == 0 and bb[-1] == n
    lens = np.diff(bb)
    assert (lens >= 0).all() and lens.max() - lens.min() <= 1


@pytest.mark.parametrize("n", [1, 63, 511, 512, 513, 4096, 9000])
def test_pool_size_invariant_small(n):
    r = np.random.default_rng(n)
    q = r.standard_normal((2, 8))
    K = r.standard_normal((n, 8))
    pool, topk, s = indexer.full(q, np.ones(2), K, 64, 8, 64)
    assert len(pool) == min(n, 64 * 8)
    assert (np.diff(pool) > 0).all()
    if n <= 512:
        np.testing.assert_array_equal(pool, np.arange(n))
    assert len(topk) == min(64, len(pool))
    assert set(topk.tolist()) <= set(pool.tolist())


def test_pool_fixed_at_16384_for_the_pages_geometry():
    g = _golden()
    nb, pb = int(g["pool_blocks"][0]), int(g["pool_per_block"][0])
    assert nb * pb == int(g["pool_size"][0])
    r = np.random.default_rng(9)
    q = r.standard_normal((4, 16))
    for n in [16384, 20000, 50001]:
        K = r.standard_normal((n, 16))
        pool, topk, s = indexer.full(q, np.ones(4), K, nb, pb, int(g["top_k"][0]))
        assert len(pool) == int(g["pool_size"][0])
        assert len(topk) == int(g["top_k"][0])


def test_block_top8_is_exact_per_block():
    r = np.random.default_rng(10)
    n, nb, pb = 1000, 16, 8
    q = r.standard_normal((2, 4))
    K = r.standard_normal((n, 4))
    pool, topk, s = indexer.full(q, np.ones(2), K, nb, pb, 20)
    bb = indexer.block_bounds(n, nb)
    for b in range(nb):
        blk = np.arange(bb[b], bb[b + 1])
        want = bb[b] + _top_by_counting(s[blk], pb)
        got = pool[(pool >= bb[b]) & (pool < bb[b + 1])]
        np.testing.assert_array_equal(got, want)


def test_full_topk_equals_global_topk_when_no_block_overflows():
    r = np.random.default_rng(11)
    for trial in range(20):
        n = 3000
        q = r.standard_normal((3, 8))
        K = r.standard_normal((n, 8))
        pool, topk, s = indexer.full(q, np.ones(3), K, 64, 8, 32)
        glob = indexer.top_positions(s, 32)
        bb = indexer.block_bounds(n, 64)
        per_blk = np.bincount(np.searchsorted(bb, glob, side="right") - 1, minlength=64)
        if per_blk.max() <= 8:
            np.testing.assert_array_equal(topk, glob)


def test_reindex_over_whole_range_equals_unpooled_topk():
    r = np.random.default_rng(12)
    q = r.standard_normal((2, 8))
    K = r.standard_normal((300, 8))
    topk, s = indexer.reindex(q, np.ones(2), K, np.arange(300), 25)
    np.testing.assert_array_equal(topk, indexer.top_positions(indexer.scores(q, np.ones(2), K), 25))


def test_reindex_scores_only_the_pool():
    r = np.random.default_rng(13)
    q = r.standard_normal((2, 8))
    K = r.standard_normal((300, 8))
    pool = np.sort(r.choice(300, 40, replace=False))
    topk, s = indexer.reindex(q, np.ones(2), K, pool, 10)
    assert set(topk.tolist()) <= set(pool.tolist())
    # the best entry outside the pool is never chosen even if it beats them all
    K2 = K.copy()
    outside = np.setdiff1d(np.arange(300), pool)[0]
    K2[outside] = 50 * q[0]
    topk2, _ = indexer.reindex(q, np.ones(2), K2, pool, 10)
    np.testing.assert_array_equal(topk, topk2)


def test_reuse_is_identity():
    t = np.array([3, 9, 27, -1])
    np.testing.assert_array_equal(indexer.reuse(t), t)


def test_fp8_form_scores_equal_the_scaled_byte_products():
    # the FP8 indexer's score of an entry is sk * sum_h w_h sq_h ReLU(sum_c q8 k8): the row
    # scales (>= 0) factor out of the ReLU
    r = np.random.default_rng(31)
    H, dk, n = 8, 128, 300
    q = formats.bf16_value(synth.bf16_normal(r, (H, dk)))
    K = formats.bf16_value(synth.bf16_normal(r, (n, dk)))
    w = r.standard_normal(H)
    K8, Ks = formats.fp8_rows_quantize(K.astype(np.float32))
    qh, Kh = indexer.fp8_form(q, K8, Ks)
    s = indexer.scores(qh, w, Kh)
    q8, qs = formats.fp8_rows_quantize(q.astype(np.float32))
    dots = formats.e4m3_value(K8) @ formats.e4m3_value(q8).T          # exact integer-grid products
    want = Ks.astype(np.float64) * (np.maximum(dots, 0) @ (w * qs.astype(np.float64)))
    np.testing.assert_allclose(s, want, rtol=1e-12, atol=0)
    # and the quantised K is within half an E4M3 step of K (relative 2^-4 of each value, or
    # an absolute 2^-10 s below the normal range)
    assert (np.abs(Kh - K) <= np.maximum(np.abs(K) * 2.0 ** -4, Ks[:, None] * 2.0 ** -10) + 1e-30).all()
