"""GPU parity of csa2_index_full / csa2_index_reindex against the oracle indexer, on
identical indexer-K caches (drawn by the input generator)."""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import csa2, synth
from oracle import formats, indexer
from parity_utils import bf16_dev, check_index_set, logical_to_paged, to_dev

pytestmark = pytest.mark.gpu


def _setup(r, ns, n_max, d_ik, H_i, B, sigma=1.0):
    """ns sequences of n_max entries of random bf16 indexer K, paged through a random
    page table; B queries with random q / w."""
    mp = (n_max + 63) // 64
    pt = synth.page_table(r, ns, mp)
    K = [synth.bf16_normal(r, (n_max, d_ik), sigma) for _ in range(ns)]
    plane = logical_to_paged(K, pt, ns * mp, d_ik, np.uint16)
    cache = csa2.PagedCache.allocate(ns, n_max, 512, d_ik, "cuda", torch.from_numpy(pt))
    cache.idx_k.copy_(bf16_dev(plane))
    q = synth.bf16_normal(r, (B, H_i, d_ik))
    w = synth.f32_normal(r, (B, H_i), 1 / np.sqrt(H_i))
    return cache, K, q, w


def _run_full(cache, q, w, seq_of, n_vis, NB, P, k, relu=True):
    pool, plen, topk, tlen = csa2.index_full(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), to_dev(n_vis),
                                             int(n_vis.max()), NB, P, k, relu)
    assert csa2.device_error() == 0
    return pool.cpu().numpy(), plen.cpu().numpy(), topk.cpu().numpy(), tlen.cpu().numpy()


def _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got, relu=True):
    pool, plen, topk, tlen = got
    swaps = 0
    for b in range(len(n_vis)):
        n = int(n_vis[b])
        Kb = formats.bf16_value(K[seq_of[b]][:n])
        rpool, rtopk, s = indexer.full(formats.bf16_value(q[b]), w[b], Kb, NB, P, k, relu)
        assert plen[b] == len(rpool)
        assert tlen[b] == len(rtopk)
        assert (pool[b, plen[b]:] == -1).all() and (topk[b, tlen[b]:] == -1).all()
        gp = pool[b, :plen[b]]
        bb = indexer.block_bounds(n, NB)
        score = lambda e: s[e]
        if n >= NB * P:
            for j in range(NB):
                seg = gp[P * j:P * j + P]
                assert ((seg >= bb[j]) & (seg < bb[j + 1])).all(), f"query {b} block {j} out of range"
                rseg = rpool[P * j:P * j + P]
                swaps += check_index_set(seg, rseg, score, f"q{b} block {j}")
        else:
            np.testing.assert_array_equal(gp, rpool)
        swaps += check_index_set(topk[b, :tlen[b]], rtopk, score, f"q{b} topk")
    return swaps


@pytest.mark.parametrize("relu", [True, False])
def test_full_tiny_geometry_ragged(relu):
    r = np.random.default_rng(1 + relu)
    NB, P, k, d_ik, H_i = 64, 8, 64, 64, 4
    n_vis = np.array([0, 1, 5, 63, 64, 300, 512, 513, 4096, 4097, 9001, 20011], dtype=np.int32)
    B = len(n_vis)
    cache, K, q, w = _setup(r, 3, int(n_vis.max()), d_ik, H_i, B)
    seq_of = (np.arange(B) % 3).astype(np.int32)
    got = _run_full(cache, q, w, seq_of, n_vis, NB, P, k, relu)
    swaps = _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got, relu)
    assert swaps <= 4


def test_full_pages_geometry():
    r = np.random.default_rng(3)
    NB, P, k, d_ik, H_i = 2048, 8, 512, 128, 8
    n_vis = np.array([16384, 20000, 50001, 1000, 131072 // 2 + 7, 16383, 600, 100000], dtype=np.int32)
    B = len(n_vis)
    cache, K, q, w = _setup(r, 2, int(n_vis.max()), d_ik, H_i, B)
    seq_of = (np.arange(B) % 2).astype(np.int32)
    got = _run_full(cache, q, w, seq_of, n_vis, NB, P, k)
    swaps = _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got)
    assert swaps <= 8
    assert (got[1][n_vis >= NB * P] == NB * P).all()        # pool fixed at 16,384


@pytest.mark.parametrize("H_i", [1, 8, 12, 32])
def test_full_head_counts(H_i):
    r = np.random.default_rng(10 + H_i)
    NB, P, k = 256, 8, 128
    n_vis = np.array([5000, 2048, 777], dtype=np.int32)
    cache, K, q, w = _setup(r, 1, 5000, 128, H_i, 3)
    seq_of = np.zeros(3, np.int32)
    got = _run_full(cache, q, w, seq_of, n_vis, NB, P, k)
    assert _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got) <= 4


def _run_full_group(cache, q, w, seq_of, n_vis, NB, P, k, group):
    pool, plen, topk, tlen = csa2.index_full(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), to_dev(n_vis),
                                             int(n_vis.max()), NB, P, k, group=group)
    assert csa2.device_error() == 0
    return pool.cpu().numpy(), plen.cpu().numpy(), topk.cpu().numpy(), tlen.cpu().numpy()


@pytest.mark.parametrize("d_ik,H_i,NB,group", [(128, 8, 2048, 6), (64, 4, 64, 2), (128, 3, 256, 8), (128, 8, 512, 5)])
def test_full_grouped_queries(d_ik, H_i, NB, group):
    # groups of consecutive queries of one sequence (a verification step: positions n-g+1
    # .. n, one entry apart) scanned together: equal to the oracle per query and to the
    # same queries scanned one by one, bit for bit
    r = np.random.default_rng(40 + group + NB)
    P, k = 8, min(512, NB * 8 // 4)
    nseq = 3
    ends = [20000, 16384 + group // 2, 70001] if NB == 2048 else [5000, 1500, 9001]
    n_vis = np.array([e - group + 1 + t for e in ends for t in range(group)], dtype=np.int32)
    seq_of = np.repeat(np.arange(nseq), group).astype(np.int32)
    B = len(n_vis)
    cache, K, q, w = _setup(r, nseq, int(n_vis.max()), d_ik, H_i, B)
    got = _run_full_group(cache, q, w, seq_of, n_vis, NB, P, k, group)
    assert _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got) <= 8
    if not _tensor_core_scored(d_ik, H_i, group):
        # the grouped scan gives the results of scanning every query alone, bit for bit
        alone = _run_full(cache, q, w, seq_of, n_vis, NB, P, k)
        for x, y in zip(got, alone):
            np.testing.assert_array_equal(x, y)


def _tensor_core_scored(d_ik, H_i, group):
    return d_ik == 128 and H_i in (8, 16, 32) and max(group, 1) * H_i >= 16


@pytest.mark.parametrize("H_i,G,NB,ends", [(32, 1, 2048, (20000, 131072 // 2 + 3, 5000)),
                                           (16, 1, 256, (9001, 3000)),
                                           (32, 6, 512, (40000, 7001)),
                                           (8, 6, 2048, (150001, 20000))])
def test_full_tensor_core_decode(H_i, G, NB, ends):
    # single queries with 16 or 32 heads, and verification groups of 6: one tcgen05 product
    # per group; blocks of more than 64 entries (long contexts) take the warp-per-block
    # selection
    r = np.random.default_rng(80 + H_i + G + NB)
    P, k, d_ik = 8, 512, 128
    n_vis = np.array([e - G + 1 + t for e in ends for t in range(G)], dtype=np.int32)
    seq_of = np.repeat(np.arange(len(ends)), G).astype(np.int32)
    cache, K, q, w = _setup(r, len(ends), int(n_vis.max()), d_ik, H_i, len(n_vis))
    got = _run_full_group(cache, q, w, seq_of, n_vis, NB, P, k, G)
    assert _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got) <= 4 * len(n_vis)
    assert (got[1][n_vis >= NB * P] == NB * P).all()


@pytest.mark.parametrize("ends,NB", [((3000, 2200), 256), ((1500, 700), 256), ((9000, 5000), 2048)])
def test_full_tensor_core_group(ends, NB):
    # a large group of causal queries per sequence (a prefill chunk): the scores are one
    # tensor-core product; pools and top-k against the oracle per query
    r = np.random.default_rng(60 + ends[0] + NB)
    P, k, d_ik, H_i, G = 8, 128, 128, 8, 64
    n_vis = np.array([e - G + 1 + t for e in ends for t in range(G)], dtype=np.int32)
    seq_of = np.repeat(np.arange(len(ends)), G).astype(np.int32)
    cache, K, q, w = _setup(r, len(ends), int(n_vis.max()), d_ik, H_i, len(n_vis))
    got = _run_full_group(cache, q, w, seq_of, n_vis, NB, P, k, G)
    assert _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got) <= 16


def test_full_many_queries_one_cta_each():
    # 300 queries (the per-query selection runs one CTA per query from 256 queries on):
    # equal to the oracle, and bit for bit to the same queries in batches below 256
    r = np.random.default_rng(70)
    NB, P, k, d_ik, H_i = 256, 8, 128, 128, 8
    n_vis = r.integers(0, 6000, 300).astype(np.int32)
    n_vis[:6] = [0, 1, 127, 128, 129, NB * P]
    seq_of = (np.arange(300) % 3).astype(np.int32)
    cache, K, q, w = _setup(r, 3, int(n_vis.max()), d_ik, H_i, 300)
    got = _run_full(cache, q, w, seq_of, n_vis, NB, P, k)
    assert _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got) <= 16
    for lo, hi in ((0, 150), (150, 300)):
        part = csa2.index_full(cache, bf16_dev(q[lo:hi]), to_dev(w[lo:hi]), to_dev(seq_of[lo:hi]),
                               to_dev(n_vis[lo:hi]), int(n_vis.max()), NB, P, k)
        assert csa2.device_error() == 0
        for x, y in zip(got, part):
            np.testing.assert_array_equal(x[lo:hi], y.cpu().numpy())


def test_full_tensor_core_group_many_queries():
    # 2 x 256 causal queries: tensor-core scores and one CTA per query for the selection
    r = np.random.default_rng(71)
    P, k, d_ik, H_i, G, NB = 8, 256, 128, 8, 256, 512
    ends = (6000, 4500)
    n_vis = np.array([e - G + 1 + t for e in ends for t in range(G)], dtype=np.int32)
    seq_of = np.repeat(np.arange(len(ends)), G).astype(np.int32)
    cache, K, q, w = _setup(r, len(ends), int(n_vis.max()), d_ik, H_i, len(n_vis))
    got = _run_full_group(cache, q, w, seq_of, n_vis, NB, P, k, G)
    assert _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got) <= 32


@pytest.mark.parametrize("relu", [True, False])
def test_full_tensor_core_edges(relu):
    # tensor-core scoring with ragged and degenerate groups: queries with no entry, one
    # entry, fewer than a tile, a block each or fewer than per_block; groups whose queries
    # end in different tiles; 16 heads, two queries a tile (N = 32)
    r = np.random.default_rng(90 + relu)
    NB, P, k, d_ik, H_i, G = 64, 8, 64, 128, 16, 2
    n_vis = np.array([0, 1, 5, 127, 128, 129, 64, 511, 512, 513, 3000, 0], dtype=np.int32)
    seq_of = np.repeat(np.arange(len(n_vis) // G), G).astype(np.int32)
    cache, K, q, w = _setup(r, len(n_vis) // G, int(n_vis.max()), d_ik, H_i, len(n_vis))
    got = _run_full_group(cache, q, w, seq_of, n_vis, NB, P, k, G)
    if not relu:
        got = csa2.index_full(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), to_dev(n_vis), int(n_vis.max()),
                              NB, P, k, False, group=G)
        assert csa2.device_error() == 0
        got = tuple(t.cpu().numpy() for t in got)
    assert _compare_full(K, q, w, seq_of, n_vis, NB, P, k, got, relu) <= 4
    assert (got[1] == np.minimum(n_vis, NB * P)).all()


def test_exact_ties_break_to_lower_index():
    # a cache of only three distinct rows: scores tie exactly in large groups, so the
    # selection must follow the lower-index rule bit for bit.
    r = np.random.default_rng(20)
    NB, P, k, d_ik, H_i = 128, 8, 200, 128, 8
    n = 5000
    cache, _, q, w = _setup(r, 1, n, d_ik, H_i, 2)
    rows = synth.bf16_normal(r, (3, d_ik))
    K = rows[r.integers(0, 3, n)]
    pt = cache.page_table.cpu().numpy()
    cache.idx_k.copy_(bf16_dev(logical_to_paged([K], pt, cache.num_pages, d_ik, np.uint16)))
    n_vis = np.array([n, 3000], dtype=np.int32)
    seq_of = np.zeros(2, np.int32)
    pool, plen, topk, tlen = _run_full(cache, q, w, seq_of, n_vis, NB, P, k)
    for b in range(2):
        rpool, rtopk, s = indexer.full(formats.bf16_value(q[b]), w[b], formats.bf16_value(K[:n_vis[b]]), NB, P, k)
        np.testing.assert_array_equal(pool[b, :plen[b]], rpool)
        np.testing.assert_array_equal(topk[b, :tlen[b]], rtopk)


def _exact_score_problem(r, n, kinds):
    """Indexer K rows whose scores are exact in float32 whatever the summation order: every
    head's q is (1, 2^-12, 0, ...), every weight 1/8, and row i holds (A_i, B_i) in its first
    two dims (integers, exact in bf16) and random values elsewhere, so that its score is
    A_i + B_i / 4096.  kinds[s] picks sequence s's (A, B): 'low' -- A in {200, 201}, B in
    [0, 256): thousands of keys share their top 22 bits and ties are exact; 'spread' -- A in
    [1, 256), B = 0; 'flat' -- every score equal."""
    d_ik, H_i = 128, 8
    mp = (n + 63) // 64
    pt = synth.page_table(r, len(kinds), mp)
    K = []
    for kind in kinds:
        Kb = synth.bf16_normal(r, (n, d_ik)).astype(np.float32)
        if kind == "low":
            A, Bv = r.integers(200, 202, n), r.integers(0, 256, n)
        elif kind == "spread":
            A, Bv = r.integers(1, 256, n), np.zeros(n, np.int64)
        else:
            A, Bv = np.full(n, 37), np.full(n, 5)
        Kb[:, 0], Kb[:, 1] = A, Bv
        K.append(synth.bf16_bits_from_f32(Kb))
    cache = csa2.PagedCache.allocate(len(kinds), n, 512, d_ik, "cuda", torch.from_numpy(pt))
    cache.idx_k.copy_(bf16_dev(logical_to_paged(K, pt, len(kinds) * mp, d_ik, np.uint16)))
    qh = np.zeros((len(kinds), H_i, d_ik), np.float32)
    qh[:, :, 0], qh[:, :, 1] = 1.0, 2.0 ** -12
    q = synth.bf16_bits_from_f32(qh)
    w = np.full((len(kinds), H_i), 0.125, np.float32)
    return cache, K, q, w


@pytest.mark.parametrize("B", [3, 40, 300])
def test_select_resolves_every_key_bit(B):
    # scores exact on both sides, so the pool and the Top-k must equal the oracle's bit for
    # bit: the radix select must resolve keys that agree on their top 22 bits (all three of
    # its passes), stop early when a digit's keys are all taken, and break exact ties by
    # position, in the Full call's select and in Reindex.  At 40 queries Reindex runs its
    # 128-thread CTAs (40 clusters of 8 do not fit at two 256-thread CTAs an SM); from 256
    # queries on the Full call's Top-k is one CTA per query.
    r = np.random.default_rng(25 + B)
    NB, P, k, n = 2048, 8, 512, 40000
    kinds = ["low", "spread", "flat"]
    cache, K, q3, w3 = _exact_score_problem(r, n, kinds)
    seq_of = (np.arange(B) % 3).astype(np.int32)                 # query i reads sequence i % 3
    n_vis = np.array([n - 37 * (i // 3) - (777 if i % 3 == 1 else 0) for i in range(B)], dtype=np.int32)
    q, w = q3[seq_of], w3[seq_of]
    pool, plen, topk, tlen = _run_full(cache, q, w, seq_of, n_vis, NB, P, k)
    for b in range(B):
        Kb = formats.bf16_value(K[seq_of[b]][:n_vis[b]])
        rpool, rtopk, _ = indexer.full(formats.bf16_value(q[b]), w[b].astype(np.float64), Kb, NB, P, k)
        np.testing.assert_array_equal(pool[b, :plen[b]], rpool, err_msg=f"{b} {kinds[seq_of[b]]}")
        np.testing.assert_array_equal(topk[b, :tlen[b]], rtopk, err_msg=f"{b} {kinds[seq_of[b]]}")
    # Reindex over the same pools
    topk2, tlen2 = csa2.index_reindex(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), to_dev(pool), to_dev(plen), k)
    assert csa2.device_error() == 0
    topk2, tlen2 = topk2.cpu().numpy(), tlen2.cpu().numpy()
    for b in range(B):
        Kb = formats.bf16_value(K[seq_of[b]])
        rt, _ = indexer.reindex(formats.bf16_value(q[b]), w[b].astype(np.float64), Kb, pool[b, :plen[b]], k)
        np.testing.assert_array_equal(topk2[b, :tlen2[b]], rt, err_msg=f"{b} {kinds[seq_of[b]]}")


@pytest.mark.parametrize("H_i", [8, 12, 16, 32])
def test_reindex_matches_oracle(H_i):
    # one head group kept in registers (8), two (12, 16), or four streamed from L1 (32)
    r = np.random.default_rng(30 + H_i)
    NB, P, k, d_ik = 2048, 8, 512, 128
    n_vis = np.array([40000, 16384, 9000, 70000], dtype=np.int32)
    B = len(n_vis)
    cache, K, q_full, w_full = _setup(r, 4, int(n_vis.max()), d_ik, H_i, B)
    seq_of = np.arange(B, dtype=np.int32)
    stride = NB * P
    pools = np.full((B, stride), -1, dtype=np.int32)
    plen = np.zeros(B, dtype=np.int32)
    for b in range(B):
        rp, _, _ = indexer.full(formats.bf16_value(q_full[b]), w_full[b], formats.bf16_value(K[b][:n_vis[b]]),
                                NB, P, k)
        pools[b, :len(rp)] = rp
        plen[b] = len(rp)
    q = synth.bf16_normal(r, (B, H_i, d_ik))
    w = synth.f32_normal(r, (B, H_i), 1 / np.sqrt(H_i))
    topk, tlen = csa2.index_reindex(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), to_dev(pools), to_dev(plen), k)
    assert csa2.device_error() == 0
    topk, tlen = topk.cpu().numpy(), tlen.cpu().numpy()
    swaps = 0
    for b in range(B):
        Kb = formats.bf16_value(K[b])
        rt, rs = indexer.reindex(formats.bf16_value(q[b]), w[b], Kb, pools[b, :plen[b]], k)
        assert tlen[b] == len(rt)
        s_all = indexer.scores(formats.bf16_value(q[b]), w[b], Kb[pools[b, :plen[b]]])
        smap = dict(zip(pools[b, :plen[b]].tolist(), s_all.tolist()))
        swaps += check_index_set(topk[b, :tlen[b]], rt, lambda e: smap[e], f"reindex q{b}")
        assert set(topk[b, :tlen[b]].tolist()) <= set(pools[b, :plen[b]].tolist())
    assert swaps <= 4


def test_reindex_short_pools():
    r = np.random.default_rng(31)
    d_ik, H_i, k = 64, 4, 64
    cache, K, q, w = _setup(r, 1, 3000, d_ik, H_i, 3)
    pools = np.full((3, 512), -1, dtype=np.int32)
    plen = np.array([0, 40, 512], dtype=np.int32)
    pools[1, :40] = synth.sorted_distinct(r, 3000, 40)
    pools[2] = synth.sorted_distinct(r, 3000, 512)
    seq_of = np.zeros(3, np.int32)
    topk, tlen = csa2.index_reindex(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), to_dev(pools), to_dev(plen), k)
    topk, tlen = topk.cpu().numpy(), tlen.cpu().numpy()
    assert tlen.tolist() == [0, 40, 64]
    assert (topk[0] == -1).all()
    np.testing.assert_array_equal(topk[1, :40], pools[1, :40])
    Kb = formats.bf16_value(K[0])
    rt, _ = indexer.reindex(formats.bf16_value(q[2]), w[2], Kb, pools[2], k)
    s_all = indexer.scores(formats.bf16_value(q[2]), w[2], Kb)
    check_index_set(topk[2], rt, lambda e: s_all[e], "short pool")


def test_n_vis_beyond_max_n_is_flagged():
    r = np.random.default_rng(40)
    cache, K, q, w = _setup(r, 1, 1000, 64, 4, 1)
    n_vis = np.array([1000], dtype=np.int32)
    csa2.index_full(cache, bf16_dev(q), to_dev(w), to_dev(np.zeros(1, np.int32)), to_dev(n_vis), 900, 64, 8, 64)
    assert csa2.device_error() & 0x4


class _OffsetWorkspace(csa2.Workspace):
    """A workspace whose buffer starts 16 bytes past an aligned allocation."""

    def get(self, nbytes):
        return super().get(nbytes + 16)[16:]


def test_misaligned_workspace_is_rejected():
    r = np.random.default_rng(40)
    cache, K, q, w = _setup(r, 1, 3000, 128, 8, 2)
    n_vis = np.array([3000, 2000], dtype=np.int32)
    outs = [torch.full((2, 16384), -7, dtype=torch.int32, device="cuda"),
            torch.full((2,), -7, dtype=torch.int32, device="cuda"),
            torch.full((2, 512), -7, dtype=torch.int32, device="cuda"),
            torch.full((2,), -7, dtype=torch.int32, device="cuda")]
    with pytest.raises(csa2._lib.Csa2Error, match="256-byte aligned"):
        csa2.index_full(cache, bf16_dev(q), to_dev(w), to_dev(np.zeros(2, np.int32)), to_dev(n_vis), 3000,
                        out=outs, ws=_OffsetWorkspace("cuda"))
    torch.cuda.synchronize()
    assert all((o == -7).all() for o in outs)           # nothing was launched
