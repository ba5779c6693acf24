"""GPU parity of the compressed (FP8) indexer-K form: the compressor writes each entry's
indexer K as E4M3 bytes with one float32 scale (bit for bit the oracle's quantiser applied
to the bf16 indexer K the same kernels write in the bf16 form), and the Full and Reindex
indexers score FP8 queries against it, compared with the oracle indexer over the
dequantised values under the near-tie rule."""
import math

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import csa2, synth
from oracle import compress, formats, indexer
from parity_utils import bf16_dev, bf16_host_bits, check_index_set, logical_to_paged, to_dev

pytestmark = pytest.mark.gpu


# ---- the writers: every indexer-K path of the compressor -----------------------------------

def _compress_both(run):
    """Run the same compressor call on a bf16-form and an FP8-form cache; return the bf16
    plane and the FP8 bytes and scales, all entry-major [pages * 64, ...]."""
    c16, c8 = run(False), run(True)
    ik = bf16_host_bits(c16.idx_k).reshape(-1, c16.idx_k.shape[-1])
    k8 = c8.idx_k8.cpu().numpy().reshape(-1, c8.idx_k8.shape[-1])
    ks = c8.idx_k8_scale.cpu().numpy().reshape(-1)
    np.testing.assert_array_equal(c16.codes.cpu().numpy(), c8.codes.cpu().numpy())
    return ik, k8, ks


def _check_fp8_of_bf16(ik, k8, ks, used):
    want_b, want_s = compress.index_k_fp8(ik[used])
    np.testing.assert_array_equal(ks[used].view(np.uint32), want_s.view(np.uint32))
    np.testing.assert_array_equal(k8[used], want_b)


@pytest.mark.parametrize("G,d,d_ik", [(37, 512, 128), (300, 128, 64), (2100, 512, 64), (2100, 512, 128)])
def test_fp8_index_k_given_rows(G, d, d_ik):
    # G < 2048 without the tensor-core projection: quantisation and indexer K in one launch;
    # 2,100 entries at d_ik = 64: eight entries a CTA; at d_ik = 128: the tensor-core kernel
    r = np.random.default_rng(1300 + G + d_ik)
    C = r.standard_normal((G, d)).astype(np.float32)
    Wik = synth.bf16_normal(r, (d, d_ik), 1 / np.sqrt(d))
    pt = synth.page_table(r, 1, (G + 63) // 64)

    def run(fp8):
        cache = csa2.PagedCache.allocate(1, G, d, d_ik, "cuda", torch.from_numpy(pt), idx_k_fp8=fp8)
        csa2.compress_quant(cache, to_dev(np.zeros(G, np.int32)), to_dev(np.arange(G, dtype=np.int32)), m=1,
                            C=to_dev(C), W_ik=bf16_dev(Wik))
        assert csa2.device_error() == 0
        return cache

    ik, k8, ks = _compress_both(run)
    e = np.arange(G)
    _check_fp8_of_bf16(ik, k8, ks, pt[0, e // 64] * 64 + e % 64)


def test_fp8_index_k_prefill_projection_and_append():
    # the fused tensor-core projection of many tokens (m = 2), and the decode append
    r = np.random.default_rng(1400)
    T, m, d, d_model, d_ik = 4096, 2, 512, 512, 128
    G = T // m
    H = bf16_dev(synth.bf16_normal(r, (T, d_model)))
    Wkv = bf16_dev(synth.bf16_normal(r, (d_model, d), 1 / math.sqrt(d_model)))
    Wz = bf16_dev(synth.bf16_normal(r, (d_model, d), 1 / math.sqrt(d_model)))
    Wik = bf16_dev(synth.bf16_normal(r, (d, d_ik), 1 / math.sqrt(d)))
    cos, sin = (to_dev(t) for t in synth.rope_tables(T, 64))
    pt = synth.page_table(r, 1, G // 64)

    def run(fp8):
        cache = csa2.PagedCache.allocate(1, G, d, d_ik, "cuda", torch.from_numpy(pt), idx_k_fp8=fp8)
        csa2.compress_quant(cache, to_dev(np.zeros(G, np.int32)), to_dev(np.arange(G, dtype=np.int32)), m=m, H=H,
                            W_kv=Wkv, W_z=Wz, pos=to_dev((np.arange(G) * m + m - 1).astype(np.int32)),
                            rope_cos=cos, rope_sin=sin, W_ik=Wik)
        assert csa2.device_error() == 0
        return cache

    ik, k8, ks = _compress_both(run)
    e = np.arange(G)
    _check_fp8_of_bf16(ik, k8, ks, pt[0, e // 64] * 64 + e % 64)

    B = 6
    pt2 = synth.page_table(r, B, 1)
    Hb = bf16_dev(synth.bf16_normal(r, (B, d_model)))

    def run_append(fp8):
        cache = csa2.PagedCache.allocate(B, 64, d, d_ik, "cuda", torch.from_numpy(pt2), idx_k_fp8=fp8)
        csa2.compress_append(cache, Hb, to_dev(np.arange(B, dtype=np.int32)), to_dev(np.full(B, 9, np.int32)), Wkv,
                             rope_cos=cos, rope_sin=sin, W_ik=Wik)
        assert csa2.device_error() == 0
        return cache

    ik, k8, ks = _compress_both(run_append)
    _check_fp8_of_bf16(ik, k8, ks, pt2[:, 0] * 64 + 9)


# ---- the readers: Full and Reindex over an FP8 cache ----------------------------------------

def _setup8(r, ns, n_max, d_ik, H_i, B):
    """ns sequences of n_max entries: N(0,1) bf16 indexer-K rows quantised by the oracle's
    FP8 row quantiser, paged through a random page table; B queries with random q / w."""
    mp = (n_max + 63) // 64
    pt = synth.page_table(r, ns, mp)
    K8, Ks = [], []
    for _ in range(ns):
        b, s = compress.index_k_fp8(synth.bf16_normal(r, (n_max, d_ik)))
        K8.append(b)
        Ks.append(s)
    cache = csa2.PagedCache.allocate(ns, n_max, 512, d_ik, "cuda", torch.from_numpy(pt), idx_k_fp8=True)
    cache.idx_k8.copy_(to_dev(logical_to_paged(K8, pt, ns * mp, d_ik, np.uint8)))
    cache.idx_k8_scale.copy_(to_dev(logical_to_paged([s[:, None] for s in Ks], pt, ns * mp, 1, np.float32)[..., 0]))
    q = synth.bf16_normal(r, (B, H_i, d_ik))
    w = synth.f32_normal(r, (B, H_i), 1 / np.sqrt(H_i))
    return cache, K8, Ks, q, w


def _compare_full8(K8, Ks, q, w, seq_of, n_vis, NB, P, k, got, relu=True):
    pool, plen, topk, tlen = got
    swaps = 0
    for b in range(len(n_vis)):
        n = int(n_vis[b])
        qh, Kh = indexer.fp8_form(formats.bf16_value(q[b]), K8[seq_of[b]][:n], Ks[seq_of[b]][:n])
        rpool, rtopk, s = indexer.full(qh, w[b], Kh, NB, P, k, relu)
        assert plen[b] == len(rpool) and tlen[b] == len(rtopk)
        assert (pool[b, plen[b]:] == -1).all() and (topk[b, tlen[b]:] == -1).all()
        score = lambda e: s[e]
        gp = pool[b, :plen[b]]
        if n >= NB * P:
            bb = indexer.block_bounds(n, NB)
            for j in range(NB):
                seg = gp[P * j:P * j + P]
                assert ((seg >= bb[j]) & (seg < bb[j + 1])).all()
                swaps += check_index_set(seg, rpool[P * j:P * j + P], score, f"q{b} block {j}")
        else:
            np.testing.assert_array_equal(gp, rpool)
        swaps += check_index_set(topk[b, :tlen[b]], rtopk, score, f"q{b} topk")
    return swaps


@pytest.mark.parametrize("d_ik,H_i,NB,P,k,relu", [(128, 8, 2048, 8, 512, True), (64, 4, 64, 8, 64, True),
                                                  (128, 16, 256, 8, 128, True), (128, 32, 256, 8, 128, True),
                                                  (128, 12, 512, 8, 256, False), (128, 1, 128, 8, 64, True)])
def test_fp8_full(d_ik, H_i, NB, P, k, relu):
    r = np.random.default_rng(1500 + d_ik + H_i + NB)
    n_vis = np.array([0, 5, 777, NB * P - 1, NB * P, 20011, 50000], dtype=np.int32)
    B = len(n_vis)
    cache, K8, Ks, q, w = _setup8(r, 2, int(n_vis.max()), d_ik, H_i, B)
    seq_of = (np.arange(B) % 2).astype(np.int32)
    got = csa2.index_full(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), to_dev(n_vis), int(n_vis.max()), NB, P, k,
                          relu)
    assert csa2.device_error() == 0
    got = [t.cpu().numpy() for t in got]
    assert _compare_full8(K8, Ks, q, w, seq_of, n_vis, NB, P, k, got, relu) <= 8


@pytest.mark.parametrize("group", [2, 6])
def test_fp8_full_grouped(group):
    r = np.random.default_rng(1600 + group)
    NB, P, k, d_ik, H_i = 2048, 8, 512, 128, 8
    ends = [20000, 70001]
    n_vis = np.array([e - group + 1 + t for e in ends for t in range(group)], dtype=np.int32)
    seq_of = np.repeat(np.arange(2), group).astype(np.int32)
    B = len(n_vis)
    cache, K8, Ks, q, w = _setup8(r, 2, int(n_vis.max()), d_ik, H_i, B)
    got = csa2.index_full(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), to_dev(n_vis), int(n_vis.max()), NB, P, k,
                          group=group)
    assert csa2.device_error() == 0
    got = [t.cpu().numpy() for t in got]
    assert _compare_full8(K8, Ks, q, w, seq_of, n_vis, NB, P, k, got) <= 8


@pytest.mark.parametrize("H_i", [8, 32])
def test_fp8_reindex(H_i):
    r = np.random.default_rng(1700 + H_i)
    NB, P, k, d_ik = 2048, 8, 512, 128
    n_vis = np.array([60000, 16384, 9000, 131072], dtype=np.int32)
    B = len(n_vis)
    cache, K8, Ks, q, w = _setup8(r, 2, int(n_vis.max()), d_ik, H_i, B)
    seq_of = (np.arange(B) % 2).astype(np.int32)
    # the pool of a Full call (any index set works: Reindex scores whatever pool it is given)
    q0 = synth.bf16_normal(r, (B, H_i, d_ik))
    pool, plen, _, _ = csa2.index_full(cache, bf16_dev(q0), to_dev(w), to_dev(seq_of), to_dev(n_vis), int(n_vis.max()),
                                       NB, P, k)
    topk, tlen = csa2.index_reindex(cache, bf16_dev(q), to_dev(w), to_dev(seq_of), pool, plen, k)
    assert csa2.device_error() == 0
    pool, plen, topk, tlen = (t.cpu().numpy() for t in (pool, plen, topk, tlen))
    swaps = 0
    for b in range(B):
        pb = pool[b, :plen[b]]
        qh, Kh = indexer.fp8_form(formats.bf16_value(q[b]), K8[seq_of[b]], Ks[seq_of[b]])
        rt, s = indexer.reindex(qh, w[b], Kh, pb, k)
        sc = dict(zip(pb.tolist(), s))
        assert tlen[b] == len(rt)
        swaps += check_index_set(topk[b, :tlen[b]], rt, lambda e: sc[int(e)], f"q{b} reindex")
    assert swaps <= 4
