"""Parity of the encoder prefill chunk at its full size (65,536 tokens at m = 2, 8,192
causal query tokens), in two stages with independent inputs:

  * the compressor: C = H.W_KV, Z = H.W_Z, two-token softmax pooling, RoPE, FP4 and the
    indexer-K projection of all 32,768 entries on the GPU; 24 sampled groups recomputed
    by the oracle from the same hidden states;
  * one group [Full, Reuse x 5] of index + attention for the 8,192 query tokens over a
    32,768-entry cache (query token t sees the (t + 1) // 2 entries complete at t, and its
    window is its own last 128 tokens); the first, middle and last queries recomputed by
    the oracle.
The chunk's three groups repeat the second stage with other weights; one is checked."""
import math

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import csa2, synth
from fp4_compressed_sparse_02_gb300.schedule import FULL, REUSE, DecodeStep
from oracle import attention, compress, formats, indexer
from parity_utils import (ATTN_MAX_ABS, ATTN_REL_L2, check_index_k, check_index_set, fp4_mismatch_is_tolerated,
                          projection_error_bound, rel_l2)

pytestmark = pytest.mark.gpu
CFG = synth.PREFILL


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _randn_bf16(shape, g, sigma=1.0):
    return (torch.randn(shape, generator=g, device="cuda") * sigma).to(torch.bfloat16)


def test_prefill_compressor_full_size():
    T, m, d, d_model, d_ik, d_rope = (CFG[x] for x in ("T", "m", "d", "d_model", "d_ik", "d_rope"))
    G = T // m
    g = torch.Generator(device="cuda").manual_seed(21)
    H = _randn_bf16((T, d_model), g)
    Wkv = _randn_bf16((d_model, d), g, 1 / math.sqrt(d_model))
    Wz = _randn_bf16((d_model, d), g, 1 / math.sqrt(d_model))
    Wik = _randn_bf16((d, d_ik), g, 1 / math.sqrt(d))
    pt = torch.randperm(G // 64, generator=torch.Generator().manual_seed(21)).to(torch.int32).reshape(1, -1)
    cache = csa2.PagedCache.allocate(1, G, d, d_ik, "cuda", pt)
    cos, sin = synth.rope_tables(T, d_rope)
    pos = (np.arange(G) * m + m - 1).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    y = torch.empty((G, d), dtype=torch.float32, device="cuda")
    csa2.compress_quant(cache, dev(np.zeros(G, np.int32)), dev(np.arange(G, dtype=np.int32)), m=m, H=H, W_kv=Wkv,
                        W_z=Wz, pos=dev(pos), rope_cos=dev(cos), rope_sin=dev(sin), W_ik=Wik, y_out=y)
    torch.cuda.synchronize()
    assert csa2.device_error() == 0
    # the quantiser rule over every entry: the FP4 bytes are exactly those of the GPU's own
    # float32 rows
    yg_all = y.cpu().numpy()
    e_all = np.arange(G)
    pg_all = pt[0].numpy()[e_all // 64]
    c_own, s_own = formats.fp4_quantize(yg_all)
    np.testing.assert_array_equal(cache.scales.cpu().numpy()[pg_all, e_all % 64], s_own)
    np.testing.assert_array_equal(cache.codes.cpu().numpy()[pg_all, e_all % 64], c_own)
    r = np.random.default_rng(21)
    sel = np.unique(np.concatenate([[0, G - 1], r.choice(G, 22, replace=False)]))
    rows = np.stack([m * sel + j for j in range(m)], 1).reshape(-1)
    Hs = formats.bf16_value(_bits(H[torch.from_numpy(rows).cuda()]))
    Wkv_h, Wz_h, Wik_h = (formats.bf16_value(_bits(w)) for w in (Wkv, Wz, Wik))
    ref = compress.compress_quant_from_hidden(Hs, Wkv_h, Wz_h, m, pos[sel], cos, sin, d_rope, Wik_h)
    pages = pt[0].numpy()[sel // 64]
    codes = cache.codes[torch.from_numpy(pages).long().cuda(), torch.from_numpy(sel % 64).long().cuda()].cpu().numpy()
    scales = cache.scales[torch.from_numpy(pages).long().cuda(), torch.from_numpy(sel % 64).long().cuda()].cpu().numpy()
    idxk = cache.idx_k[torch.from_numpy(pages).long().cuda(), torch.from_numpy(sel % 64).long().cuda()]
    # the sampled rows against the oracle: the measured error, within the float32 summation
    # bound; FP4 groups may differ from the oracle's only where that error reaches a decision
    err = np.abs(yg_all[sel].astype(np.float64) - ref["y"])
    assert err.max() <= 1e-5 * np.abs(ref["y"]).max(), err.max()
    C = compress.project(Hs, Wkv_h)
    Z = compress.project(Hs, Wz_h)
    bound = projection_error_bound(Hs, Wkv_h, Wz_h, m, d_rope, C, Z)
    assert (err <= bound + 4 * np.spacing(np.abs(ref["y"]).astype(np.float32))).all()
    bad, tol = fp4_mismatch_is_tolerated(ref["y"], codes, scales, ref["codes"], ref["scales"], err)
    assert bad == tol and bad <= max(2, 0.002 * len(sel) * d / 16)
    same = (codes == ref["codes"]).all(1) & (scales == ref["scales"]).all(1)
    check_index_k(_bits(idxk)[same], ref["idx_k"][same], ref["codes"][same], ref["scales"][same], Wik_h)


def test_prefill_index_attention_full_size():
    T, m, d, Hq, H_i, d_ik = (CFG[x] for x in ("T", "m", "d", "Hq", "H_i", "d_ik"))
    Q, W, k, NB, P = (CFG[x] for x in ("Q", "W", "k", "NB", "P"))
    NE = T // m
    g = torch.Generator(device="cuda").manual_seed(31)
    pages = NE // 64
    pt = torch.randperm(pages, generator=torch.Generator().manual_seed(31)).to(torch.int32).reshape(1, -1).cuda()
    cache = csa2.PagedCache(codes=torch.randint(0, 256, (pages, 64, d // 2), generator=g, device="cuda",
                                                dtype=torch.uint8),
                            scales=torch.randint(0x20, 0x40, (pages, 64, d // 16), generator=g, device="cuda",
                                                 dtype=torch.uint8),
                            idx_k=_randn_bf16((pages, 64, d_ik), g), page_table=pt)
    tq = T - Q + np.arange(Q)                              # token positions of the queries
    n_vis = ((tq + 1) // m).astype(np.int32)               # entries complete at the query
    layers = []
    for mode in [FULL] + [REUSE] * 5:
        sign = torch.randint(0, 2, (T, d), generator=g, device="cuda", dtype=torch.int32) << 7
        expo = torch.randint(3, 14, (T, d), generator=g, device="cuda", dtype=torch.int32) << 3
        man = torch.randint(0, 8, (T, d), generator=g, device="cuda", dtype=torch.int32)
        L = dict(mode=mode, q=_randn_bf16((Q, Hq, d), g), swa=(sign | expo | man).to(torch.uint8),
                 swa_scale=(torch.rand(T, generator=g, device="cuda") * 0.015 + 0.005).float(),
                 swa_start=torch.from_numpy((tq - (W - 1)).astype(np.int32)).cuda(),
                 swa_len=torch.full((Q,), W, dtype=torch.int32, device="cuda"))
        if mode == FULL:
            L["q_idx"] = _randn_bf16((Q, H_i, d_ik), g)
            L["w"] = torch.randn((Q, H_i), generator=g, device="cuda") / math.sqrt(H_i)
        layers.append(L)
    # the chunk's queries form one group: the Full scores are one tensor-core product
    step = DecodeStep(cache, torch.zeros(Q, dtype=torch.int32, device="cuda"), torch.from_numpy(n_vis).cuda(), NE,
                      layers, NB, P, k, W, group=Q)
    step.run()
    torch.cuda.synchronize()
    assert csa2.device_error() == 0
    e = np.arange(NE)
    pg = pt[0].cpu().numpy()[e // 64]
    codes_all = cache.codes.cpu().numpy()[pg, e % 64]
    scales_all = cache.scales.cpu().numpy()[pg, e % 64]
    K_all = formats.bf16_value(_bits(cache.idx_k).reshape(pages, 64, d_ik)[pg, e % 64])
    swaps = compared = 0
    for b in (0, Q // 2, Q - 1):
        n = int(n_vis[b])
        codes, scales, K = codes_all[:n], scales_all[:n], K_all[:n]
        topk = None
        for l, L in enumerate(layers):
            gtk, gtl = step.result_topk(l)
            got = gtk[b].cpu().numpy()[:int(gtl[b].item())]
            if L["mode"] == FULL:
                qi = formats.bf16_value(_bits(L["q_idx"][b]))
                w = L["w"][b].cpu().numpy().astype(np.float64)
                pool, topk, sc = indexer.full(qi, w, K, NB, P, k)
                swaps += check_index_set(got, topk, lambda x: sc[x], f"query {b} (n={n}) Full")
                assert int(step.pool_len[b].item()) == len(pool)
            else:
                topk = indexer.reuse(topk)
            if not np.array_equal(got, topk):
                continue
            q = formats.bf16_value(_bits(L["q"][b]))
            o, lse = attention.sparse_attention(q, codes, scales, topk, L["swa"].cpu().numpy(),
                                                L["swa_scale"].cpu().numpy(), int(tq[b]) - (W - 1), W,
                                                1 / np.sqrt(d))
            out = step.out[l][b].float().cpu().numpy()
            assert rel_l2(out, o) <= ATTN_REL_L2 + 2.0 ** -9, (b, l, rel_l2(out, o))
            assert (np.abs(out - o) <= ATTN_MAX_ABS + 2.0 ** -8 * np.abs(o)).all(), (b, l)
            np.testing.assert_allclose(step.lse[l][b].cpu().numpy(), lse, rtol=1e-4, atol=1e-4)
            compared += 1
    assert swaps <= 12
    assert compared >= 15
