"""Parity at the benchmark's full sizes and in its launch configuration: one whole decode
step (append + the 20-layer schedule) of the N=131,072 / B=32 and N=1,048,576 / B=64
workloads (bf16 and FP8 indexer-K forms; the FP8 form's short-block scan at N=131,072), and of the mixed-context sweep (contexts of
4K..1M entries, batch 1..256), runs on the GPU.  Then, for every query of the step: its
appended entry is recomputed by the oracle, and the attention of every layer is recomputed
over the index set the GPU chose (the attention rule is stated given identical index sets),
with the index sets checked for validity; for sampled queries spread over the batch, the
oracle also recomputes every index set itself (from the same cache), and compares the
attention of the layers whose sets agree exactly (a near-tie swap, allowed by the index
rule, changes the attended set)."""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import synth, workload
from oracle import attention, compress, formats, indexer
from parity_utils import ATTN_MAX_ABS, ATTN_REL_L2, check_index_set, fp4_mismatch_is_tolerated, rel_l2

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _entries(step, b, e):
    """Main KV codes and scales (host) of entries e of query b's sequence, gathered on the
    device through the page table."""
    pt = step.cache.page_table[int(step.seq_of[b].item())]
    e = torch.as_tensor(np.asarray(e, dtype=np.int64), device=pt.device)
    pages, slots = pt[e // 64].long(), e % 64
    return step.cache.codes[pages, slots].cpu().numpy(), step.cache.scales[pages, slots].cpu().numpy(), (pages, slots)


def _assert_attention(step, b, l, codes, scales, topk, d):
    L = step.layers[l]
    q = formats.bf16_value(_bits(L["q"][b]))
    st, ln = int(L["swa_start"][b].item()), int(L["swa_len"][b].item())
    swa = L["swa"][st:st + ln].cpu().numpy()
    swa_scale = L["swa_scale"][st:st + ln].cpu().numpy()
    o, lse = attention.sparse_attention(q, codes, scales, topk, swa, swa_scale, 0, ln, 1 / np.sqrt(d))
    got = step.out[l][b].float().cpu().numpy()
    # bf16 output: half a bf16 ulp of rounding on top of the attention bar
    assert rel_l2(got, o) <= ATTN_REL_L2 + 2.0 ** -9, (b, l, rel_l2(got, o))
    assert (np.abs(got - o) <= ATTN_MAX_ABS + 2.0 ** -8 * np.abs(o)).all(), (b, l)
    np.testing.assert_allclose(step.lse[l][b].cpu().numpy(), lse, rtol=1e-4, atol=1e-4)


def _append_ref(step, info, b):
    """The oracle's own append of entry n-1 of query b's sequence from its hidden state."""
    n = int(info["Ns"][b // info.get("G", 1)])
    app = step.append
    Wkv = formats.bf16_value(_bits(app["W_kv"]))
    Wik = formats.bf16_value(_bits(app["W_ik"]))
    cos, sin = (t.cpu().numpy() for t in step.rope)
    H = formats.bf16_value(_bits(app["H"][b:b + 1]))
    return n, compress.compress_quant_from_hidden(H, Wkv, None, 1, np.array([n - 1]), cos, sin, info["d_rope"], Wik)


def _check_append(step, info, b):
    n, ref = _append_ref(step, info, b)
    codes, scales, (pg, sl) = _entries(step, b, [n - 1])
    bad, tol = fp4_mismatch_is_tolerated(ref["y"], codes, scales, ref["codes"], ref["scales"])
    assert bad == tol
    if info.get("ik8"):
        # indexer K is projected from the entry's FP4 form, so the oracle projects the GPU's own
        # entry (a tolerated FP4 code difference above changes the whole projection).  The GPU's
        # bf16 indexer K x_g is then within a bf16 ulp of the oracle's x_w, and each side's E4M3
        # rounding (a normal value) moves it by at most half a step, |x| / 16: so
        # |got - want| <= (|x_g| + |x_w|) / 16 + |x_g - x_w|, with |x| <= (17/16) |rounded x|;
        # values in the E4M3 subnormal range are within a subnormal step (2^-9 s) of either
        k8 = step.cache.idx_k8[pg, sl].cpu().numpy()
        ks = step.cache.idx_k8_scale[pg, sl].cpu().numpy()
        Wik = formats.bf16_value(_bits(step.append["W_ik"]))
        rb, rs = compress.index_k_fp8(compress.project_index_k(codes, scales, Wik))
        got, want = formats.fp8_rows_dequantize(k8, ks), formats.fp8_rows_dequantize(rb, rs)
        mag = np.maximum(np.abs(got), np.abs(want))
        tol = (17 / 16) * (np.abs(got) + np.abs(want)) / 16 + 2.0 ** -7 * mag + 2.0 ** -8 * rs[:, None] + 1e-30
        assert (np.abs(got - want) <= tol).all()


def _check_attention_of_gpu_sets(step, info, b):
    """Every layer of query b: its index set is valid, and its attention over that set
    matches the oracle's over the same set."""
    n = int(info["Ns"][b // info.get("G", 1)]) - info.get("G", 1) + 1 + b % info.get("G", 1)
    for l in range(len(step.layers)):
        gtk, gtl = step.result_topk(l)
        g = gtk[b].cpu().numpy()[:int(gtl[b].item())]
        assert len(g) == min(info["k"], n, info["NB"] * info["P"])
        assert (np.diff(g) > 0).all() and g.min() >= 0 and g.max() < n
        assert (gtk[b].cpu().numpy()[len(g):] == -1).all()
        codes, scales, _ = _entries(step, b, g)
        _assert_attention(step, b, l, codes, scales, np.arange(len(g)), info["d"])


def _check_query(step, info, b):
    """Recompute query b's index set of every Full / Reindex / Reuse layer with the oracle
    from the same cache (its own appended entry in place of the GPU's), and the attention of
    every layer whose set agrees.  Returns (tolerated swaps, attention layers compared)."""
    n, ref = _append_ref(step, info, b)
    d, k = info["d"], info["k"]
    codes, scales, idxk = workload.host_sequence(step, b, n)
    codes[n - 1], scales[n - 1] = ref["codes"][0], ref["scales"][0]
    if info.get("ik8"):
        k8, ks = idxk
        rb, rs = compress.index_k_fp8(ref["idx_k"])
        k8[n - 1], ks[n - 1] = rb[0], rs[0]
    else:
        idxk[n - 1] = ref["idx_k"][0]
        K = formats.bf16_value(idxk)
    pool = topk = None
    swaps = compared = 0
    for l, L in enumerate(step.layers):
        mode = L["mode"]
        gtk, gtl = step.result_topk(l)
        g = gtk[b].cpu().numpy()[:int(gtl[b].item())]
        if mode in ("full", "reindex"):
            qi = formats.bf16_value(_bits(L["q_idx"][b]))
            w = L["w"][b].cpu().numpy().astype(np.float64)
            if info.get("ik8"):
                qi, K = indexer.fp8_form(qi, k8, ks)
        if mode == "full":
            pool, topk, sc = indexer.full(qi, w, K, info["NB"], info["P"], k)
            swaps += check_index_set(g, topk, lambda e: sc[e], f"q{b} n={n} layer {l} full")
            gp = step.pool[b].cpu().numpy()[:int(step.pool_len[b].item())]
            assert len(gp) == len(pool) == min(n, info["NB"] * info["P"])
        elif mode == "reindex":
            topk, ps = indexer.reindex(qi, w, K, pool, k)
            smap = dict(zip(pool.tolist(), ps.tolist()))
            swaps += check_index_set(g, topk, lambda e: smap[e], f"q{b} n={n} layer {l} reindex")
        else:
            topk = indexer.reuse(topk)
        if not np.array_equal(g, topk):
            continue
        _assert_attention(step, b, l, codes, scales, topk, d)
        compared += 1
    return swaps, compared


@pytest.mark.parametrize("cfg,samples", [(synth.DEC128K, [0, 17, 31]), (synth.DEC1M, [0, 21, 42, 63]),
                                         (synth.DEC128K_IK8, [3, 29]), (synth.DEC1M_IK8, [5, 50])])
def test_decode_step_full_size(cfg, samples):
    step, info = workload.build_decode(cfg, seed=7)
    step.run()
    torch.cuda.synchronize()
    for b in range(info["B"]):                  # every query: its append and its attention
        _check_append(step, info, b)
        _check_attention_of_gpu_sets(step, info, b)
    swaps = compared = 0
    for b in samples:                           # sampled queries: the index sets themselves
        s_, c_ = _check_query(step, info, b)
        swaps += s_
        compared += c_
    assert swaps <= 4 * len(samples)
    assert compared >= 15 * len(samples)


@pytest.mark.parametrize("B", [1, 37, 256])
def test_decode_step_mixed_contexts(B):
    """The batched paged decode sweep: each sequence's context drawn from {4K, 64K, 256K,
    1M} entries (a 4K context is shorter than the 16,384-entry pool: the pool is then the
    whole range), one 20-layer step at batch B; one sampled query per context length."""
    ctx = [4096, 65536, 262144, 1048576]
    r = np.random.default_rng(900 + B)
    Ns = r.choice(ctx, size=B)
    if B >= len(ctx):
        Ns[:len(ctx)] = ctx                     # every length present
    step, info = workload.build_decode(synth.DEC1M, Ns=Ns, seed=11 + B)
    step.run()
    torch.cuda.synchronize()
    samples = sorted({int(np.nonzero(Ns == c)[0][0]) for c in set(Ns.tolist())})
    swaps = compared = 0
    for b in samples:
        s_, c_ = _check_query(step, info, b)
        swaps += s_
        compared += c_
    assert swaps <= 4 * len(samples)
    assert compared >= 15 * len(samples)
