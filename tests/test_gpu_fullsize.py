"""Parity at the benchmark's full sizes and in its launch configuration: one whole decode
step (append + the 20-layer schedule) of the N=131,072 / B=32 and N=1,048,576 / B=64
workloads, and of the mixed-context sweep (contexts of 4K..1M entries, batch 1..256),
runs on the GPU; sampled queries are then recomputed one by one by the oracle from the
same inputs.  The oracle computes its own appended entry and its own index
sets; attention outputs are compared for the layers whose index sets agree exactly (a
near-tie swap, allowed by the index rule, changes the attended set)."""
import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import synth, workload
from oracle import attention, compress, formats, indexer
from parity_utils import ATTN_MAX_ABS, ATTN_REL_L2, check_index_set, fp4_mismatch_is_tolerated, rel_l2

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_query(step, info, b):
    """Recompute query b of the step with the oracle: its appended entry, its index set of
    every Full / Reindex / Reuse layer, and the attention of every layer whose set agrees.
    Returns (tolerated swaps, attention layers compared)."""
    n = int(info["Ns"][b])
    d, k = info["d"], info["k"]
    tau = 1 / np.sqrt(d)
    app = step.append
    Wkv = formats.bf16_value(_bits(app["W_kv"]))
    Wik = formats.bf16_value(_bits(app["W_ik"]))
    cos, sin = (t.cpu().numpy() for t in step.rope)
    codes, scales, idxk = workload.host_sequence(step, b, n)
    # the oracle's own append of entry n-1 from this query's hidden state
    H = formats.bf16_value(_bits(app["H"][b:b + 1]))
    ref = compress.compress_quant_from_hidden(H, Wkv, None, 1, np.array([n - 1]), cos, sin, info["d_rope"], Wik)
    bad, tol = fp4_mismatch_is_tolerated(ref["y"], codes[n - 1:n], scales[n - 1:n], ref["codes"], ref["scales"])
    assert bad == tol
    codes[n - 1], scales[n - 1], idxk[n - 1] = ref["codes"][0], ref["scales"][0], ref["idx_k"][0]
    K = formats.bf16_value(idxk)
    pool = topk = None
    swaps = compared = 0
    for l, L in enumerate(step.layers):
        mode = L["mode"]
        gtk, gtl = step.result_topk(l)
        g = gtk[b].cpu().numpy()[:int(gtl[b].item())]
        if mode == "full":
            qi = formats.bf16_value(_bits(L["q_idx"][b]))
            w = L["w"][b].cpu().numpy().astype(np.float64)
            pool, topk, sc = indexer.full(qi, w, K, info["NB"], info["P"], k)
            swaps += check_index_set(g, topk, lambda e: sc[e], f"q{b} n={n} layer {l} full")
            gp = step.pool[b].cpu().numpy()[:int(step.pool_len[b].item())]
            assert len(gp) == len(pool) == min(n, info["NB"] * info["P"])
        elif mode == "reindex":
            qi = formats.bf16_value(_bits(L["q_idx"][b]))
            w = L["w"][b].cpu().numpy().astype(np.float64)
            topk, ps = indexer.reindex(qi, w, K, pool, k)
            smap = dict(zip(pool.tolist(), ps.tolist()))
            swaps += check_index_set(g, topk, lambda e: smap[e], f"q{b} n={n} layer {l} reindex")
        else:
            topk = indexer.reuse(topk)
        if not np.array_equal(g, topk):
            continue
        q = formats.bf16_value(_bits(L["q"][b]))
        swa = L["swa"].cpu().numpy()
        swa_scale = L["swa_scale"].cpu().numpy()
        st = int(L["swa_start"][b].item())
        ln = int(L["swa_len"][b].item())
        o, lse = attention.sparse_attention(q, codes, scales, topk, swa, swa_scale, st, ln, tau)
        got = step.out[l][b].float().cpu().numpy()
        # bf16 output: half a bf16 ulp of rounding on top of the attention bar
        assert rel_l2(got, o) <= ATTN_REL_L2 + 2.0 ** -9, (b, l, rel_l2(got, o))
        assert (np.abs(got - o) <= ATTN_MAX_ABS + 2.0 ** -8 * np.abs(o)).all(), (b, l)
        np.testing.assert_allclose(step.lse[l][b].cpu().numpy(), lse, rtol=1e-4, atol=1e-4)
        compared += 1
    return swaps, compared


@pytest.mark.parametrize("cfg,samples", [(synth.DEC128K, [0, 17]), (synth.DEC1M, [5])])
def test_decode_step_full_size(cfg, samples):
    step, info = workload.build_decode(cfg, seed=7)
    step.run()
    torch.cuda.synchronize()
    swaps = compared = 0
    for b in samples:
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
