"""csa2_index_full_noalloc: the Full indexer for callers that cannot allocate device
memory (for example a server whose HBM is already carved into KV pages, or a host
runtime that reaches the library only through the C ABI and has no CUDA allocator).
Its candidate scores live in a fixed array inside the library instead of a caller
workspace.  Through the C ABI, two calls in a row must give exactly what the
workspace-based csa2_index_full gives on the same inputs.

This file is named to be collected last, so that a run stopping at the first failure
has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import _lib, csa2, synth
from oracle import formats, indexer
from parity_utils import bf16_dev, check_index_set, logical_to_paged, to_dev

pytestmark = pytest.mark.gpu


def _args(cache, q, w, seq_of, n_vis, max_n, NB, P, k, outs, group=1):
    a = _lib.IndexFullArgs()
    a.struct_size = ctypes.sizeof(_lib.IndexFullArgs)
    a.B, a.H_i = q.shape[0], q.shape[1]
    a.q_idx, a.w = q.data_ptr(), w.data_ptr()
    a.cache = cache.c_struct()
    a.seq_of, a.n_vis, a.max_n = seq_of.data_ptr(), n_vis.data_ptr(), max_n
    a.num_blocks, a.per_block, a.k, a.relu = NB, P, k, 1
    a.pool, a.pool_len, a.topk, a.topk_len = (t.data_ptr() for t in outs)
    a.group = group
    return a


def _outs(B, NB, P, k):
    return [torch.full((B, NB * P), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, k), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda")]


def _problem(seed, B, n_max, NB, P, k, H_i=8, group=1, host=False):
    r = np.random.default_rng(seed)
    d_ik = 128
    mp = (n_max + 63) // 64
    pt = synth.page_table(r, 2, mp)
    K = [synth.bf16_normal(r, (n_max, d_ik)) for _ in range(2)]
    cache = csa2.PagedCache.allocate(2, n_max, 128, d_ik, "cuda", torch.from_numpy(pt))
    cache.idx_k.copy_(bf16_dev(logical_to_paged(K, pt, 2 * mp, d_ik, np.uint16)))
    qh = synth.bf16_normal(r, (B, H_i, d_ik))
    wh = synth.f32_normal(r, (B, H_i), 0.35)
    seq = ((np.arange(B) // group) % 2).astype(np.int32)
    nv = r.integers(1, n_max + 1, size=B).astype(np.int32)
    out = (cache, bf16_dev(qh), to_dev(wh), to_dev(seq), to_dev(nv))
    if host:
        out += (dict(K=K, q=qh, w=wh, seq=seq, n_vis=nv),)
    return out


def _workspace_call(L, a, stream):
    need = ctypes.c_size_t(0)
    _lib.check(L.csa2_index_full_workspace(ctypes.byref(a), ctypes.byref(need)))
    ws = torch.empty(max(1, need.value), dtype=torch.uint8, device="cuda")
    _lib.check(L.csa2_index_full(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), need.value, stream))
    torch.cuda.synchronize()


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    L = _lib.lib()
    NB, P, k = 2048, 8, 512
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (seed, B, n_max) in enumerate([(1, 6, 60000), (2, 3, 20000)]):
        cache, q, w, seq_of, n_vis = _problem(seed, B, n_max, NB, P, k)
        ref = _outs(B, NB, P, k)
        a = _args(cache, q, w, seq_of, n_vis, n_max, NB, P, k, ref)
        need = ctypes.c_size_t(0)
        _lib.check(L.csa2_index_full_workspace(ctypes.byref(a), ctypes.byref(need)))
        ws = torch.empty(need.value, dtype=torch.uint8, device="cuda")
        _lib.check(L.csa2_index_full(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), need.value, stream))
        got = _outs(B, NB, P, k)
        b = _args(cache, q, w, seq_of, n_vis, n_max, NB, P, k, got)
        _lib.check(L.csa2_index_full_noalloc(ctypes.byref(b), stream))
        torch.cuda.synchronize()
        for x, y in zip(got, ref):
            assert torch.equal(x, y), f"call {call}: allocation-free result differs"
        assert (got[1] > 0).all() and (got[3] > 0).all()


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    L = _lib.lib()
    NB, P, k = 2048, 8, 512
    B = (1 << 20) // (NB * P) + 1            # one query more than the array holds
    cache, q, w, seq_of, n_vis = _problem(3, B, 4096, NB, P, k)
    outs = _outs(B, NB, P, k)
    a = _args(cache, q, w, seq_of, n_vis, 4096, NB, P, k, outs)
    st = L.csa2_index_full_noalloc(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 2
    assert b"fixed scratch" in L.csa2_last_error_message()
    torch.cuda.synchronize()
    assert (outs[3] == -7).all()                           # nothing was launched


def _device_error_word(L):
    word = ctypes.c_uint32(0)
    _lib.check(L.csa2_get_device_error(ctypes.byref(word)))
    return word.value


def test_noalloc_at_its_exact_limit():
    # B * NB * P = 2^20 exactly: the last query writes and reads the array's last slots
    # (every query sees more entries than the pool holds, so all 16,384 slots are used)
    L = _lib.lib()
    NB, P, k, B, n = 2048, 8, 512, 64, 20000
    assert B * NB * P == (1 << 20)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cache, q, w, seq_of, _ = _problem(4, B, n, NB, P, k)
    n_vis = torch.full((B,), n, dtype=torch.int32, device="cuda")
    ref = _outs(B, NB, P, k)
    _workspace_call(L, _args(cache, q, w, seq_of, n_vis, n, NB, P, k, ref), stream)
    got = _outs(B, NB, P, k)
    _lib.check(L.csa2_index_full_noalloc(ctypes.byref(_args(cache, q, w, seq_of, n_vis, n, NB, P, k, got)), stream))
    torch.cuda.synchronize()
    assert _device_error_word(L) == 0
    for x, y in zip(got, ref):
        assert torch.equal(x, y)
    assert (got[1] == NB * P).all() and (got[3] == k).all()


@pytest.mark.parametrize("H_i,group", [(16, 1), (8, 2)])
def test_noalloc_where_the_workspace_call_scores_on_tensor_cores(H_i, group):
    # csa2_index_full scores these on the tensor cores (group x H_i >= 16), the
    # allocation-free call scans: both must meet the near-tie rule against the oracle
    L = _lib.lib()
    NB, P, k, B, n_max = 2048, 8, 512, 4, 30000
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cache, q, w, seq_of, n_vis, h = _problem(5 + H_i, B, n_max, NB, P, k, H_i=H_i, group=group, host=True)
    ref = _outs(B, NB, P, k)
    _workspace_call(L, _args(cache, q, w, seq_of, n_vis, n_max, NB, P, k, ref, group), stream)
    got = _outs(B, NB, P, k)
    _lib.check(L.csa2_index_full_noalloc(ctypes.byref(_args(cache, q, w, seq_of, n_vis, n_max, NB, P, k, got, group)),
                                         stream))
    torch.cuda.synchronize()
    assert _device_error_word(L) == 0
    for b in range(B):
        n = int(h["n_vis"][b])
        Kb = formats.bf16_value(h["K"][h["seq"][b]][:n])
        pool, topk, sc = indexer.full(formats.bf16_value(h["q"][b]), h["w"][b].astype(np.float64), Kb, NB, P, k)
        for name, outs in (("no-alloc", got), ("workspace", ref)):
            pl, tl = int(outs[1][b]), int(outs[3][b])
            assert pl == len(pool) and tl == len(topk), name
            check_index_set(outs[0][b, :pl].cpu().numpy(), pool, lambda e: sc[e], f"{name} pool b={b}")
            check_index_set(outs[2][b, :tl].cpu().numpy(), topk, lambda e: sc[e], f"{name} topk b={b}")
