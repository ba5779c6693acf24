"""Host-side validation of every entry point, one rule at a time, on CPU: a valid argument
struct (device pointers faked, never dereferenced) passes the workspace query; changing one
field returns the stated status and names the problem.  Validation runs before any CUDA
call, so no GPU is needed."""
import ctypes

import pytest

from fp4_compressed_sparse_02_gb300 import _lib, build

P = 0x10000           # a 16-byte aligned fake device address
U = 0x10008           # an unaligned one
OK, INVALID, SHAPE = 0, 1, 2


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.lib()


def _cache(**kw):
    c = _lib.Cache(P, P, P, P, 1024, 64, 4, 256, 512, 128)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _compress(**kw):
    a = _lib.CompressArgs()
    a.struct_size = ctypes.sizeof(a)
    a.T, a.m, a.d_model, a.h_dtype = 8, 1, 0, 0
    a.C, a.seq, a.entry, a.pos = P, P, P, P
    a.cache = _cache()
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _full(**kw):
    a = _lib.IndexFullArgs()
    a.struct_size = ctypes.sizeof(a)
    a.B, a.H_i, a.k, a.relu = 4, 8, 512, 1
    a.q_idx = a.w = a.seq_of = a.n_vis = a.pool = a.pool_len = a.topk = a.topk_len = P
    a.cache = _cache()
    a.max_n, a.num_blocks, a.per_block = 4096, 2048, 8
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _reindex(**kw):
    a = _lib.IndexReindexArgs()
    a.struct_size = ctypes.sizeof(a)
    a.B, a.H_i, a.k, a.relu, a.pool_stride = 4, 8, 512, 1, 16384
    a.q_idx = a.w = a.seq_of = a.pool = a.pool_len = a.topk = a.topk_len = P
    a.cache = _cache()
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _attn(**kw):
    a = _lib.AttnArgs()
    a.struct_size = ctypes.sizeof(a)
    a.B, a.Hq, a.k, a.swa_max, a.swa_rows = 4, 64, 512, 128, 512
    a.q = a.seq_of = a.topk = a.topk_len = a.swa = a.swa_scale = a.swa_start = a.swa_len = a.out = P
    a.softmax_scale, a.out_dtype = 0.044, 0
    a.cache = _cache()
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _ws(L, fn, a):
    n = ctypes.c_size_t(0)
    return getattr(L, fn + "_workspace")(ctypes.byref(a), ctypes.byref(n)), L.csa2_last_error_message()


BASES = {"csa2_compress_quant": _compress, "csa2_index_full": _full, "csa2_index_reindex": _reindex,
         "csa2_sparse_attn": _attn}


@pytest.mark.parametrize("fn", sorted(BASES))
def test_valid_struct_passes(L, fn):
    assert _ws(L, fn, BASES[fn]())[0] == OK


CASES = [
    # compressor
    ("csa2_compress_quant", dict(T=-1), INVALID, b"T < 0"),
    ("csa2_compress_quant", dict(m=0), SHAPE, b"m must be"),
    ("csa2_compress_quant", dict(m=9), SHAPE, b"m must be"),
    ("csa2_compress_quant", dict(T=9, m=2, Z=P), INVALID, b"multiple of m"),
    ("csa2_compress_quant", dict(C=None), INVALID, b"C is NULL"),
    ("csa2_compress_quant", dict(T=8, m=2), INVALID, b"Z is NULL"),
    ("csa2_compress_quant", dict(W_kv=P, H=None, d_model=256), INVALID, b"H is NULL"),
    ("csa2_compress_quant", dict(W_kv=P, H=P, d_model=256, h_dtype=7), INVALID, b"h_dtype"),
    ("csa2_compress_quant", dict(W_kv=P, H=P, d_model=100), SHAPE, b"d_model"),
    ("csa2_compress_quant", dict(W_kv=P, H=P, d_model=256, m=2, T=8), INVALID, b"W_z"),
    ("csa2_compress_quant", dict(d_rope=16), SHAPE, b"d_rope"),
    ("csa2_compress_quant", dict(d_rope=64, rope_cos=None, rope_sin=P, rope_max_pos=10), INVALID, b"RoPE"),
    ("csa2_compress_quant", dict(d_rope=64, rope_cos=P, rope_sin=P, rope_max_pos=0), INVALID, b"rope_max_pos"),
    ("csa2_compress_quant", dict(seq=None), INVALID, b"seq/entry"),
    ("csa2_compress_quant", dict(W_ik=P, cache=_cache(idx_k=None)), INVALID, b"idx_k"),
    ("csa2_compress_quant", dict(cache=_cache(page_size=32)), SHAPE, b"page_size"),
    ("csa2_compress_quant", dict(cache=_cache(d=256)), SHAPE, b"cache.d"),
    ("csa2_compress_quant", dict(cache=_cache(codes=U)), INVALID, b"aligned"),
    ("csa2_compress_quant", dict(cache=_cache(page_table=None)), INVALID, b"page_table"),
    ("csa2_compress_quant", dict(cache=_cache(num_seqs=0)), INVALID, b"positive"),
    ("csa2_compress_quant", dict(cache=_cache(num_pages=(1 << 25) + 1)), SHAPE, b"2^25"),
    # Full indexer
    ("csa2_index_full", dict(B=-1), INVALID, b"B < 0"),
    ("csa2_index_full", dict(H_i=0), SHAPE, b"H_i"),
    ("csa2_index_full", dict(H_i=33), SHAPE, b"H_i"),
    ("csa2_index_full", dict(k=0), SHAPE, b"k must be"),
    ("csa2_index_full", dict(k=2049), SHAPE, b"k must be"),
    ("csa2_index_full", dict(per_block=33), SHAPE, b"per_block"),
    ("csa2_index_full", dict(num_blocks=0), SHAPE, b"num_blocks"),
    ("csa2_index_full", dict(num_blocks=4096, per_block=8), SHAPE, b"16384"),
    ("csa2_index_full", dict(max_n=256 * 64 + 1), INVALID, b"max_n"),
    ("csa2_index_full", dict(max_n=-1), INVALID, b"max_n"),
    ("csa2_index_full", dict(pool=None), INVALID, b"NULL"),
    ("csa2_index_full", dict(topk=None), INVALID, b"NULL"),
    ("csa2_index_full", dict(group=3), INVALID, b"multiple of group"),
    ("csa2_index_full", dict(group=-2), INVALID, b"group"),
    ("csa2_index_full", dict(cache=_cache(idx_k=U)), INVALID, b"aligned"),
    ("csa2_index_full", dict(cache=_cache(d_ik=96)), SHAPE, b"d_ik"),
    # Reindex
    ("csa2_index_reindex", dict(pool_stride=0), SHAPE, b"pool_stride"),
    ("csa2_index_reindex", dict(pool_stride=16385), SHAPE, b"pool_stride"),
    ("csa2_index_reindex", dict(pool_len=None), INVALID, b"pool"),
    ("csa2_index_reindex", dict(w=None), INVALID, b"NULL"),
    ("csa2_index_reindex", dict(H_i=64), SHAPE, b"H_i"),
    # attention
    ("csa2_sparse_attn", dict(B=-1), INVALID, b"B < 0"),
    ("csa2_sparse_attn", dict(Hq=12), SHAPE, b"Hq"),
    ("csa2_sparse_attn", dict(k=4000, swa_max=128), SHAPE, b"4096"),
    ("csa2_sparse_attn", dict(k=-1), SHAPE, b"k >= 0"),
    ("csa2_sparse_attn", dict(out_dtype=9), INVALID, b"out_dtype"),
    ("csa2_sparse_attn", dict(q=U), INVALID, b"aligned"),
    ("csa2_sparse_attn", dict(out=None), INVALID, b"NULL"),
    ("csa2_sparse_attn", dict(topk=None), INVALID, b"topk"),
    ("csa2_sparse_attn", dict(swa_rows=0), INVALID, b"SWA"),
    ("csa2_sparse_attn", dict(swa_start=None), INVALID, b"SWA"),
    ("csa2_sparse_attn", dict(cache=_cache(scales=None)), INVALID, b"codes/scales"),
]


@pytest.mark.parametrize("fn,change,status,msg", CASES,
                         ids=[f"{c[0][5:]}-{'-'.join(c[1])}" for c in CASES])
def test_one_bad_field(L, fn, change, status, msg):
    st, text = _ws(L, fn, BASES[fn](**change))
    assert st == status, text
    assert msg in text, text


def test_empty_batches_need_no_pointers(L):
    # B = 0 (or T = 0) is a valid no-op: the per-query pointers may be NULL
    assert _ws(L, "csa2_sparse_attn", _attn(B=0, q=None, seq_of=None, out=None, topk=None))[0] == OK
    assert _ws(L, "csa2_index_full", _full(B=0, q_idx=None, w=None, pool=None, topk=None))[0] == OK
    assert _ws(L, "csa2_index_reindex", _reindex(B=0, pool=None, pool_len=None))[0] == OK
    assert _ws(L, "csa2_compress_quant", _compress(T=0, seq=None, entry=None))[0] == OK
    # window-only attention needs no topk, selected-only no window
    assert _ws(L, "csa2_sparse_attn", _attn(k=0, topk=None))[0] == OK
    assert _ws(L, "csa2_sparse_attn", _attn(swa_max=0, swa=None, swa_scale=None, swa_start=None,
                                            swa_len=None))[0] == OK


def _swaq(**kw):
    a = _lib.SwaQuantArgs()
    a.struct_size = ctypes.sizeof(a)
    a.R, a.d, a.x_dtype, a.x, a.row_idx, a.swa, a.swa_scale, a.swa_rows = 4, 512, 0, P, 0, P, P, 16
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("change,status,msg", [
    (dict(struct_size=8), INVALID, "struct_size"),
    (dict(R=-1), INVALID, "R < 0"),
    (dict(d=256), SHAPE, "d must be"),
    (dict(x_dtype=7), INVALID, "x_dtype"),
    (dict(x=0), INVALID, "NULL"),
    (dict(swa_scale=0), INVALID, "NULL"),
    (dict(swa_rows=0), INVALID, "swa_rows"),
    (dict(R=17), INVALID, "R > swa_rows"),
    (dict(x=U), INVALID, "x must be 16-byte aligned"),
    (dict(swa=U), INVALID, "swa must be"),
])
def test_swa_quant_one_bad_field(L, change, status, msg):
    a = _swaq(**change)
    assert L.csa2_swa_quant(ctypes.byref(a), None) == status
    assert msg in L.csa2_last_error_message().decode()


def test_swa_quant_empty_needs_no_pointers(L):
    a = _swaq(R=0, x=0, swa=0, swa_scale=0, swa_rows=0)
    assert L.csa2_swa_quant(ctypes.byref(a), None) == OK


def _append(**kw):
    a = _lib.AppendArgs()
    a.struct_size = ctypes.sizeof(a)
    a.B, a.m, a.d_model, a.h_dtype = 4, 2, 512, 0
    a.H, a.W_kv, a.W_z, a.seq, a.tok_pos, a.pend = P, P, P, P, P, P
    a.cache = _cache()
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_append_valid_struct_passes(L):
    n = ctypes.c_size_t(0)
    assert L.csa2_compress_append_workspace(ctypes.byref(_append()), ctypes.byref(n)) == OK


@pytest.mark.parametrize("change,status,msg", [
    (dict(struct_size=8), INVALID, "struct_size"),
    (dict(B=-1), INVALID, "B < 0"),
    (dict(m=9), SHAPE, "m must be"),
    (dict(d_model=100), SHAPE, "d_model"),
    (dict(h_dtype=5), INVALID, "h_dtype"),
    (dict(H=0), INVALID, "NULL"),
    (dict(tok_pos=0), INVALID, "NULL"),
    (dict(pend=0), INVALID, "pend"),
    (dict(W_z=0), INVALID, "W_z"),
    (dict(d_rope=16), SHAPE, "d_rope"),
    (dict(d_rope=32, rope_cos=0), INVALID, "RoPE"),
    (dict(H=U), INVALID, "16-byte aligned"),
])
def test_append_one_bad_field(L, change, status, msg):
    n = ctypes.c_size_t(0)
    assert L.csa2_compress_append_workspace(ctypes.byref(_append(**change)), ctypes.byref(n)) == status
    assert msg in L.csa2_last_error_message().decode()


def test_append_at_m1_needs_no_pending_buffer(L):
    n = ctypes.c_size_t(0)
    assert L.csa2_compress_append_workspace(ctypes.byref(_append(m=1, pend=0, W_z=0)), ctypes.byref(n)) == OK


def test_fp8_form_needs_its_planes(L):
    n = ctypes.c_size_t(0)
    a = _full(cache=_cache(idx_k_dtype=2))                 # FP8 form without idx_k8
    assert L.csa2_index_full_workspace(ctypes.byref(a), ctypes.byref(n)) == INVALID
    assert "idx_k8" in L.csa2_last_error_message().decode()
    a = _full(cache=_cache(idx_k_dtype=2, idx_k8=P, idx_k8_scale=P))
    assert L.csa2_index_full_workspace(ctypes.byref(a), ctypes.byref(n)) == OK
    a = _full(cache=_cache(idx_k_dtype=9))
    assert L.csa2_index_full_workspace(ctypes.byref(a), ctypes.byref(n)) == INVALID


def test_noalloc_rejects_the_fp8_form_before_any_cuda_call(L):
    a = _full(cache=_cache(idx_k_dtype=2, idx_k8=P, idx_k8_scale=P))
    assert L.csa2_index_full_noalloc(ctypes.byref(a), None) == SHAPE
    assert "FP8" in L.csa2_last_error_message().decode()
