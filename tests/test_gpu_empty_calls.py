"""Zero-size calls through the C ABI on the GPU: B = 0 queries (or T = 0 tokens, R = 0 window
rows) is a valid no-op for every compute entry point.  The per-query pointers may be NULL (the
compressor still needs its mode's input pointer), nothing is launched, the status is CSA2_OK
and the device error word stays clear."""
import ctypes

import numpy as np
import pytest
import torch

from fp4_compressed_sparse_02_gb300 import _lib, csa2, synth

pytestmark = pytest.mark.gpu


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.fixture(scope="module")
def cache():
    r = np.random.default_rng(0)
    pt = synth.page_table(r, 1, 4)
    return csa2.PagedCache.allocate(1, 256, 512, 128, "cuda", torch.from_numpy(pt))


def _call(L, fn, a):
    need = ctypes.c_size_t(123)
    assert getattr(L, fn + "_workspace")(ctypes.byref(a), ctypes.byref(need)) == 0, L.csa2_last_error_message()
    ws = torch.empty(max(1, need.value), dtype=torch.uint8, device="cuda")
    st = getattr(L, fn)(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), need.value, _stream())
    assert st == 0, (fn, L.csa2_last_error_message())


def test_zero_size_calls_are_no_ops(cache):
    L = _lib.lib()
    csa2.device_error()                                   # (clears the word)
    a = _lib.IndexFullArgs()
    a.struct_size = ctypes.sizeof(a)
    a.B, a.H_i, a.k, a.relu, a.max_n, a.num_blocks, a.per_block = 0, 8, 512, 1, 256, 2048, 8
    a.cache = cache.c_struct()
    _call(L, "csa2_index_full", a)
    assert L.csa2_index_full_noalloc(ctypes.byref(a), _stream()) == 0
    r = _lib.IndexReindexArgs()
    r.struct_size = ctypes.sizeof(r)
    r.B, r.H_i, r.k, r.relu, r.pool_stride = 0, 8, 512, 1, 16384
    r.cache = cache.c_struct()
    _call(L, "csa2_index_reindex", r)
    t = _lib.AttnArgs()
    t.struct_size = ctypes.sizeof(t)
    t.B, t.Hq, t.k, t.swa_max, t.swa_rows = 0, 64, 512, 0, 0
    t.softmax_scale, t.out_dtype = 0.044, 0
    t.cache = cache.c_struct()
    _call(L, "csa2_sparse_attn", t)
    c = _lib.CompressArgs()
    c.struct_size = ctypes.sizeof(c)
    c.T, c.m = 0, 1
    C = torch.zeros((1, 512), dtype=torch.float32, device="cuda")   # the given mode's input (no rows)
    c.C = C.data_ptr()
    c.cache = cache.c_struct()
    _call(L, "csa2_compress_quant", c)
    s = _lib.SwaQuantArgs()
    s.struct_size = ctypes.sizeof(s)
    s.R, s.d, s.x_dtype, s.swa_rows = 0, 512, 0, 0
    assert L.csa2_swa_quant(ctypes.byref(s), _stream()) == 0, L.csa2_last_error_message()
    torch.cuda.synchronize()
    assert csa2.device_error() == 0
