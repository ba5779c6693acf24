"""CPU-side checks of the C ABI: the library builds, loads, exports every function that
include/csa2.h declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from fp4_compressed_sparse_02_gb300 import _lib, build

HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z_]+)\s*\(", text)))


def test_header_declares_the_four_calls_and_helpers():
    fns = declared_functions()
    for name in ["csa2_compress_quant", "csa2_index_full", "csa2_index_reindex", "csa2_sparse_attn",
                 "csa2_get_device_error", "csa2_last_error_message", "csa2_version"]:
        assert name in fns


def test_library_exports_every_declared_function(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version(L):
    assert L.csa2_version() >= 100


def _cache(**kw):
    c = _lib.Cache(None, None, None, None, 1, 64, 1, 1, 512, 128)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails before any launch


def test_null_args_rejected(L):
    for fn in ["csa2_compress_quant", "csa2_index_full", "csa2_index_reindex", "csa2_sparse_attn"]:
        st = getattr(L, fn)(None, None, 0, None)
        assert st == 1
        assert b"NULL" in L.csa2_last_error_message()


def test_attn_shape_checks_on_host(L):
    a = _lib.AttnArgs()
    a.struct_size = ctypes.sizeof(a)
    a.B, a.Hq, a.k, a.swa_max = 1, 12, 512, 128
    a.cache = _cache(codes=FAKE, scales=FAKE, page_table=FAKE)
    st = L.csa2_sparse_attn(ctypes.byref(a), None, 0, None)
    assert st == 2 and b"Hq" in L.csa2_last_error_message()
    a.Hq = 64
    a.cache = _cache(codes=FAKE, scales=FAKE, page_table=FAKE, d=256)
    assert L.csa2_sparse_attn(ctypes.byref(a), None, 0, None) == 2
    a.cache = _cache(codes=FAKE, scales=FAKE, page_table=FAKE, page_size=32)
    assert L.csa2_sparse_attn(ctypes.byref(a), None, 0, None) == 2


def test_workspace_too_small_is_reported(L):
    a = _lib.IndexFullArgs()
    a.struct_size = ctypes.sizeof(a)
    a.B, a.H_i, a.k = 2, 8, 512
    a.cache = _cache(idx_k=FAKE, page_table=FAKE, max_pages=4)
    a.q_idx = a.w = a.seq_of = a.n_vis = a.pool = a.pool_len = a.topk = a.topk_len = FAKE
    a.max_n, a.num_blocks, a.per_block = 256, 2048, 8
    need = ctypes.c_size_t(0)
    assert L.csa2_index_full_workspace(ctypes.byref(a), ctypes.byref(need)) == 0
    assert need.value == 2 * 2048 * 8 * 4
    assert L.csa2_index_full(ctypes.byref(a), FAKE, need.value - 1, None) == 3
    a.per_block = 9                      # 2048 * 9 > 16384
    assert L.csa2_index_full(ctypes.byref(a), FAKE, 1 << 30, None) == 2
    a.per_block = 8
    a.max_n = 4 * 64 + 1                 # beyond the page table
    assert L.csa2_index_full(ctypes.byref(a), FAKE, 1 << 30, None) == 1


def test_full_group_checks_on_host(L):
    a = _lib.IndexFullArgs()
    a.struct_size = ctypes.sizeof(a)
    a.B, a.H_i, a.k = 6, 8, 512
    a.cache = _cache(idx_k=FAKE, page_table=FAKE, max_pages=4)
    a.q_idx = a.w = a.seq_of = a.n_vis = a.pool = a.pool_len = a.topk = a.topk_len = FAKE
    a.max_n, a.num_blocks, a.per_block = 256, 2048, 8
    a.group = 4                          # B = 6 is not a multiple of 4
    assert L.csa2_index_full(ctypes.byref(a), FAKE, 1 << 30, None) == 1
    assert b"multiple of group" in L.csa2_last_error_message()
    a.group = -1
    assert L.csa2_index_full(ctypes.byref(a), FAKE, 1 << 30, None) == 1
    a.group, a.H_i = 3, 16               # any head count: tensor-core scoring or a scan per query
    nbytes = ctypes.c_size_t(0)
    assert L.csa2_index_full_workspace(ctypes.byref(a), ctypes.byref(nbytes)) == 0
    assert nbytes.value >= 6 * 2048 * 8 * 4


def test_compress_rejects_partial_group_and_bad_m(L):
    a = _lib.CompressArgs()
    a.struct_size = ctypes.sizeof(a)
    a.T, a.m = 5, 2
    a.C = a.Z = a.seq = a.entry = FAKE
    a.cache = _cache(codes=FAKE, scales=FAKE, page_table=FAKE)
    assert L.csa2_compress_quant(ctypes.byref(a), None, 0, None) == 1
    assert b"multiple of m" in L.csa2_last_error_message()
    a.T, a.m = 9, 9
    assert L.csa2_compress_quant(ctypes.byref(a), None, 0, None) == 2


def test_struct_size_mismatch_rejected(L):
    a = _lib.AttnArgs()
    a.struct_size = ctypes.sizeof(a) - 8
    assert L.csa2_sparse_attn(ctypes.byref(a), None, 0, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.lib()
