"""Python face of the CSA2 C ABI: torch tensors in, device pointers to libcsa2.so.

Names follow include/csa2.h: compress_quant, index_full, index_reindex, sparse_attn.
PyTorch provides device memory and the current stream; every computation runs in the
library's kernels.  Outputs are allocated here when the caller passes none (pass them
in, together with a pre-sized Workspace, to capture calls in a CUDA graph).
"""
import ctypes
import math
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib

PAGE = 64
BF16, F32, FP8E4M3 = 0, 1, 2


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _expect(t, dtypes, name):
    if t is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")


_I32 = (torch.int32,)
_B16 = (torch.bfloat16, torch.int16)
_U8 = (torch.uint8,)
_F32 = (torch.float32,)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@dataclass
class PagedCache:
    """Paged Main KV planes: codes uint8 [pages, 64, d/2], scales uint8 [pages, 64, d/16],
    page_table int32 [seqs, max_pages], and indexer K in one of two forms: idx_k bf16
    [pages, 64, d_ik], or (compressed) idx_k8 uint8 E4M3 [pages, 64, d_ik] with
    idx_k8_scale float32 [pages, 64].  The FP8 form is used when idx_k8 is set."""
    codes: torch.Tensor
    scales: torch.Tensor
    idx_k: Optional[torch.Tensor]
    page_table: torch.Tensor
    idx_k8: Optional[torch.Tensor] = None
    idx_k8_scale: Optional[torch.Tensor] = None

    @property
    def d(self):
        return self.codes.shape[-1] * 2

    @property
    def d_ik(self):
        if self.idx_k8 is not None:
            return self.idx_k8.shape[-1]
        return self.idx_k.shape[-1] if self.idx_k is not None else 0

    @property
    def num_pages(self):
        return self.codes.shape[0]

    @property
    def num_seqs(self):
        return self.page_table.shape[0]

    @property
    def max_pages(self):
        return self.page_table.shape[1]

    @staticmethod
    def allocate(num_seqs, entries_per_seq, d, d_ik, device, page_table=None, idx_k_fp8=False):
        mp = (entries_per_seq + PAGE - 1) // PAGE
        npg = num_seqs * mp
        if page_table is None:
            page_table = torch.arange(npg, dtype=torch.int32).reshape(num_seqs, mp)
        page_table = page_table.to(device=device, dtype=torch.int32).contiguous()
        npg = max(npg, int(page_table.max().item()) + 1) if page_table.numel() else npg
        codes = torch.zeros((npg, PAGE, d // 2), dtype=torch.uint8, device=device)
        scales = torch.zeros((npg, PAGE, d // 16), dtype=torch.uint8, device=device)
        idx_k = idx_k8 = idx_k8_scale = None
        if d_ik and idx_k_fp8:
            idx_k8 = torch.zeros((npg, PAGE, d_ik), dtype=torch.uint8, device=device)
            idx_k8_scale = torch.zeros((npg, PAGE), dtype=torch.float32, device=device)
        elif d_ik:
            idx_k = torch.zeros((npg, PAGE, d_ik), dtype=torch.bfloat16, device=device)
        return PagedCache(codes, scales, idx_k, page_table, idx_k8, idx_k8_scale)

    def c_struct(self):
        for t, n in [(self.codes, "codes"), (self.scales, "scales"), (self.idx_k8, "idx_k8")]:
            _expect(t, _U8, n)
        _expect(self.idx_k, _B16, "idx_k")
        _expect(self.idx_k8_scale, _F32, "idx_k8_scale")
        _expect(self.page_table, _I32, "page_table")
        fp8 = self.idx_k8 is not None
        return _lib.Cache(_ptr(self.codes), _ptr(self.scales), _ptr(self.idx_k), _ptr(self.page_table),
                          self.num_pages, PAGE, self.num_seqs, self.max_pages, self.d, self.d_ik,
                          FP8E4M3 if fp8 else BF16, _ptr(self.idx_k8), _ptr(self.idx_k8_scale))


class Workspace:
    """Grow-only device scratch buffer handed to the library calls."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = torch.empty(0, dtype=torch.uint8, device=device)

    def get(self, nbytes):
        if self.buf.numel() < nbytes:
            if torch.cuda.is_current_stream_capturing():
                raise RuntimeError("workspace must be sized before CUDA graph capture")
            self.buf = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _ws(ws, device):
    if ws is not None:
        return ws
    key = str(device)
    if key not in _default_ws:
        _default_ws[key] = Workspace(device)
    return _default_ws[key]


def _call(fn, args, ws, device):
    L = _lib.lib()
    need = ctypes.c_size_t(0)
    _lib.check(getattr(L, fn + "_workspace")(ctypes.byref(args), ctypes.byref(need)))
    buf = _ws(ws, device).get(need.value)
    _lib.check(getattr(L, fn)(ctypes.byref(args), ctypes.c_void_p(buf.data_ptr()), need.value, _stream()))


def compress_quant(cache: PagedCache, seq, entry, *, m=1, C=None, Z=None, H=None, W_kv=None, W_z=None,
                   pos=None, rope_cos=None, rope_sin=None, W_ik=None, y_out=None, ws=None):
    """Compress m-token groups into FP4 Main KV entries written through the page table.
    Given mode: C (and Z when m > 1) float32 [T, d].  Projection mode: H [T, d_model]
    (bf16 or float32) with W_kv, W_z bf16 [d_model, d].  seq/entry/pos: int32 [T/m]."""
    if W_kv is not None:
        T, d_model = H.shape
        _expect(H, _B16 + _F32, "H")
        h_dtype = F32 if H.dtype == torch.float32 else BF16
    else:
        T, d_model, h_dtype = C.shape[0], 0, BF16
        _expect(C, _F32, "C")
        _expect(Z, _F32, "Z")
    for t, n in [(seq, "seq"), (entry, "entry"), (pos, "pos")]:
        _expect(t, _I32, n)
    d_rope = 0 if rope_cos is None else rope_cos.shape[1] * 2
    a = _lib.CompressArgs()
    a.struct_size = ctypes.sizeof(_lib.CompressArgs)
    a.T, a.m, a.d_model, a.h_dtype = T, m, d_model, h_dtype
    a.H, a.W_kv, a.W_z, a.C, a.Z = _ptr(H), _ptr(W_kv), _ptr(W_z), _ptr(C), _ptr(Z)
    a.d_rope = d_rope
    a.rope_max_pos = rope_cos.shape[0] if rope_cos is not None else 0
    a.rope_cos, a.rope_sin, a.pos = _ptr(rope_cos), _ptr(rope_sin), _ptr(pos)
    a.seq, a.entry, a.W_ik = _ptr(seq), _ptr(entry), _ptr(W_ik)
    a.cache = cache.c_struct()
    a.y_out = _ptr(y_out)
    _call("csa2_compress_quant", a, ws, cache.codes.device)


def compress_append(cache: PagedCache, H, seq, tok_pos, W_kv, *, m=1, W_z=None, pend=None, rope_cos=None,
                    rope_sin=None, W_ik=None, y_out=None, ws=None):
    """The decode-time append: H [B, d_model] (bf16 or float32) holds one new token of each
    of B distinct sequences seq[b] at position tok_pos[b].  At m > 1 a token that does not
    complete its group waits in pend (float32 [num_seqs, 2, m, d], kept by the caller
    between calls); the completing token writes entry tok_pos // m."""
    B, d_model = H.shape
    _expect(H, _B16 + _F32, "H")
    _expect(pend, _F32, "pend")
    for t, n in [(seq, "seq"), (tok_pos, "tok_pos")]:
        _expect(t, _I32, n)
    a = _lib.AppendArgs()
    a.struct_size = ctypes.sizeof(_lib.AppendArgs)
    a.B, a.m, a.d_model = B, m, d_model
    a.h_dtype = F32 if H.dtype == torch.float32 else BF16
    a.H, a.W_kv, a.W_z = _ptr(H), _ptr(W_kv), _ptr(W_z)
    a.d_rope = 0 if rope_cos is None else rope_cos.shape[1] * 2
    a.rope_max_pos = rope_cos.shape[0] if rope_cos is not None else 0
    a.rope_cos, a.rope_sin = _ptr(rope_cos), _ptr(rope_sin)
    a.seq, a.tok_pos, a.pend, a.W_ik = _ptr(seq), _ptr(tok_pos), _ptr(pend), _ptr(W_ik)
    a.cache = cache.c_struct()
    a.y_out = _ptr(y_out)
    _call("csa2_compress_append", a, ws, cache.codes.device)


def index_full(cache: PagedCache, q_idx, w, seq_of, n_vis, max_n, num_blocks=2048, per_block=8, k=512,
               relu=True, out=None, ws=None, group=1):
    """Full-mode indexer.  q_idx bf16 [B, H_i, d_ik], w float32 [B, H_i], seq_of / n_vis
    int32 [B].  group > 1: queries g*group .. g*group+group-1 share one sequence, whose
    indexer-K rows are read once for all of them (tensor-core scoring when group x H_i >= 16
    and the shape allows it; see include/csa2.h).  Returns (pool [B, NB*P], pool_len [B],
    topk [B, k], topk_len [B])."""
    B, H_i, _ = q_idx.shape
    dev = q_idx.device
    if out is None:
        out = (torch.empty((B, num_blocks * per_block), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty((B, k), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev))
    pool, pool_len, topk, topk_len = out
    _expect(q_idx, _B16, "q_idx")
    _expect(w, _F32, "w")
    a = _lib.IndexFullArgs()
    a.struct_size = ctypes.sizeof(_lib.IndexFullArgs)
    a.B, a.H_i = B, H_i
    a.q_idx, a.w = _ptr(q_idx), _ptr(w)
    a.cache = cache.c_struct()
    a.seq_of, a.n_vis, a.max_n = _ptr(seq_of), _ptr(n_vis), int(max_n)
    a.num_blocks, a.per_block, a.k, a.relu = num_blocks, per_block, k, int(bool(relu))
    a.pool, a.pool_len, a.topk, a.topk_len = _ptr(pool), _ptr(pool_len), _ptr(topk), _ptr(topk_len)
    a.group = int(group)
    _call("csa2_index_full", a, ws, dev)
    return out


def index_reindex(cache: PagedCache, q_idx, w, seq_of, pool, pool_len, k=512, relu=True, out=None, ws=None):
    """Reindex mode: re-score only the pool.  Returns (topk [B, k], topk_len [B])."""
    B, H_i, _ = q_idx.shape
    dev = q_idx.device
    if out is None:
        out = (torch.empty((B, k), dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
    topk, topk_len = out
    a = _lib.IndexReindexArgs()
    a.struct_size = ctypes.sizeof(_lib.IndexReindexArgs)
    a.B, a.H_i = B, H_i
    a.q_idx, a.w = _ptr(q_idx), _ptr(w)
    a.cache = cache.c_struct()
    a.seq_of, a.pool, a.pool_len, a.pool_stride = _ptr(seq_of), _ptr(pool), _ptr(pool_len), pool.shape[1]
    a.k, a.relu = k, int(bool(relu))
    a.topk, a.topk_len = _ptr(topk), _ptr(topk_len)
    _call("csa2_index_reindex", a, ws, dev)
    return out


def sparse_attn(cache: PagedCache, q, seq_of, topk, topk_len, swa, swa_scale, swa_start, swa_len, swa_max,
                softmax_scale=None, out_dtype=torch.bfloat16, out=None, lse=None, ws=None, inputs_ready=False):
    """One softmax over the selected FP4 entries plus the SWA window.  q bf16 [B, Hq, d].
    inputs_ready: the kernel launched just before on the stream writes none of this call's
    inputs (a Reuse layer after the previous layer's attention), so the call may read them
    before that kernel completes.  Returns (out [B, Hq, d], lse float32 [B, Hq])."""
    B, Hq, d = q.shape
    dev = q.device
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=out_dtype, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _expect(q, _B16, "q")
    a = _lib.AttnArgs()
    a.struct_size = ctypes.sizeof(_lib.AttnArgs)
    a.B, a.Hq, a.q = B, Hq, _ptr(q)
    a.cache = cache.c_struct()
    a.seq_of, a.topk, a.topk_len, a.k = _ptr(seq_of), _ptr(topk), _ptr(topk_len), topk.shape[1]
    a.swa, a.swa_scale = _ptr(swa), _ptr(swa_scale)
    a.swa_rows = swa.shape[0] if swa is not None else 0
    a.swa_start, a.swa_len, a.swa_max = _ptr(swa_start), _ptr(swa_len), int(swa_max)
    a.softmax_scale = float(softmax_scale)
    a.out = _ptr(out)
    a.out_dtype = F32 if out.dtype == torch.float32 else BF16
    a.lse = _ptr(lse)
    a.inputs_ready = int(bool(inputs_ready))
    _call("csa2_sparse_attn", a, ws, dev)
    return out, lse


def swa_quant(x, swa, swa_scale, row_idx=None):
    """FP8 window rows (a bounded replay's rebuilt SWA window): each row of x (bf16 or
    float32 [R, d]) becomes E4M3 bytes with one float32 scale amax/448, written to
    swa[row_idx[r]] / swa_scale[row_idx[r]] (row r when row_idx is None)."""
    R, d = x.shape
    _expect(x, _B16 + _F32, "x")
    _expect(swa, _U8, "swa")
    _expect(swa_scale, _F32, "swa_scale")
    _expect(row_idx, _I32, "row_idx")
    a = _lib.SwaQuantArgs()
    a.struct_size = ctypes.sizeof(_lib.SwaQuantArgs)
    a.R, a.d = R, d
    a.x_dtype = F32 if x.dtype == torch.float32 else BF16
    a.x, a.row_idx, a.swa, a.swa_scale = _ptr(x), _ptr(row_idx), _ptr(swa), _ptr(swa_scale)
    a.swa_rows = swa.shape[0]
    _lib.check(_lib.lib().csa2_swa_quant(ctypes.byref(a), _stream()))


def device_error():
    """Synchronise and return (and clear) the device error word (a non-zero word is
    returned, not raised: the library reports it as CSA2_ERR_DEVICE_CHECK / _TIMEOUT)."""
    w = ctypes.c_uint32(0)
    st = _lib.lib().csa2_get_device_error(ctypes.byref(w))
    if st not in (0, 5, 6):
        _lib.check(st)
    return w.value


def version():
    return _lib.lib().csa2_version()


def selftest_wait_timeout(polls=1000):
    """Run the bounded-wait failure path once (one CTA waits on an mbarrier nothing
    arrives on, gives up after `polls` polls and sets the timeout bit of the device error
    word)."""
    _lib.check(_lib.lib().csa2_selftest_wait_timeout(int(polls), _stream()))
