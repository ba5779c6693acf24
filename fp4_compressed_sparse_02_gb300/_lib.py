"""ctypes binding of libcsa2.so (include/csa2.h).  Argument marshalling only: every
step of the hot path runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or fails to load, every call raises."""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcsa2.so")

c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p


class Cache(ctypes.Structure):
    _fields_ = [("codes", c_vp), ("scales", c_vp), ("idx_k", c_vp), ("page_table", c_vp),
                ("num_pages", c_i32), ("page_size", c_i32), ("num_seqs", c_i32),
                ("max_pages", c_i32), ("d", c_i32), ("d_ik", c_i32), ("idx_k_dtype", c_i32), ("idx_k8", c_vp),
                ("idx_k8_scale", c_vp)]


class CompressArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_size_t), ("T", c_i32), ("m", c_i32), ("d_model", c_i32),
                ("h_dtype", c_i32), ("H", c_vp), ("W_kv", c_vp), ("W_z", c_vp), ("C", c_vp),
                ("Z", c_vp), ("d_rope", c_i32), ("rope_max_pos", c_i32), ("rope_cos", c_vp),
                ("rope_sin", c_vp), ("pos", c_vp), ("seq", c_vp), ("entry", c_vp), ("W_ik", c_vp),
                ("cache", Cache), ("y_out", c_vp)]


class IndexFullArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_size_t), ("B", c_i32), ("H_i", c_i32), ("q_idx", c_vp),
                ("w", c_vp), ("cache", Cache), ("seq_of", c_vp), ("n_vis", c_vp), ("max_n", c_i32),
                ("num_blocks", c_i32), ("per_block", c_i32), ("k", c_i32), ("relu", c_i32),
                ("pool", c_vp), ("pool_len", c_vp), ("topk", c_vp), ("topk_len", c_vp), ("group", c_i32)]


class IndexReindexArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_size_t), ("B", c_i32), ("H_i", c_i32), ("q_idx", c_vp),
                ("w", c_vp), ("cache", Cache), ("seq_of", c_vp), ("pool", c_vp), ("pool_len", c_vp),
                ("pool_stride", c_i32), ("k", c_i32), ("relu", c_i32), ("topk", c_vp),
                ("topk_len", c_vp)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_size_t), ("B", c_i32), ("Hq", c_i32), ("q", c_vp),
                ("cache", Cache), ("seq_of", c_vp), ("topk", c_vp), ("topk_len", c_vp), ("k", c_i32),
                ("swa", c_vp), ("swa_scale", c_vp), ("swa_rows", c_i32), ("swa_start", c_vp),
                ("swa_len", c_vp), ("swa_max", c_i32), ("softmax_scale", ctypes.c_float),
                ("out", c_vp), ("out_dtype", c_i32), ("lse", c_vp), ("inputs_ready", c_i32)]


class AppendArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_size_t), ("B", c_i32), ("m", c_i32), ("d_model", c_i32),
                ("h_dtype", c_i32), ("H", c_vp), ("W_kv", c_vp), ("W_z", c_vp), ("d_rope", c_i32),
                ("rope_max_pos", c_i32), ("rope_cos", c_vp), ("rope_sin", c_vp), ("seq", c_vp), ("tok_pos", c_vp),
                ("pend", c_vp), ("W_ik", c_vp), ("cache", Cache), ("y_out", c_vp)]


class SwaQuantArgs(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_size_t), ("R", c_i32), ("d", c_i32), ("x_dtype", c_i32), ("x", c_vp),
                ("row_idx", c_vp), ("swa", c_vp), ("swa_scale", c_vp), ("swa_rows", c_i32)]


STATUS = {0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED_SHAPE", 3: "ERR_WORKSPACE_TOO_SMALL",
          4: "ERR_CUDA", 5: "ERR_DEVICE_CHECK", 6: "ERR_TIMEOUT"}

EXPORTS = ["csa2_compress_quant", "csa2_compress_quant_workspace", "csa2_index_full",
           "csa2_index_full_workspace", "csa2_index_reindex", "csa2_index_reindex_workspace",
           "csa2_sparse_attn", "csa2_sparse_attn_workspace", "csa2_last_error_message",
           "csa2_get_device_error", "csa2_version", "csa2_index_full_noalloc", "csa2_selftest_wait_timeout",
           "csa2_swa_quant", "csa2_compress_append", "csa2_compress_append_workspace"]

_lib = None


class Csa2Error(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


def lib():
    """Load libcsa2.so once.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m fp4_compressed_sparse_02_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    pairs = [("csa2_compress_quant", CompressArgs), ("csa2_compress_append", AppendArgs),
             ("csa2_index_full", IndexFullArgs),
             ("csa2_index_reindex", IndexReindexArgs), ("csa2_sparse_attn", AttnArgs)]
    for name, st in pairs:
        f = getattr(L, name)
        f.argtypes = [ctypes.POINTER(st), c_vp, ctypes.c_size_t, c_vp]
        f.restype = c_i32
        g = getattr(L, name + "_workspace")
        g.argtypes = [ctypes.POINTER(st), ctypes.POINTER(ctypes.c_size_t)]
        g.restype = c_i32
    L.csa2_swa_quant.argtypes = [ctypes.POINTER(SwaQuantArgs), c_vp]
    L.csa2_swa_quant.restype = c_i32
    L.csa2_index_full_noalloc.argtypes = [ctypes.POINTER(IndexFullArgs), c_vp]
    L.csa2_index_full_noalloc.restype = c_i32
    L.csa2_last_error_message.argtypes = []
    L.csa2_last_error_message.restype = ctypes.c_char_p
    L.csa2_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.csa2_get_device_error.restype = c_i32
    L.csa2_selftest_wait_timeout.argtypes = [c_i32, c_vp]
    L.csa2_selftest_wait_timeout.restype = c_i32
    L.csa2_version.argtypes = []
    L.csa2_version.restype = c_i32
    _lib = L
    return L


def check(status):
    if status != 0:
        msg = lib().csa2_last_error_message().decode(errors="replace")
        raise Csa2Error(status, msg)
