// Host-side C ABI: argument validation, workspace sizing and dispatch.  No kernel
// launches happen before every host-visible argument has been checked.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "csa2.h"
#include <cstdint>
#include "internal.h"

namespace {

thread_local char g_msg[512] = "";

csa2_status fail(csa2_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

csa2_status ok() {
  g_msg[0] = 0;
  return CSA2_OK;
}

csa2_status cuda_status(cudaError_t e, const char* where) {
  if (e != cudaSuccess) return fail(CSA2_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
  return ok();
}

#define REQUIRE(cond, st, ...) \
  do {                         \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

csa2_status check_cache(const csa2_cache& c, bool need_codes, bool need_idx) {
  REQUIRE(c.page_table, CSA2_ERR_INVALID_ARG, "cache.page_table is NULL");
  REQUIRE(c.page_size == CSA2_PAGE_SIZE, CSA2_ERR_UNSUPPORTED_SHAPE, "cache.page_size must be 64 (got %d)",
          c.page_size);
  REQUIRE(c.num_pages > 0 && c.num_seqs > 0 && c.max_pages > 0, CSA2_ERR_INVALID_ARG,
          "cache.num_pages/num_seqs/max_pages must be positive");
  REQUIRE(c.num_pages <= (1 << 25), CSA2_ERR_UNSUPPORTED_SHAPE,
          "cache.num_pages must be <= 2^25 (row indices are 31-bit)");
  REQUIRE(c.d == 128 || c.d == 512, CSA2_ERR_UNSUPPORTED_SHAPE, "cache.d must be 128 or 512 (got %d)", c.d);
  if (need_codes) {
    REQUIRE(c.codes && c.scales, CSA2_ERR_INVALID_ARG, "cache.codes/scales is NULL");
    REQUIRE(((uintptr_t)c.codes & 15) == 0 && ((uintptr_t)c.scales & 15) == 0, CSA2_ERR_INVALID_ARG,
            "cache.codes/scales must be 16-byte aligned");
  }
  REQUIRE(c.idx_k_dtype == CSA2_BF16 || c.idx_k_dtype == CSA2_FP8E4M3, CSA2_ERR_INVALID_ARG,
          "cache.idx_k_dtype must be CSA2_BF16 or CSA2_FP8E4M3");
  if (need_idx) {
    if (c.idx_k_dtype == CSA2_BF16) {
      REQUIRE(c.idx_k, CSA2_ERR_INVALID_ARG, "cache.idx_k is NULL");
      REQUIRE(((uintptr_t)c.idx_k & 15) == 0, CSA2_ERR_INVALID_ARG, "cache.idx_k must be 16-byte aligned");
    } else {
      REQUIRE(c.idx_k8 && c.idx_k8_scale, CSA2_ERR_INVALID_ARG, "cache.idx_k8 / idx_k8_scale is NULL");
      REQUIRE(((uintptr_t)c.idx_k8 & 15) == 0 && ((uintptr_t)c.idx_k8_scale & 15) == 0, CSA2_ERR_INVALID_ARG,
              "cache.idx_k8 and idx_k8_scale must be 16-byte aligned");
    }
    REQUIRE(c.d_ik == 64 || c.d_ik == 128, CSA2_ERR_UNSUPPORTED_SHAPE, "cache.d_ik must be 64 or 128 (got %d)",
            c.d_ik);
  }
  return CSA2_OK;
}

csa2_status check_compress(const csa2_compress_args* a) {
  REQUIRE(a, CSA2_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->struct_size == sizeof(csa2_compress_args), CSA2_ERR_INVALID_ARG, "struct_size mismatch");
  REQUIRE(a->T >= 0, CSA2_ERR_INVALID_ARG, "T < 0");
  REQUIRE(a->m >= 1 && a->m <= 8, CSA2_ERR_UNSUPPORTED_SHAPE, "m must be in 1..8 (got %d)", a->m);
  REQUIRE(a->T % a->m == 0, CSA2_ERR_INVALID_ARG, "T (%d) is not a multiple of m (%d)", a->T, a->m);
  csa2_status s = check_cache(a->cache, true, a->W_ik != nullptr);
  if (s != CSA2_OK) return s;
  const int d = a->cache.d;
  if (a->W_kv) {
    REQUIRE(a->H, CSA2_ERR_INVALID_ARG, "H is NULL");
    REQUIRE(a->h_dtype == CSA2_BF16 || a->h_dtype == CSA2_F32, CSA2_ERR_INVALID_ARG, "bad h_dtype");
    REQUIRE(a->d_model > 0 && a->d_model % 32 == 0, CSA2_ERR_UNSUPPORTED_SHAPE,
            "d_model must be a positive multiple of 32 (got %d)", a->d_model);
    REQUIRE(a->m == 1 || a->W_z, CSA2_ERR_INVALID_ARG, "W_z is NULL with m > 1");
  } else {
    REQUIRE(a->C, CSA2_ERR_INVALID_ARG, "given mode: C is NULL");
    REQUIRE(a->m == 1 || a->Z, CSA2_ERR_INVALID_ARG, "given mode: Z is NULL with m > 1");
  }
  REQUIRE(a->d_rope == 0 || a->d_rope == 32 || a->d_rope == 64, CSA2_ERR_UNSUPPORTED_SHAPE,
          "d_rope must be 0, 32 or 64 (got %d)", a->d_rope);
  REQUIRE(a->d_rope <= d, CSA2_ERR_UNSUPPORTED_SHAPE, "d_rope > d");
  if (a->d_rope) {
    REQUIRE(a->rope_cos && a->rope_sin && a->pos, CSA2_ERR_INVALID_ARG, "RoPE tables or pos is NULL");
    REQUIRE(a->rope_max_pos > 0, CSA2_ERR_INVALID_ARG, "rope_max_pos must be positive");
  }
  if (a->T > 0) REQUIRE(a->seq && a->entry, CSA2_ERR_INVALID_ARG, "seq/entry is NULL");
  return CSA2_OK;
}

csa2_status check_append(const csa2_append_args* a) {
  REQUIRE(a, CSA2_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->struct_size == sizeof(csa2_append_args), CSA2_ERR_INVALID_ARG, "struct_size mismatch");
  REQUIRE(a->B >= 0, CSA2_ERR_INVALID_ARG, "B < 0");
  REQUIRE(a->m >= 1 && a->m <= 8, CSA2_ERR_UNSUPPORTED_SHAPE, "m must be in 1..8 (got %d)", a->m);
  csa2_status s = check_cache(a->cache, true, a->W_ik != nullptr);
  if (s != CSA2_OK) return s;
  REQUIRE(a->h_dtype == CSA2_BF16 || a->h_dtype == CSA2_F32, CSA2_ERR_INVALID_ARG, "bad h_dtype");
  REQUIRE(a->d_model > 0 && a->d_model % 32 == 0, CSA2_ERR_UNSUPPORTED_SHAPE,
          "d_model must be a positive multiple of 32 (got %d)", a->d_model);
  REQUIRE(a->d_rope == 0 || a->d_rope == 32 || a->d_rope == 64, CSA2_ERR_UNSUPPORTED_SHAPE,
          "d_rope must be 0, 32 or 64 (got %d)", a->d_rope);
  REQUIRE(a->d_rope <= a->cache.d, CSA2_ERR_UNSUPPORTED_SHAPE, "d_rope > d");
  if (a->B > 0) {
    REQUIRE(a->H && a->W_kv && a->seq && a->tok_pos, CSA2_ERR_INVALID_ARG, "H/W_kv/seq/tok_pos is NULL");
    REQUIRE(a->m == 1 || (a->W_z && a->pend), CSA2_ERR_INVALID_ARG, "W_z and pend are required when m > 1");
    if (a->d_rope)
      REQUIRE(a->rope_cos && a->rope_sin && a->rope_max_pos > 0, CSA2_ERR_INVALID_ARG,
              "RoPE tables are NULL or rope_max_pos <= 0");
    REQUIRE(((uintptr_t)a->H & 15) == 0 && ((uintptr_t)a->W_kv & 15) == 0 && ((uintptr_t)a->W_z & 15) == 0,
            CSA2_ERR_INVALID_ARG, "H, W_kv and W_z must be 16-byte aligned");
  }
  return CSA2_OK;
}

csa2_status check_index_common(int B, int H_i, const uint16_t* q, const float* w, const csa2_cache& c,
                               const int32_t* seq_of, int k, int* topk, int* topk_len) {
  REQUIRE(B >= 0, CSA2_ERR_INVALID_ARG, "B < 0");
  REQUIRE(H_i >= 1 && H_i <= 32, CSA2_ERR_UNSUPPORTED_SHAPE, "H_i must be in 1..32 (got %d)", H_i);
  REQUIRE(k >= 1 && k <= 2048, CSA2_ERR_UNSUPPORTED_SHAPE, "k must be in 1..2048 (got %d)", k);
  csa2_status s = check_cache(c, false, true);
  if (s != CSA2_OK) return s;
  if (B > 0) REQUIRE(q && w && seq_of && topk && topk_len, CSA2_ERR_INVALID_ARG, "a required pointer is NULL");
  return CSA2_OK;
}

csa2_status check_full(const csa2_index_full_args* a) {
  REQUIRE(a, CSA2_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->struct_size == sizeof(csa2_index_full_args), CSA2_ERR_INVALID_ARG, "struct_size mismatch");
  csa2_status s = check_index_common(a->B, a->H_i, a->q_idx, a->w, a->cache, a->seq_of, a->k, a->topk, a->topk_len);
  if (s != CSA2_OK) return s;
  REQUIRE(a->num_blocks >= 1 && a->per_block >= 1 && a->per_block <= 32, CSA2_ERR_UNSUPPORTED_SHAPE,
          "need num_blocks >= 1 and per_block in 1..32");
  REQUIRE((long long)a->num_blocks * a->per_block <= 16384, CSA2_ERR_UNSUPPORTED_SHAPE,
          "num_blocks * per_block must be <= 16384");
  REQUIRE(a->max_n >= 0 && (long long)a->max_n <= (long long)a->cache.max_pages * CSA2_PAGE_SIZE,
          CSA2_ERR_INVALID_ARG, "max_n must be in [0, max_pages*64]");
  if (a->B > 0) REQUIRE(a->n_vis && a->pool && a->pool_len, CSA2_ERR_INVALID_ARG, "a required pointer is NULL");
  REQUIRE(a->group >= 0, CSA2_ERR_INVALID_ARG, "group must be >= 0 (got %d)", a->group);
  if (a->group > 1) {
    REQUIRE(a->B % a->group == 0, CSA2_ERR_INVALID_ARG, "B (%d) must be a multiple of group (%d)", a->B, a->group);
  }
  return CSA2_OK;
}

csa2_status check_reindex(const csa2_index_reindex_args* a) {
  REQUIRE(a, CSA2_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->struct_size == sizeof(csa2_index_reindex_args), CSA2_ERR_INVALID_ARG, "struct_size mismatch");
  csa2_status s = check_index_common(a->B, a->H_i, a->q_idx, a->w, a->cache, a->seq_of, a->k, a->topk, a->topk_len);
  if (s != CSA2_OK) return s;
  REQUIRE(a->pool_stride >= 1 && a->pool_stride <= 16384, CSA2_ERR_UNSUPPORTED_SHAPE,
          "pool_stride must be in 1..16384");
  if (a->B > 0) REQUIRE(a->pool && a->pool_len, CSA2_ERR_INVALID_ARG, "pool/pool_len is NULL");
  return CSA2_OK;
}

csa2_status check_attn(const csa2_attn_args* a) {
  REQUIRE(a, CSA2_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->struct_size == sizeof(csa2_attn_args), CSA2_ERR_INVALID_ARG, "struct_size mismatch");
  REQUIRE(a->B >= 0, CSA2_ERR_INVALID_ARG, "B < 0");
  REQUIRE(a->Hq == 8 || a->Hq == 16 || a->Hq == 32 || a->Hq == 64, CSA2_ERR_UNSUPPORTED_SHAPE,
          "Hq must be 8, 16, 32 or 64 (got %d)", a->Hq);
  csa2_status s = check_cache(a->cache, true, false);
  if (s != CSA2_OK) return s;
  REQUIRE(a->k >= 0 && a->swa_max >= 0 && a->k + a->swa_max <= 4096, CSA2_ERR_UNSUPPORTED_SHAPE,
          "need k >= 0, swa_max >= 0, k + swa_max <= 4096");
  REQUIRE(a->out_dtype == CSA2_BF16 || a->out_dtype == CSA2_F32, CSA2_ERR_INVALID_ARG, "bad out_dtype");
  if (a->B > 0) {
    REQUIRE(a->q && a->seq_of && a->out, CSA2_ERR_INVALID_ARG, "q/seq_of/out is NULL");
    REQUIRE(((uintptr_t)a->q & 15) == 0, CSA2_ERR_INVALID_ARG, "q must be 16-byte aligned");
    if (a->k > 0) REQUIRE(a->topk, CSA2_ERR_INVALID_ARG, "topk is NULL");
    if (a->swa_max > 0)
      REQUIRE(a->swa && a->swa_scale && a->swa_start && a->swa_len && a->swa_rows > 0, CSA2_ERR_INVALID_ARG,
              "SWA pointers are NULL or swa_rows <= 0");
  }
  return CSA2_OK;
}

csa2_status check_swa_quant(const csa2_swa_quant_args* a) {
  REQUIRE(a, CSA2_ERR_INVALID_ARG, "args is NULL");
  REQUIRE(a->struct_size == sizeof(csa2_swa_quant_args), CSA2_ERR_INVALID_ARG, "struct_size mismatch");
  REQUIRE(a->R >= 0, CSA2_ERR_INVALID_ARG, "R < 0");
  REQUIRE(a->d == 128 || a->d == 512, CSA2_ERR_UNSUPPORTED_SHAPE, "d must be 128 or 512 (got %d)", a->d);
  REQUIRE(a->x_dtype == CSA2_BF16 || a->x_dtype == CSA2_F32, CSA2_ERR_INVALID_ARG, "bad x_dtype");
  if (a->R > 0) {
    REQUIRE(a->x && a->swa && a->swa_scale, CSA2_ERR_INVALID_ARG, "x/swa/swa_scale is NULL");
    REQUIRE(a->swa_rows > 0, CSA2_ERR_INVALID_ARG, "swa_rows must be positive");
    REQUIRE(a->row_idx || a->R <= a->swa_rows, CSA2_ERR_INVALID_ARG, "R > swa_rows without row_idx");
    REQUIRE(((uintptr_t)a->x & 15) == 0, CSA2_ERR_INVALID_ARG, "x must be 16-byte aligned");
    REQUIRE(((uintptr_t)a->swa & (a->d == 512 ? 15 : 3)) == 0, CSA2_ERR_INVALID_ARG,
            "swa must be 16-byte (d = 512) or 4-byte (d = 128) aligned");
  }
  return CSA2_OK;
}

csa2_status check_ws(size_t need, void* ws, size_t have) {
  REQUIRE(have >= need, CSA2_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes, got %zu", need, have);
  REQUIRE(need == 0 || ws, CSA2_ERR_INVALID_ARG, "workspace is NULL");
  REQUIRE(need == 0 || ((uintptr_t)ws & 255) == 0, CSA2_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return CSA2_OK;
}

}  // namespace

extern "C" {

csa2_status csa2_compress_quant_workspace(const csa2_compress_args* a, size_t* bytes) {
  csa2_status s = check_compress(a);
  if (s != CSA2_OK) return s;
  REQUIRE(bytes, CSA2_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = csa2::compress_workspace_bytes(*a);
  return ok();
}

csa2_status csa2_compress_quant(const csa2_compress_args* a, void* ws, size_t ws_bytes, void* stream) {
  csa2_status s = check_compress(a);
  if (s != CSA2_OK) return s;
  s = check_ws(csa2::compress_workspace_bytes(*a), ws, ws_bytes);
  if (s != CSA2_OK) return s;
  if (a->T == 0) return ok();
  return cuda_status(csa2::launch_compress(*a, ws, static_cast<cudaStream_t>(stream)), "csa2_compress_quant");
}

csa2_status csa2_compress_append_workspace(const csa2_append_args* a, size_t* bytes) {
  csa2_status s = check_append(a);
  if (s != CSA2_OK) return s;
  REQUIRE(bytes, CSA2_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = csa2::append_workspace_bytes(*a);
  return ok();
}

csa2_status csa2_compress_append(const csa2_append_args* a, void* ws, size_t ws_bytes, void* stream) {
  csa2_status s = check_append(a);
  if (s != CSA2_OK) return s;
  s = check_ws(csa2::append_workspace_bytes(*a), ws, ws_bytes);
  if (s != CSA2_OK) return s;
  return cuda_status(csa2::launch_append(*a, ws, static_cast<cudaStream_t>(stream)), "csa2_compress_append");
}

csa2_status csa2_index_full_workspace(const csa2_index_full_args* a, size_t* bytes) {
  csa2_status s = check_full(a);
  if (s != CSA2_OK) return s;
  REQUIRE(bytes, CSA2_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = csa2::index_full_workspace_bytes(*a);
  return ok();
}

csa2_status csa2_index_full(const csa2_index_full_args* a, void* ws, size_t ws_bytes, void* stream) {
  csa2_status s = check_full(a);
  if (s != CSA2_OK) return s;
  s = check_ws(csa2::index_full_workspace_bytes(*a), ws, ws_bytes);
  if (s != CSA2_OK) return s;
  return cuda_status(csa2::launch_index_full(*a, ws, static_cast<cudaStream_t>(stream)), "csa2_index_full");
}

csa2_status csa2_index_full_noalloc(const csa2_index_full_args* a, void* stream) {
  csa2_status s = check_full(a);
  if (s != CSA2_OK) return s;
  REQUIRE(a->cache.idx_k_dtype == CSA2_BF16, CSA2_ERR_UNSUPPORTED_SHAPE,
          "csa2_index_full_noalloc: the FP8 indexer-K form needs workspace for the quantised indexer Q; "
          "use csa2_index_full");
  const long long need = (long long)a->B * a->num_blocks * a->per_block;
  REQUIRE(need <= CSA2_NOALLOC_MAX_SCORES, CSA2_ERR_UNSUPPORTED_SHAPE,
          "csa2_index_full_noalloc: B*num_blocks*per_block = %lld exceeds the fixed scratch of %d scores",
          need, CSA2_NOALLOC_MAX_SCORES);
  void* scratch = nullptr;
  size_t have = 0;
  cudaError_t e = csa2::index_noalloc_scratch(&scratch, &have);
  if (e != cudaSuccess) return cuda_status(e, "csa2_index_full_noalloc: scratch address lookup");
  // the fixed scratch holds the pool scores only: no tensor-core score matrix
  return cuda_status(csa2::launch_index_full(*a, scratch, static_cast<cudaStream_t>(stream), false),
                     "csa2_index_full_noalloc");
}

csa2_status csa2_index_reindex_workspace(const csa2_index_reindex_args* a, size_t* bytes) {
  csa2_status s = check_reindex(a);
  if (s != CSA2_OK) return s;
  REQUIRE(bytes, CSA2_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = csa2::index_reindex_workspace_bytes(*a);
  return ok();
}

csa2_status csa2_index_reindex(const csa2_index_reindex_args* a, void* ws, size_t ws_bytes, void* stream) {
  csa2_status s = check_reindex(a);
  if (s != CSA2_OK) return s;
  s = check_ws(csa2::index_reindex_workspace_bytes(*a), ws, ws_bytes);
  if (s != CSA2_OK) return s;
  return cuda_status(csa2::launch_index_reindex(*a, ws, static_cast<cudaStream_t>(stream)), "csa2_index_reindex");
}

csa2_status csa2_sparse_attn_workspace(const csa2_attn_args* a, size_t* bytes) {
  csa2_status s = check_attn(a);
  if (s != CSA2_OK) return s;
  REQUIRE(bytes, CSA2_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = csa2::attn_workspace_bytes(*a);
  return ok();
}

csa2_status csa2_sparse_attn(const csa2_attn_args* a, void* ws, size_t ws_bytes, void* stream) {
  csa2_status s = check_attn(a);
  if (s != CSA2_OK) return s;
  s = check_ws(csa2::attn_workspace_bytes(*a), ws, ws_bytes);
  if (s != CSA2_OK) return s;
  return cuda_status(csa2::launch_attn(*a, ws, static_cast<cudaStream_t>(stream)), "csa2_sparse_attn");
}

csa2_status csa2_swa_quant(const csa2_swa_quant_args* a, void* stream) {
  csa2_status s = check_swa_quant(a);
  if (s != CSA2_OK) return s;
  return cuda_status(csa2::launch_swa_quant(*a, static_cast<cudaStream_t>(stream)), "csa2_swa_quant");
}

const char* csa2_last_error_message(void) { return g_msg; }

csa2_status csa2_get_device_error(uint32_t* word) {
  REQUIRE(word, CSA2_ERR_INVALID_ARG, "word is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e, "csa2_get_device_error");
  *word = csa2::read_clear_error_compress() | csa2::read_clear_error_proj() | csa2::read_clear_error_index() |
          csa2::read_clear_error_score() | csa2::read_clear_error_attn();
  csa2_status s = cuda_status(cudaGetLastError(), "csa2_get_device_error");
  if (s != CSA2_OK) return s;
  if (*word & CSA2_DEVERR_TIMEOUT) return fail(CSA2_ERR_TIMEOUT, "a bounded wait gave up (device word 0x%x)", *word);
  if (*word) return fail(CSA2_ERR_DEVICE_CHECK, "a device-side check failed (device word 0x%x)", *word);
  return CSA2_OK;
}

int32_t csa2_version(void) { return 100; }

csa2_status csa2_selftest_wait_timeout(int32_t polls, void* stream) {
  REQUIRE(polls >= 1 && polls <= (1 << 20), CSA2_ERR_INVALID_ARG, "polls must be in 1..2^20 (got %d)", polls);
  return cuda_status(csa2::launch_selftest_wait(polls, static_cast<cudaStream_t>(stream)),
                     "csa2_selftest_wait_timeout");
}

}  // extern "C"
