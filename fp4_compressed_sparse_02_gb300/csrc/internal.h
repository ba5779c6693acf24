// Launchers shared between the kernel units and the host API layer.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "csa2.h"

namespace csa2 {

// compress.cu
size_t compress_workspace_bytes(const csa2_compress_args& a);
cudaError_t launch_compress(const csa2_compress_args& a, void* ws, cudaStream_t st);
uint32_t read_clear_error_compress();
cudaError_t launch_swa_quant(const csa2_swa_quant_args& a, cudaStream_t st);
size_t append_workspace_bytes(const csa2_append_args& a);
cudaError_t launch_append(const csa2_append_args& a, void* ws, cudaStream_t st);

// proj_tc.cu: tensor-core projection for many bf16 tokens (out[T][d or 2d], fp32)
bool project_tc_supported(const csa2_compress_args& a);
bool project_tc_fused(const csa2_compress_args& a);     // pooling, RoPE and FP4 in the epilogue
cudaError_t launch_project_tc(const csa2_compress_args& a, float* out, bool fuse, cudaStream_t st);
uint32_t read_clear_error_proj();
bool index_k_tc_supported(const csa2_compress_args& a, int G);
cudaError_t launch_index_k_tc(const csa2_compress_args& a, int G, cudaStream_t st);

// score_tc.cu: Full-indexer scores of many queries of one sequence on the tensor cores
// (csa2_index_full with group >= 32), then each block's best entries into the pool
bool full_scores_tc_supported(const csa2_index_full_args& a);
size_t full_scores_tc_bytes(const csa2_index_full_args& a);
cudaError_t launch_full_scores_tc(const csa2_index_full_args& a, float* S, float* pool_score, cudaStream_t st);
uint32_t read_clear_error_score();

// index.cu
size_t index_full_workspace_bytes(const csa2_index_full_args& a);
// allow_tc = false keeps the scan (the workspace then holds the pool scores only)
cudaError_t launch_index_full(const csa2_index_full_args& a, void* ws, cudaStream_t st, bool allow_tc = true);
// whether the Full call scores on the tensor cores (supported and chosen for this shape)
bool full_scores_tc_chosen(const csa2_index_full_args& a);
size_t index_reindex_workspace_bytes(const csa2_index_reindex_args& a);
cudaError_t launch_index_reindex(const csa2_index_reindex_args& a, void* ws, cudaStream_t st);
uint32_t read_clear_error_index();
// device address of the fixed score array used by csa2_index_full_noalloc on the
// current device (looked up once per device)
cudaError_t index_noalloc_scratch(void** ptr, size_t* bytes);

// attn.cu
size_t attn_workspace_bytes(const csa2_attn_args& a);
cudaError_t launch_attn(const csa2_attn_args& a, void* ws, cudaStream_t st);
uint32_t read_clear_error_attn();
cudaError_t launch_selftest_wait(int polls, cudaStream_t st);

}  // namespace csa2
