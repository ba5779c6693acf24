// Compressor projection on the tensor cores (tcgen05), for many tokens:
//   out[t][n] = sum_k H[t][k] * W[k][n],  W = [W_KV | W_Z] (columns n < d from W_KV,
//   n >= d from W_Z when the group size m > 1),  bf16 inputs, fp32 accumulation and output.
//
// "DeepSeek-V4.1-Flash deep dive", section 2: C = H . W_KV and Z = H . W_Z are the
// layer's linear projections of the hidden states; the pooling, RoPE and FP4 quantisation
// that follow read `out` (k_quant).
//
// CTA = one 128 x 256 output tile, 192 threads:
//   warp 0      TMA producer: per 64-deep K block, H box [128 rows x 64] (K-major) and
//               four W boxes [64 K rows x 64 columns] (MN-major), 128-byte swizzle, into a
//               4-stage ring (48 KB a stage); the stage's mbarrier counts the bytes.
//   warp 1      allocates 256 TMEM columns and issues the MMAs (M = 128, N = 256, K = 16,
//               4 per stage); each stage is released to the producer by tcgen05.commit.
//   warps 2..5  epilogue: TMEM lanes 32 (w % 4).. -> fp32 rows of `out`.
// Every wait is bounded: on expiry the kernel sets CSA2_DEVERR_TIMEOUT and stops issuing.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace csa2 {

CSA2_DEFINE_ERROR_WORD(g_err_proj);

namespace ptc {
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;                 // 16 KB
constexpr int B_BYTES = BN * BK * 2;                 // 32 KB: four 64-column blocks of 8 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM = STAGES * STAGE_BYTES + 128;     // + mbarriers and the TMEM slot
constexpr int THREADS = 192;
constexpr uint32_t MAX_POLL = 1u << 24;
}  // namespace ptc

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      :: "r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(map), "r"((uint32_t)__cvta_generic_to_shared(mbar)),
         "r"(x), "r"(y)
      : "memory");
}

__global__ void __launch_bounds__(ptc::THREADS, 1)
    k_proj_tc(const __grid_constant__ CUtensorMap mh, const __grid_constant__ CUtensorMap mkv,
              const __grid_constant__ CUtensorMap mz, float* __restrict__ out, int T, int d_model, int d, int N) {
  using namespace ptc;
  pdl_wait();                                        // many waves: dependents start at completion
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023) != 0) {                // the same in every CTA
    if (tid == 0) raise_error(&g_err_proj, CSA2_DEVERR_SMEM_ALIGN);
    return;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accf + 1);
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const CUtensorMap* mw = (n0 < d) ? &mkv : &mz;
  const int nw0 = (n0 < d) ? n0 : n0 - d;
  if (warp == 1) tc::tmem_alloc(tslot, BN);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(accf, 1);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  const int nk = d_model / BK;
  if (warp == 0) {
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % STAGES;
        if (kb >= STAGES && !tc::mbar_wait(&empty[s], ((kb / STAGES) - 1) & 1, MAX_POLL)) {
          raise_error(&g_err_proj, CSA2_DEVERR_TIMEOUT);
          break;
        }
        uint8_t* st = smem + s * STAGE_BYTES;
        tc::mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
        tma_load_2d(st, &mh, kb * BK, m0, &full[s]);
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) tma_load_2d(st + A_BYTES + j * 8192, mw, nw0 + 64 * j, kb * BK, &full[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_f16(BM, BN, 1, 0, 1);   // bf16; A K-major, B MN-major
      bool ok = true;
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % STAGES;
        if (!tc::mbar_wait(&full[s], (kb / STAGES) & 1, MAX_POLL)) {
          raise_error(&g_err_proj, CSA2_DEVERR_TIMEOUT);
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a = smem_u32(smem + s * STAGE_BYTES), bb = a + A_BYTES;
#pragma unroll
        for (int k16 = 0; k16 < BK / 16; ++k16) {
          const uint64_t ad = tc::smem_desc_sw128(a + 32 * k16, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(bb + 2048 * k16, 8192, 1024);
          tc::mma_f16_ss(tb, ad, bd, idesc, (kb | k16) != 0 ? 1u : 0u);
        }
        tc::mma_commit(&empty[s]);                 // the stage is free once these have read it
      }
      tc::mma_commit(accf);                        // the accumulator is complete
    }
  } else {
    const int q = warp & 3;                        // warps 2..5 -> lane quarters 2, 3, 0, 1
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(accf, 0, MAX_POLL));
    if (!ok && lane == 0) raise_error(&g_err_proj, CSA2_DEVERR_TIMEOUT);
    tc::fence_after_sync();
    if (ok) {
      const int row = m0 + 32 * q + lane;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tc::tmem_ld32(tb + ((uint32_t)(32 * q) << 16) + (uint32_t)c, r);
        tc::tmem_ld_wait();
        if (row < T) {
          float4* o = reinterpret_cast<float4*>(out + (long long)row * N + n0 + c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                               __uint_as_float(r[4 * i + 3]));
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tb, BN);
}

// ---------------------------------------------------------------------------------
// Indexer K of many entries on the tensor cores: idx_k[g] = bf16_RNE(dequant(entry g) .
// W_IK), "DeepSeek-V4.1-Flash deep dive", section 3.1 (indexer K projected from Main K).
// CTA = 128 entries, 256 threads, d = 512 and d_ik = 128, K in two halves of 256:
// threads gather the entries' FP4 codes and scales through the page table and dequantise
// them to bf16 (E2M1 x E4M3 is exact in bf16) into a 128-byte-swizzled K-major tile, and
// stage W_IK rows into an MN-major tile; one thread issues M = 128, N = 128 MMAs into 128
// TMEM columns; four warps round the rows to bf16 and store them through the page table.
// ---------------------------------------------------------------------------------
namespace iktc {
constexpr int M = 128, NK = 128, KH = 256;
constexpr int A_ATOM = M / 8 * 1024;                 // bytes per 64-dim atom of the A tile
constexpr int A_BYTES = M * KH * 2;                  // 64 KB
constexpr int B_BYTES = KH * NK * 2;                 // 64 KB: two 64-column blocks
constexpr int SMEM = A_BYTES + B_BYTES + 64 + M * 8;   // + mbarrier, TMEM slot, flag, rows
constexpr int THREADS = 256;
constexpr uint32_t MAX_POLL = 1u << 24;
}  // namespace iktc

__global__ void __launch_bounds__(iktc::THREADS, 1)
    k_index_k_tc(csa2_cache cache, const int* __restrict__ seq, const int* __restrict__ entry, int G,
                 const uint16_t* __restrict__ Wik) {
  using namespace iktc;
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023) != 0) {
    if (tid == 0) raise_error(&g_err_proj, CSA2_DEVERR_SMEM_ALIGN);
    return;
  }
  uint8_t* sA = smem;
  uint8_t* sB = smem + A_BYTES;
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + A_BYTES + B_BYTES);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mb + 1);
  int& ok_flag = *reinterpret_cast<int*>(mb + 2);
  long long* rows = reinterpret_cast<long long*>(smem + A_BYTES + B_BYTES + 64);
  if (warp == 0) tc::tmem_alloc(tslot, NK);
  if (tid == 32) {
    tc::mbar_init(mb, 1);
    ok_flag = 1;
  }
  if (tid < M) {
    const int g = blockIdx.x * M + tid;
    rows[tid] = (g < G) ? entry_row(cache, __ldg(seq + g), __ldg(entry + g), &g_err_proj) : -1;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  const uint32_t a_s = smem_u32(sA), b_s = smem_u32(sB);
  const int r = tid >> 1, part = tid & 1;            // A: entry r, 128 dims of the half
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    if (h == 1) {                                    // the first half's products have read the tiles
      if (tid == 0 && ok_flag && !tc::mbar_wait(mb, 0, MAX_POLL)) {
        raise_error(&g_err_proj, CSA2_DEVERR_TIMEOUT);
        ok_flag = 0;
      }
      __syncthreads();
      tc::fence_after_sync();
    }
    const long long row = rows[r];
    uint4 cw[4];
    uint2 sw = make_uint2(0, 0);
    if (row >= 0) {
      const uint4* cp = reinterpret_cast<const uint4*>(cache.codes + row * 256 + 128 * h + 64 * part);
#pragma unroll
      for (int i = 0; i < 4; ++i) cw[i] = __ldg(cp + i);
      sw = __ldg(reinterpret_cast<const uint2*>(cache.scales + row * 32 + 16 * h + 8 * part));
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) cw[i] = make_uint4(0, 0, 0, 0);
    }
    const uint32_t sbytes[2] = {sw.x, sw.y};
    const uint32_t words[16] = {cw[0].x, cw[0].y, cw[0].z, cw[0].w, cw[1].x, cw[1].y, cw[1].z, cw[1].w,
                                cw[2].x, cw[2].y, cw[2].z, cw[2].w, cw[3].x, cw[3].y, cw[3].z, cw[3].w};
#pragma unroll
    for (int c = 0; c < 16; ++c) {                   // chunk of 8 dims: 4 code bytes, scale c / 2
      const float sc = e4m3_to_f32((sbytes[c >> 3] >> (8 * ((c >> 1) & 3))) & 0xffu);
      uint32_t o[4];
#pragma unroll
      for (int b2 = 0; b2 < 4; ++b2) {
        const uint32_t h2 = e2m1x2_to_f16x2((words[c] >> (8 * b2)) & 0xffu);
        const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
        const __nv_bfloat162 bv = __floats2bfloat162_rn(__low2float(hv) * sc, __high2float(hv) * sc);
        o[b2] = *reinterpret_cast<const uint32_t*>(&bv);
      }
      const int ch = 16 * part + c;                  // 16-byte chunk of the half's row
      *reinterpret_cast<uint4*>(sA + (ch >> 3) * A_ATOM + (r >> 3) * 1024 + (r & 7) * 128 + (((ch & 7) ^ (r & 7)) << 4)) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {                   // W_IK rows [256 h, 256 h + 256), 16 chunks each
      const int idx = tid + i * THREADS, k = idx >> 4, n8 = idx & 15;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(Wik + (long long)(KH * h + k) * NK + 8 * n8));
      *reinterpret_cast<uint4*>(sB + (n8 >> 3) * (KH * 128) + (k >> 3) * 1024 + (k & 7) * 128 + (((n8 & 7) ^ (k & 7)) << 4)) = v;
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0 && ok_flag) {
      constexpr uint32_t idesc = tc::idesc_f16(M, NK, 1, 0, 1);   // bf16; A K-major, B MN-major
#pragma unroll
      for (int ks = 0; ks < KH / 16; ++ks) {
        const uint64_t ad = tc::smem_desc_sw128(a_s + (ks >> 2) * A_ATOM + (ks & 3) * 32, 16, 1024);
        const uint64_t bd = tc::smem_desc_sw128(b_s + ks * 2048, KH * 128, 1024);
        tc::mma_f16_ss(tb, ad, bd, idesc, (h | ks) != 0 ? 1u : 0u);
      }
      tc::mma_commit(mb);
    }
  }
  if (tid == 0 && ok_flag && !tc::mbar_wait(mb, 1, MAX_POLL)) {
    raise_error(&g_err_proj, CSA2_DEVERR_TIMEOUT);
    ok_flag = 0;
  }
  __syncthreads();
  tc::fence_after_sync();
  if (warp < 4 && ok_flag) {                         // warp w: TMEM lanes (rows) 32 w ..
    const long long row = rows[32 * warp + lane];
#pragma unroll 1
    for (int c = 0; c < NK; c += 32) {
      uint32_t v[32];
      tc::tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, v);
      tc::tmem_ld_wait();
      if (row >= 0) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 bv = __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          pk[i] = *reinterpret_cast<const uint32_t*>(&bv);
        }
        uint4* dst = reinterpret_cast<uint4*>(cache.idx_k + row * NK + c);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, NK);
}

bool index_k_tc_supported(const csa2_compress_args& a, int G) {
  return G >= 256 && a.cache.d == 512 && a.cache.d_ik == iktc::NK && ((uintptr_t)a.W_ik & 15) == 0;
}

cudaError_t launch_index_k_tc(const csa2_compress_args& a, int G, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_index_k_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, iktc::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_k(k_index_k_tc, (G + iktc::M - 1) / iktc::M, iktc::THREADS, iktc::SMEM, st, a.cache, a.seq, a.entry,
                  G, a.W_ik);
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

// bf16 matrix [rows][cols] (row stride `cols` elements), boxes of box_rows x 64 columns,
// 128-byte swizzle (the canonical operand layout of the MMA).
static bool bf16_map(CUtensorMap* map, const void* base, long long rows, long long cols, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool project_tc_supported(const csa2_compress_args& a) {
  const int N = a.cache.d * (a.m > 1 ? 2 : 1);
  const bool aligned = ((uintptr_t)a.H & 15) == 0 && ((uintptr_t)a.W_kv & 15) == 0 &&
                       (a.m == 1 || ((uintptr_t)a.W_z & 15) == 0);
  return a.h_dtype == CSA2_BF16 && a.T > 64 && a.d_model % ptc::BK == 0 && a.cache.d % ptc::BN == 0 &&
         N % ptc::BN == 0 && aligned && tensor_map_encoder() != nullptr;
}

cudaError_t launch_project_tc(const csa2_compress_args& a, float* out, cudaStream_t st) {
  const int d = a.cache.d, N = d * (a.m > 1 ? 2 : 1);
  CUtensorMap mh, mkv, mz;
  if (!bf16_map(&mh, a.H, a.T, a.d_model, ptc::BM) || !bf16_map(&mkv, a.W_kv, a.d_model, d, ptc::BK) ||
      !bf16_map(&mz, a.m > 1 ? a.W_z : a.W_kv, a.d_model, d, ptc::BK))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_proj_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, ptc::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const dim3 grid(N / ptc::BN, (a.T + ptc::BM - 1) / ptc::BM);
  return launch_k(k_proj_tc, grid, ptc::THREADS, ptc::SMEM, st, mh, mkv, mz, out, a.T, a.d_model, d, N);
}

uint32_t read_clear_error_proj() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_proj, sizeof(v));
  if (v) cudaMemcpyToSymbol(g_err_proj, &z, sizeof(z));
  return v;
}

}  // namespace csa2
