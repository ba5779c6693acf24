// Indexer scores of many queries of one sequence on the tensor cores (tcgen05), for the
// Full indexer of a prefill chunk, where thousands of causal queries score the same cache:
//   S[b][e] = sum_h w[b][h] * ReLU(q_idx[b][h] . idx_k[e])      (relu = 0: no ReLU)
// for every entry e below the tile's largest n_vis (entries past a query's own n_vis are
// written but never read).  Then every pool block keeps its best per_block entries.
//
// "DeepSeek-V4.1-Flash deep dive", section 3.1 (Indexer Q x Indexer K -> score) and 3.3
// (block top positions -> the shared candidate pool); the prefill form of that scan is a
// dense product of the chunk's indexer Q against the cache's indexer K.
//
// GEMM view: rows = 128 entries (two cache pages, by TMA through the page table), columns =
// 32 queries x 8 heads = 256, K = 128 dims; both operands K-major with a 128-byte swizzle.
// A persistent CTA takes units (query tile, run of CHUNK entry tiles): the query tile's
// 64 KB of Q stays in shared memory for the unit while the entry tiles stream through a
// 3-stage ring.
//   warp 0      TMA producer (Q tile once per unit, then the entry tiles)
//   warp 1      allocates 512 TMEM columns (two 256-column accumulators) and issues the
//               MMAs (M = 128, N = 256, K = 16, 8 per entry tile)
//   warps 2..5  epilogue: TMEM lane quarter w % 4 -> 32 entries; per query the weighted ReLU
//               sum of its 8 head columns, stored as S[b][e] (a warp writes 128 contiguous
//               bytes per query)
// Every wait is bounded: on expiry the kernel sets CSA2_DEVERR_TIMEOUT and stops issuing.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace csa2 {

CSA2_DEFINE_ERROR_WORD(g_err_score);

namespace stc {
constexpr int BM = 128;                    // entries per tile (two pages)
constexpr int QT = 32;                     // queries per tile
constexpr int HI = 8;                      // heads per query
constexpr int BN = QT * HI;                // 256 columns
constexpr int DK = 128;
constexpr int A_BYTES = BM * DK * 2;       // 32 KB: two 64-dim halves of 16 KB
constexpr int B_BYTES = BN * DK * 2;       // 64 KB: two halves of 32 KB
constexpr int STAGES = 3;
constexpr int CHUNK = 32;                  // entry tiles per unit
constexpr int SMEM = B_BYTES + STAGES * A_BYTES + 256;
constexpr int THREADS = 192;
constexpr uint32_t MAX_POLL = 1u << 24;
}  // namespace stc

struct ScoreParams {
  const int* n_vis;        // [B]
  const int* seq_of;       // [B]
  const float* w;          // [B][8]
  const int* page_table;   // [num_seqs][max_pages]
  int num_seqs, max_pages, num_pages;
  int B, max_n, ldS, relu;
  int ntiles, nchunks, units;
  float* S;                // [B][ldS]
};

// The unit's query tile, its entry tiles [t0, t1) (t1 <= t0: nothing to do) and sequence;
// called by a whole warp, every role computing the same values.
__device__ __forceinline__ void unit_span(const ScoreParams& p, int u, int& qt, int& t0, int& t1, int& seq) {
  const int lane = threadIdx.x & 31;
  qt = u / p.nchunks;
  const int ch = u % p.nchunks;
  const int b = qt * stc::QT + lane;
  const int n = max(0, min(__ldg(p.n_vis + b), p.max_n));
  const int nmax = __reduce_max_sync(0xffffffffu, n);
  seq = __ldg(p.seq_of + qt * stc::QT);
  t0 = ch * stc::CHUNK;
  t1 = min(t0 + stc::CHUNK, (nmax + stc::BM - 1) / stc::BM);
}

__global__ void __launch_bounds__(stc::THREADS, 1)
    k_score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap, ScoreParams p) {
  using namespace stc;
  pdl_wait();
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023) != 0) {                // the same in every CTA
    if (tid == 0) raise_error(&g_err_score, CSA2_DEVERR_SMEM_ALIGN);
    return;
  }
  uint8_t* sB = smem;
  uint8_t* sA = smem + B_BYTES;
  uint64_t* afull = reinterpret_cast<uint64_t*>(smem + B_BYTES + STAGES * A_BYTES);
  uint64_t* aempty = afull + STAGES;
  uint64_t* accf = aempty + STAGES;                  // [2]
  uint64_t* acce = accf + 2;                         // [2]
  uint64_t* bfull = acce + 2;
  uint64_t* bempty = bfull + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bempty + 1);
  if (warp == 1) tc::tmem_alloc(tslot, 2 * BN);
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&afull[s], 1);
      tc::mbar_init(&aempty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&accf[i], 1);
      tc::mbar_init(&acce[i], 4);                    // one arrival per epilogue warp
    }
    tc::mbar_init(bfull, 1);
    tc::mbar_init(bempty, 1);
    tc::fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  if (warp == 0) {                                   // ---- TMA producer
    long long it = 0;                                // entry tiles issued by this CTA
    int ul = 0;                                      // units with work
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      int qt, t0, t1, seq;
      unit_span(p, u, qt, t0, t1, seq);
      if (t1 <= t0) continue;
      // the queries of a tile share one sequence (a group of the call)
      if (__any_sync(0xffffffffu, __ldg(p.seq_of + qt * QT + lane) != seq) && lane == 0)
        raise_error(&g_err_score, CSA2_DEVERR_SEQ);
      if (lane == 0) {
        if (ul > 0 && !tc::mbar_wait(bempty, (uint32_t)((ul - 1) & 1), MAX_POLL)) {
          raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
          ok = false;
        }
        if (ok) {
          tc::mbar_arrive_expect_tx(bfull, B_BYTES);
          tc::tma_load_2d(sB, &qmap, 0, qt * BN, bfull);
          tc::tma_load_2d(sB + B_BYTES / 2, &qmap, 64, qt * BN, bfull);
        }
        const bool seq_ok = seq >= 0 && seq < p.num_seqs;
        if (!seq_ok) raise_error(&g_err_score, CSA2_DEVERR_SEQ);
        for (int t = t0; t < t1 && ok; ++t, ++it) {
          const int s = (int)(it % STAGES);
          if (it >= STAGES && !tc::mbar_wait(&aempty[s], (uint32_t)(((it / STAGES) - 1) & 1), MAX_POLL)) {
            raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
            ok = false;
            break;
          }
          int pg[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int slot = 2 * t + h;              // page slot of the sequence
            int v = 0;
            if (seq_ok && slot < p.max_pages) {
              v = __ldg(p.page_table + (long long)seq * p.max_pages + slot);
              if (v < 0 || v >= p.num_pages) {
                raise_error(&g_err_score, CSA2_DEVERR_PAGE_ID);
                v = 0;
              }
            }
            pg[h] = v;
          }
          uint8_t* st = sA + s * A_BYTES;
          tc::mbar_arrive_expect_tx(&afull[s], A_BYTES);
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tc::tma_load_2d(st + kh * (A_BYTES / 2) + h * (A_BYTES / 4), &kmap, 64 * kh, pg[h] * 64, &afull[s]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      it = __shfl_sync(0xffffffffu, it, 0);
      ++ul;
    }
  } else if (warp == 1) {                            // ---- MMA issuer
    constexpr uint32_t idesc = tc::idesc_f16(BM, BN, 1, 0, 0);   // bf16, both K-major
    long long it = 0;
    int tl = 0, ul = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      int qt, t0, t1, seq;
      unit_span(p, u, qt, t0, t1, seq);
      if (t1 <= t0) continue;
      if (lane == 0) {
        if (!tc::mbar_wait(bfull, (uint32_t)(ul & 1), MAX_POLL)) {
          raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
          ok = false;
        }
        tc::fence_after_sync();
        for (int t = t0; t < t1 && ok; ++t, ++it, ++tl) {
          const int s = (int)(it % STAGES), buf = tl & 1;
          if (tl >= 2 && !tc::mbar_wait(&acce[buf], (uint32_t)(((tl >> 1) - 1) & 1), MAX_POLL)) {
            raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
            ok = false;
            break;
          }
          if (!tc::mbar_wait(&afull[s], (uint32_t)((it / STAGES) & 1), MAX_POLL)) {
            raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a = smem_u32(sA + s * A_BYTES), bb = smem_u32(sB);
#pragma unroll
          for (int k16 = 0; k16 < DK / 16; ++k16) {
            const uint32_t off = (uint32_t)((k16 & 3) * 32);
            const uint64_t ad = tc::smem_desc_sw128(a + (k16 >> 2) * (A_BYTES / 2) + off, 16, 1024);
            const uint64_t bd = tc::smem_desc_sw128(bb + (k16 >> 2) * (B_BYTES / 2) + off, 16, 1024);
            tc::mma_f16_ss(tb + (uint32_t)(BN * buf), ad, bd, idesc, k16 > 0 ? 1u : 0u);
          }
          tc::mma_commit(&aempty[s]);
          tc::mma_commit(&accf[buf]);
        }
        tc::mma_commit(bempty);                      // the Q tile may be replaced
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      it = __shfl_sync(0xffffffffu, it, 0);
      tl = __shfl_sync(0xffffffffu, tl, 0);
      ++ul;
    }
  } else {                                           // ---- epilogue
    const int q4 = warp & 3;                         // TMEM lane quarter
    int tl = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      int qt, t0, t1, seq;
      unit_span(p, u, qt, t0, t1, seq);
      for (int t = t0; t < t1; ++t, ++tl) {
        const int buf = tl & 1;
        ok = tc::mbar_wait_warp(&accf[buf], (uint32_t)((tl >> 1) & 1), MAX_POLL);
        if (!ok) {
          if (lane == 0) raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
          break;
        }
        tc::fence_after_sync();
        const int e = t * BM + 32 * q4 + lane;       // this thread's entry
        const uint32_t tq = tb + ((uint32_t)(32 * q4) << 16) + (uint32_t)(BN * buf);
#pragma unroll 1
        for (int qc = 0; qc < QT / 4; ++qc) {        // 4 queries (32 columns) at a time
          uint32_t r[32];
          tc::tmem_ld32(tq + (uint32_t)(32 * qc), r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int b = qt * QT + 4 * qc + k;
            const float4 w0 = __ldg(reinterpret_cast<const float4*>(p.w + (long long)b * HI));
            const float4 w1 = __ldg(reinterpret_cast<const float4*>(p.w + (long long)b * HI) + 1);
            const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            float sc = 0.f;
#pragma unroll
            for (int h = 0; h < HI; ++h) {
              float x = __uint_as_float(r[8 * k + h]);
              if (p.relu) x = fmaxf(x, 0.f);
              sc = fmaf(wv[h], x, sc);
            }
            p.S[(long long)b * p.ldS + e] = sc;
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce[buf]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tb, 2 * BN);
}

// Best per_block entries of every block of every query from the score matrix.  A warp takes
// 32 consecutive blocks of one query: it copies their scores (at most 64 per block) into
// shared memory with coalesced loads, then lane i keeps the best of block i and writes them
// to the pool (and their scores to pool_score) in ascending entry order, at the offsets of
// the scan kernels.  "Best" = larger score, then lower entry.
constexpr int BT_WARPS = 4;
// A warp's scores sit in shared memory with one pad word after every 32, so that lanes
// walking blocks of ~16 entries side by side read distinct banks.
__device__ __forceinline__ int bt_pad(int i) { return i + (i >> 5); }
__host__ __device__ constexpr int bt_warp_floats(int per_blk) { return 32 * per_blk + per_blk + 1; }
template <int P>
__global__ void __launch_bounds__(BT_WARPS * 32) k_block_topp(const float* __restrict__ S, int ldS,
                                                              const int* __restrict__ n_vis, int max_n, int B, int NB,
                                                              int wfloats, int* __restrict__ pool,
                                                              float* __restrict__ pool_score) {
  pdl_wait();
  extern __shared__ float bt_sh[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int segs = (NB + 31) / 32;
  const long long gw = (long long)blockIdx.x * BT_WARPS + warp;
  if (gw >= (long long)B * segs) return;
  const int b = (int)(gw / segs), j0 = (int)(gw % segs) * 32;
  const int n = max(0, min(__ldg(n_vis + b), max_n));
  // block bounds floor(j n / NB): in 32 bits when j n fits (the usual case), one per lane,
  // the next lane's lower bound being this lane's upper one
  const bool narrow = (unsigned long long)n * (unsigned)NB <= 0xFFFFFFFFull;
  auto bound = [&](int jj) -> int {
    return narrow ? (int)(((unsigned)jj * (unsigned)n) / (unsigned)NB) : (int)(((long long)jj * n) / NB);
  };
  const int j = j0 + lane;
  const int lo = bound(min(j, NB));
  int hi = __shfl_down_sync(0xffffffffu, lo, 1);
  if (lane == 31) hi = bound(min(j + 1, NB));
  const int e0 = __shfl_sync(0xffffffffu, lo, 0);
  const int e1 = __shfl_sync(0xffffffffu, hi, min(31, NB - 1 - j0));
  const float* s = S + (long long)b * ldS;
  float* w = bt_sh + warp * wfloats;
  // the warp's slice, eight loads in flight per lane
  for (int e = e0 + lane; e < e1; e += 256) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = (e + 32 * u < e1) ? __ldg(s + e + 32 * u) : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (e + 32 * u < e1) w[bt_pad(e + 32 * u - e0)] = v[u];
  }
  __syncwarp();
  if (j >= NB) return;
  // the P best values, descending: each score bubbles down the sorted list (a later
  // entry never displaces an equal earlier one, so this is the best-first order of the
  // tie rule "larger score, then lower entry")
  float kv[P];
#pragma unroll
  for (int i = 0; i < P; ++i) kv[i] = -INFINITY;
  for (int e = lo; e < hi; ++e) {
    float v = w[bt_pad(e - e0)];
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const float t = fmaxf(v, kv[i]);
      v = fminf(v, kv[i]);
      kv[i] = t;
    }
  }
  const int cnt = hi - lo;
  if (cnt <= 0) return;
  // kept: every entry above the P-th best tv, then entries equal to tv in ascending order
  // up to P in all; a block of fewer than P entries keeps them all
  const float tv = (cnt >= P) ? kv[P - 1] : -INFINITY;
  int quota = P;
#pragma unroll
  for (int i = 0; i < P; ++i) quota -= (kv[i] > tv) ? 1 : 0;
  const long long off = ((long long)n >= (long long)P * NB) ? (long long)P * j : lo;
  const long long o = (long long)b * NB * P + off;
  int c = 0;
  for (int e = lo; e < hi; ++e) {                     // ascending entries that are kept
    const float v = w[bt_pad(e - e0)];
    if (v > tv || (v == tv && quota-- > 0)) {
      pool[o + c] = e;
      pool_score[o + c] = v;
      ++c;
    }
  }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
bool full_scores_tc_supported(const csa2_index_full_args& a) {
  return a.group >= stc::QT && a.group % stc::QT == 0 && a.B % a.group == 0 && a.H_i == stc::HI &&
         a.cache.d_ik == stc::DK && a.per_block <= 16 && (long long)a.max_n <= 64LL * a.num_blocks &&
         a.max_n > 0 && ((uintptr_t)a.q_idx & 15) == 0 && ((uintptr_t)a.cache.idx_k & 15) == 0 &&
         ((uintptr_t)a.w & 15) == 0 && tensor_map_encoder() != nullptr;
}

size_t full_scores_tc_bytes(const csa2_index_full_args& a) {
  const long long ld = ((long long)a.max_n + stc::BM - 1) / stc::BM * stc::BM;
  return (size_t)a.B * ld * sizeof(float);
}

cudaError_t launch_full_scores_tc(const csa2_index_full_args& a, float* S, float* pool_score, cudaStream_t st) {
  using namespace stc;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_score_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  ScoreParams p{};
  p.n_vis = a.n_vis;
  p.seq_of = a.seq_of;
  p.w = a.w;
  p.page_table = a.cache.page_table;
  p.num_seqs = a.cache.num_seqs;
  p.max_pages = a.cache.max_pages;
  p.num_pages = a.cache.num_pages;
  p.B = a.B;
  p.max_n = a.max_n;
  p.ntiles = (a.max_n + BM - 1) / BM;
  p.ldS = p.ntiles * BM;
  p.relu = a.relu;
  p.nchunks = (p.ntiles + CHUNK - 1) / CHUNK;
  p.units = (a.B / QT) * p.nchunks;
  p.S = S;
  CUtensorMap kmap, qmap;                            // idx_k rows (64-row boxes: one page), Q rows (256)
  if (!bf16_map(&kmap, a.cache.idx_k, (long long)a.cache.num_pages * 64, DK, 64) ||
      !bf16_map(&qmap, a.q_idx, (long long)a.B * HI, DK, BN))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::max(1, std::min(p.units, sms > 0 ? sms : 1));
  cudaError_t e = launch_k(k_score_tc, grid, THREADS, SMEM, st, kmap, qmap, p);
  if (e != cudaSuccess) return e;
  const long long warps = (long long)a.B * ((a.num_blocks + 31) / 32);
  const unsigned grid2 = (unsigned)((warps + BT_WARPS - 1) / BT_WARPS);
  // entries per block at most: ceil(max_n / NB) <= 64
  const int per_blk = (int)(((long long)a.max_n + a.num_blocks - 1) / a.num_blocks);
  const int wfloats = bt_warp_floats(per_blk);
  const size_t smem2 = (size_t)BT_WARPS * wfloats * sizeof(float);
  switch (a.per_block) {                             // the kept list lives in registers
#define CSA2_BT(PP) \
  case PP: return launch_k(k_block_topp<PP>, grid2, BT_WARPS * 32, smem2, st, S, p.ldS, a.n_vis, a.max_n, a.B, \
                           a.num_blocks, wfloats, a.pool, pool_score);
    CSA2_BT(1) CSA2_BT(2) CSA2_BT(3) CSA2_BT(4) CSA2_BT(5) CSA2_BT(6) CSA2_BT(7) CSA2_BT(8)
    CSA2_BT(9) CSA2_BT(10) CSA2_BT(11) CSA2_BT(12) CSA2_BT(13) CSA2_BT(14) CSA2_BT(15) CSA2_BT(16)
#undef CSA2_BT
    default: return cudaErrorInvalidValue;
  }
}

uint32_t read_clear_error_score() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_score, sizeof(v));
  cudaMemcpyToSymbol(g_err_score, &z, sizeof(z));
  return v;
}

}  // namespace csa2
