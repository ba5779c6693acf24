// Indexer scores of groups of queries of one sequence on the tensor cores (tcgen05):
//   S[b][e] = sum_h w[b][h] * ReLU(q_idx[b][h] . idx_k[e])      (relu = 0: no ReLU)
// for every entry e below the tile's largest n_vis (entries past a query's own n_vis are
// written but never read).  Then every pool block keeps its best per_block entries.  The
// groups are a prefill chunk's causal queries, the positions of a decode verification
// step, or single decode queries with many indexer heads: the rows of the cache are
// streamed once per group and scored against all of its heads in one product.
//
// "DeepSeek-V4.1-Flash deep dive", section 3.1 (Indexer Q x Indexer K -> score) and 3.3
// (block top positions -> the shared candidate pool).
//
// GEMM view: rows = 128 entries (two cache pages, by TMA through the page table), columns =
// QT queries x HI heads (padded to a multiple of 16, at most 256), K = 128 dims; both
// operands K-major with a 128-byte swizzle.  A persistent CTA takes units (query tile, run
// of `chunk` entry tiles): the query tile's Q stays in shared memory for the unit while the
// entry tiles stream through a 4-stage ring.
//   warp 0      TMA producer (Q tile once per unit, then the entry tiles)
//   warp 1      allocates TMEM (two accumulators) and issues the MMAs (M = 128, N = BN,
//               K = 16, 8 per entry tile)
//   warps 2..5  epilogue: TMEM lane quarter w % 4 -> 32 entries; per query the weighted ReLU
//               sum of its HI head columns, stored as S[b][e] (a warp writes 128 contiguous
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
constexpr int BN_MAX = 256;                // columns (queries x heads) at most
constexpr int DK = 128;
constexpr int A_BYTES = BM * DK * 2;       // 32 KB: two 64-dim halves of 16 KB
constexpr int STAGES = 4;
constexpr int W_BYTES = 4 * BN_MAX * 4;      // each epilogue warp's copy of the unit's head weights
constexpr int SMEM_MAX = BN_MAX * DK * 2 + STAGES * A_BYTES + 256 + W_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t MAX_POLL = 1u << 24;
}  // namespace stc

struct ScoreParams {
  const int* n_vis;        // [B]
  const int* seq_of;       // [B]
  const float* w;          // [B][HI]
  const int* page_table;   // [num_seqs][max_pages]
  int num_seqs, max_pages, num_pages;
  int B, max_n, ldS, relu;
  int QT, BN, bufcols;     // queries per tile, MMA columns (QT * HI padded to 16), TMEM columns per accumulator
  int ntiles, chunk, nchunks, units;
  float* S;                // [B][ldS]
};

// The unit's query tile, its entry tiles [t0, t1) (t1 <= t0: nothing to do) and sequence;
// called by a whole warp, every role computing the same values.
__device__ __forceinline__ void unit_span(const ScoreParams& p, int u, int& qt, int& t0, int& t1, int& seq) {
  const int lane = threadIdx.x & 31;
  qt = u / p.nchunks;
  const int ch = u % p.nchunks;
  const int b = qt * p.QT + lane;
  const int n = lane < p.QT ? max(0, min(__ldg(p.n_vis + b), p.max_n)) : 0;
  const int nmax = __reduce_max_sync(0xffffffffu, n);
  seq = __ldg(p.seq_of + qt * p.QT);
  t0 = ch * p.chunk;
  t1 = min(t0 + p.chunk, (nmax + stc::BM - 1) / stc::BM);
}

template <int HI>
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
  const int BN = p.BN;
  const int B_BYTES = BN * DK * 2;                   // a multiple of 4 KB
  uint8_t* sB = smem;
  uint8_t* sA = smem + B_BYTES;
  uint64_t* afull = reinterpret_cast<uint64_t*>(smem + B_BYTES + STAGES * A_BYTES);
  uint64_t* aempty = afull + STAGES;
  uint64_t* accf = aempty + STAGES;                  // [2]
  uint64_t* acce = accf + 2;                         // [2]
  uint64_t* bfull = acce + 2;
  uint64_t* bempty = bfull + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bempty + 1);
  const uint32_t tcols = (uint32_t)(2 * p.bufcols);  // a power of two >= 32
  if (warp == 1) tc::tmem_alloc(tslot, tcols);
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
      if (__any_sync(0xffffffffu, lane < p.QT && __ldg(p.seq_of + qt * p.QT + lane) != seq) && lane == 0)
        raise_error(&g_err_score, CSA2_DEVERR_SEQ);
      if (lane == 0) {
        if (ul > 0 && !tc::mbar_wait(bempty, (uint32_t)((ul - 1) & 1), MAX_POLL)) {
          raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
          ok = false;
        }
        if (ok) {                                    // rows past the tile's heads: unused columns
          tc::mbar_arrive_expect_tx(bfull, (uint32_t)B_BYTES);
          tc::tma_load_2d(sB, &qmap, 0, qt * p.QT * HI, bfull);
          tc::tma_load_2d(sB + B_BYTES / 2, &qmap, 64, qt * p.QT * HI, bfull);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // the page ids of the unit's tiles (at most 64 slots), one load round for the warp:
      // lane l holds slots 2 t0 + l and 2 t0 + 32 + l
      const bool seq_ok = seq >= 0 && seq < p.num_seqs;
      if (!seq_ok && lane == 0) raise_error(&g_err_score, CSA2_DEVERR_SEQ);
      int pgl[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int slot = 2 * t0 + 32 * h + lane;
        int v = 0;
        if (seq_ok && slot < 2 * t1 && slot < p.max_pages) {
          v = __ldg(p.page_table + (long long)seq * p.max_pages + slot);
          if (v < 0 || v >= p.num_pages) {
            raise_error(&g_err_score, CSA2_DEVERR_PAGE_ID);
            v = 0;
          }
        }
        pgl[h] = v;
      }
      for (int t = t0; t < t1 && ok; ++t, ++it) {
        const int i2 = 2 * (t - t0);                 // the tile's first slot in the unit (even, < 64)
        const int pg0 = __shfl_sync(0xffffffffu, i2 < 32 ? pgl[0] : pgl[1], i2 & 31);
        const int pg1 = __shfl_sync(0xffffffffu, i2 < 32 ? pgl[0] : pgl[1], (i2 + 1) & 31);
        if (lane == 0) {
          const int s = (int)(it % STAGES);
          if (it >= STAGES && !tc::mbar_wait(&aempty[s], (uint32_t)(((it / STAGES) - 1) & 1), MAX_POLL)) {
            raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
            ok = false;
          } else {
            uint8_t* st = sA + s * A_BYTES;
            tc::mbar_arrive_expect_tx(&afull[s], A_BYTES);
#pragma unroll
            for (int kh = 0; kh < 2; ++kh) {
              tc::tma_load_2d(st + kh * (A_BYTES / 2), &kmap, 64 * kh, pg0 * 64, &afull[s]);
              tc::tma_load_2d(st + kh * (A_BYTES / 2) + A_BYTES / 4, &kmap, 64 * kh, pg1 * 64, &afull[s]);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      it = __shfl_sync(0xffffffffu, it, 0);
      ++ul;
    }
  } else if (warp == 1) {                            // ---- MMA issuer
    const uint32_t idesc = tc::idesc_f16(BM, BN, 1, 0, 0);   // bf16, both K-major
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
            tc::mma_f16_ss(tb + (uint32_t)(p.bufcols * buf), ad, bd, idesc, k16 > 0 ? 1u : 0u);
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
    constexpr int QPC = 32 / HI;                     // queries per 32 columns
    const int q4 = warp & 3;                         // TMEM lane quarter
    float* sW = reinterpret_cast<float*>(smem + B_BYTES + STAGES * A_BYTES + 256) + q4 * BN_MAX;
    int tl = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      int qt, t0, t1, seq;
      unit_span(p, u, qt, t0, t1, seq);
      // the unit's head weights (QT x HI floats), once per unit
      __syncwarp();
      for (int i = lane; i < p.QT * HI; i += 32) sW[i] = __ldg(p.w + (long long)qt * p.QT * HI + i);
      __syncwarp();
      for (int t = t0; t < t1; ++t, ++tl) {
        const int buf = tl & 1;
        ok = tc::mbar_wait_warp(&accf[buf], (uint32_t)((tl >> 1) & 1), MAX_POLL);
        if (!ok) {
          if (lane == 0) raise_error(&g_err_score, CSA2_DEVERR_TIMEOUT);
          break;
        }
        tc::fence_after_sync();
        const int e = t * BM + 32 * q4 + lane;       // this thread's entry
        const uint32_t tq = tb + ((uint32_t)(32 * q4) << 16) + (uint32_t)(p.bufcols * buf);
#pragma unroll 1
        for (int qc = 0; qc * QPC < p.QT; ++qc) {    // QPC queries (32 columns) at a time
          uint32_t r[32];
          tc::tmem_ld32(tq + (uint32_t)(32 * qc), r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < QPC; ++k) {
            const int qi = qc * QPC + k;
            if (qi >= p.QT) break;
            const int b = qt * p.QT + qi;
            const float4* wp = reinterpret_cast<const float4*>(sW + qi * HI);
            float sc = 0.f;
#pragma unroll
            for (int h4 = 0; h4 < HI / 4; ++h4) {
              const float4 w4 = wp[h4];
              const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float x = __uint_as_float(r[HI * k + 4 * h4 + j]);
                if (p.relu) x = fmaxf(x, 0.f);
                sc = fmaf(wv[j], x, sc);
              }
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
  if (warp == 1) tc::tmem_dealloc(tb, tcols);
}

// Best per_block entries of every block of every query from the score matrix.  A warp takes
// 32 consecutive blocks of one query: it copies their scores (at most 64 per block) into
// shared memory with coalesced loads, then lane i keeps the best of block i in ascending entry
// order, at the offsets of the scan kernels.  "Best" = larger score, then lower entry.  The 32
// blocks' kept entries form one contiguous run of the pool (P per block, or every entry when
// the query has fewer than P x NB), so they are staged in shared memory and written with
// coalesced stores (per-lane stores of P consecutive words made the kernel twice as slow).
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
  float* w = bt_sh + warp * (wfloats + 64 * P);
  int* oid = reinterpret_cast<int*>(w + wfloats);      // the warp's kept entries, then scores
  float* osc = w + wfloats + 32 * P;
  // the warp's slice in 16-byte loads, four in flight a lane (a score row starts 16-byte
  // aligned and is a whole number of 128-entry tiles long, so a load that starts below e1
  // stays inside the row)
  for (int e = (e0 & ~3) + 4 * lane; e < e1; e += 512) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = (e + 128 * u < e1) ? __ldg(reinterpret_cast<const float4*>(s + e + 128 * u)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int eu = e + 128 * u;
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (eu + c >= e0 && eu + c < e1) w[bt_pad(eu + c - e0)] = x[c];
    }
  }
  __syncwarp();
  // the P best values, descending: each score bubbles down the sorted list (a later
  // entry never displaces an equal earlier one, so this is the best-first order of the
  // tie rule "larger score, then lower entry"); lanes past NB have no entries
  float kv[P];
#pragma unroll
  for (int i = 0; i < P; ++i) kv[i] = -INFINITY;
  const int cnt = j < NB ? hi - lo : 0;
  for (int e = lo; e < lo + cnt; ++e) {
    float v = w[bt_pad(e - e0)];
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const float t = fmaxf(v, kv[i]);
      v = fminf(v, kv[i]);
      kv[i] = t;
    }
  }
  // kept: every entry above the P-th best tv, then entries equal to tv in ascending order
  // up to P in all; a block of fewer than P entries keeps them all
  const float tv = (cnt >= P) ? kv[P - 1] : -INFINITY;
  int quota = P;
#pragma unroll
  for (int i = 0; i < P; ++i) quota -= (kv[i] > tv) ? 1 : 0;
  const long long off = ((long long)n >= (long long)P * NB) ? (long long)P * j : lo;
  const long long off0 = __shfl_sync(0xffffffffu, off, 0);   // lane 0's block is below NB
  const int loc = (int)(off - off0);
  int c = 0;
  for (int e = lo; e < lo + cnt; ++e) {               // ascending entries that are kept
    const float v = w[bt_pad(e - e0)];
    if (v > tv || (v == tv && quota-- > 0)) {
      oid[loc + c] = e;
      osc[loc + c] = v;
      ++c;
    }
  }
  const int total = __reduce_max_sync(0xffffffffu, cnt > 0 ? loc + c : 0);
  __syncwarp();
  const long long o = (long long)b * NB * P + off0;
  for (int i = lane; i < total; i += 32) {
    pool[o + i] = oid[i];
    pool_score[o + i] = osc[i];
  }
}

// The same selection for blocks of more than 64 entries (long contexts): one warp per block.
// Each lane keeps the best P values of its strided share (a sorted list, as above); P
// rounds of a warp maximum over the lists' heads give the P-th best value tv of the block;
// one more ascending pass over the block keeps every entry above tv and then the first
// entries equal to tv, up to P in all, each lane placing its kept entry by a ballot count.
constexpr int BTW_WARPS = 8;
template <int P>
__global__ void __launch_bounds__(BTW_WARPS * 32) k_block_topp_w(const float* __restrict__ S, int ldS,
                                                                const int* __restrict__ n_vis, int max_n, int B,
                                                                int NB, int* __restrict__ pool,
                                                                float* __restrict__ pool_score) {
  pdl_wait();
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * BTW_WARPS + (threadIdx.x >> 5);
  if (gw >= (long long)B * NB) return;
  const int b = (int)(gw / NB), j = (int)(gw % NB);
  const int n = max(0, min(__ldg(n_vis + b), max_n));
  const int lo = (int)(((long long)j * n) / NB), hi = (int)(((long long)(j + 1) * n) / NB);
  const int cnt = hi - lo;
  if (cnt <= 0) return;
  const float* s = S + (long long)b * ldS;
  float tv = -INFINITY;
  if (cnt > P) {
    float kv[P];
#pragma unroll
    for (int i = 0; i < P; ++i) kv[i] = -INFINITY;
    for (int e = lo + lane; e < hi; e += 32) {
      float v = __ldg(s + e);
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const float t = fmaxf(v, kv[i]);
        v = fminf(v, kv[i]);
        kv[i] = t;
      }
    }
    int taken = 0;
#pragma unroll 1
    for (int r = 0; r < P; ++r) {                    // pop the warp maximum, with multiplicity
      float m = kv[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
      const bool hold = kv[0] == m;
      taken += __popc(__ballot_sync(FULL, hold));
      if (taken >= P) {
        tv = m;
        break;
      }
      if (hold) {
#pragma unroll
        for (int i = 0; i < P - 1; ++i) kv[i] = kv[i + 1];
        kv[P - 1] = -INFINITY;
      }
    }
  }
  // kept: every entry above tv, then the first entries equal to tv, P in all (a block of at
  // most P entries keeps them all)
  int above = 0;
  for (int e0 = lo; e0 < hi; e0 += 32) {
    const int e = e0 + lane;
    const float v = e < hi ? __ldg(s + e) : -INFINITY;
    above += __popc(__ballot_sync(FULL, e < hi && v > tv));
  }
  const int quota = (cnt > P) ? P - above : cnt;
  const long long off = ((long long)n >= (long long)P * NB) ? (long long)P * j : lo;
  float* ps = pool_score + (long long)b * NB * P + off;
  int* pp = pool + (long long)b * NB * P + off;
  const unsigned below = (1u << lane) - 1u;
  int eq_before = 0, kept = 0;
  for (int e0 = lo; e0 < hi && kept < P; e0 += 32) {
    const int e = e0 + lane;
    const float v = e < hi ? __ldg(s + e) : -INFINITY;
    const bool in = e < hi;
    const bool eq = in && v == tv && cnt > P;
    const unsigned eqm = __ballot_sync(FULL, eq);
    const bool keep = in && (cnt <= P || v > tv || (eq && eq_before + __popc(eqm & below) < quota));
    const unsigned km = __ballot_sync(FULL, keep);
    if (keep) {
      const int o = kept + __popc(km & below);
      pp[o] = e;
      ps[o] = v;
    }
    kept += __popc(km);
    eq_before += __popc(eqm);
  }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
// Queries per tile: the call's group (its queries share a sequence) when its heads fit the
// 256 columns, else the largest tile that does and divides the group; 0 = not supported.
static int tc_query_tile(const csa2_index_full_args& a) {
  if (a.H_i != 8 && a.H_i != 16 && a.H_i != 32) return 0;
  const int G = a.group > 1 ? a.group : 1;
  const int qmax = stc::BN_MAX / a.H_i;
  if (G <= qmax) return G;
  return (G % qmax == 0) ? qmax : 0;
}

bool full_scores_tc_supported(const csa2_index_full_args& a) {
  const int QT = tc_query_tile(a);
  return QT > 0 && a.B % QT == 0 && a.cache.idx_k_dtype == CSA2_BF16 && a.cache.d_ik == stc::DK &&
         a.per_block >= 1 && a.per_block <= 16 &&
         a.max_n > 0 && ((uintptr_t)a.q_idx & 15) == 0 && ((uintptr_t)a.cache.idx_k & 15) == 0 &&
         ((uintptr_t)a.w & 15) == 0 && tensor_map_encoder() != nullptr;
}

size_t full_scores_tc_bytes(const csa2_index_full_args& a) {
  const long long ld = ((long long)a.max_n + stc::BM - 1) / stc::BM * stc::BM;
  return (size_t)a.B * ld * sizeof(float);
}

template <int HI>
static cudaError_t launch_score(const CUtensorMap& kmap, const CUtensorMap& qmap, const ScoreParams& p, int smem,
                                int sms, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_score_tc<HI>, cudaFuncAttributeMaxDynamicSharedMemorySize, stc::SMEM_MAX);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = std::max(1, std::min(p.units, sms));
  // persistent (one CTA per SM): started only once the previous kernel has completed
  return launch_k_late(k_score_tc<HI>, grid, stc::THREADS, smem, st, kmap, qmap, p);
}

cudaError_t launch_full_scores_tc(const csa2_index_full_args& a, float* S, float* pool_score, cudaStream_t st) {
  using namespace stc;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  sms = sms > 0 ? sms : 1;
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
  p.QT = tc_query_tile(a);
  p.BN = (p.QT * a.H_i + 15) / 16 * 16;
  p.bufcols = 32;
  while (p.bufcols < p.BN) p.bufcols *= 2;
  // entry tiles per unit: about 8 units per CTA, 4..32 tiles each
  const long long tiles = (long long)(a.B / p.QT) * p.ntiles;
  p.chunk = (int)std::max(4LL, std::min(32LL, tiles / (8LL * sms)));
  p.nchunks = (p.ntiles + p.chunk - 1) / p.chunk;
  p.units = (a.B / p.QT) * p.nchunks;
  p.S = S;
  const int smem = p.BN * DK * 2 + STAGES * A_BYTES + 256 + W_BYTES;
  CUtensorMap kmap, qmap;                            // idx_k rows (64-row boxes: one page), Q rows (BN)
  if (!bf16_map(&kmap, a.cache.idx_k, (long long)a.cache.num_pages * 64, DK, 64) ||
      !bf16_map(&qmap, a.q_idx, (long long)a.B * a.H_i, DK, p.BN))
    return cudaErrorInvalidValue;
  cudaError_t e = a.H_i == 8    ? launch_score<8>(kmap, qmap, p, smem, sms, st)
                  : a.H_i == 16 ? launch_score<16>(kmap, qmap, p, smem, sms, st)
                                : launch_score<32>(kmap, qmap, p, smem, sms, st);
  if (e != cudaSuccess) return e;
  // entries per block at most: ceil(max_n / NB)
  const int per_blk = (int)(((long long)a.max_n + a.num_blocks - 1) / a.num_blocks);
  if (per_blk <= 64) {                               // a lane per block
    const long long warps = (long long)a.B * ((a.num_blocks + 31) / 32);
    const unsigned grid2 = (unsigned)((warps + BT_WARPS - 1) / BT_WARPS);
    const int wfloats = bt_warp_floats(per_blk);
    const size_t smem2 = (size_t)BT_WARPS * (wfloats + 64 * a.per_block) * sizeof(float);
    switch (a.per_block) {                           // the kept list lives in registers
#define CSA2_BT(PP) \
  case PP: return launch_k(k_block_topp<PP>, grid2, BT_WARPS * 32, smem2, st, S, p.ldS, a.n_vis, a.max_n, a.B, \
                           a.num_blocks, wfloats, a.pool, pool_score);
      CSA2_BT(1) CSA2_BT(2) CSA2_BT(3) CSA2_BT(4) CSA2_BT(5) CSA2_BT(6) CSA2_BT(7) CSA2_BT(8)
      CSA2_BT(9) CSA2_BT(10) CSA2_BT(11) CSA2_BT(12) CSA2_BT(13) CSA2_BT(14) CSA2_BT(15) CSA2_BT(16)
#undef CSA2_BT
      default: return cudaErrorInvalidValue;
    }
  }
  const long long warps = (long long)a.B * a.num_blocks;   // a warp per block
  const unsigned grid2 = (unsigned)((warps + BTW_WARPS - 1) / BTW_WARPS);
  switch (a.per_block) {
#define CSA2_BTW(PP) \
  case PP: return launch_k(k_block_topp_w<PP>, grid2, BTW_WARPS * 32, 0, st, S, p.ldS, a.n_vis, a.max_n, a.B, \
                           a.num_blocks, a.pool, pool_score);
    CSA2_BTW(1) CSA2_BTW(2) CSA2_BTW(3) CSA2_BTW(4) CSA2_BTW(5) CSA2_BTW(6) CSA2_BTW(7) CSA2_BTW(8)
    CSA2_BTW(9) CSA2_BTW(10) CSA2_BTW(11) CSA2_BTW(12) CSA2_BTW(13) CSA2_BTW(14) CSA2_BTW(15) CSA2_BTW(16)
#undef CSA2_BTW
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
