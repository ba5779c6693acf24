// Hierarchical sparse indexer: Full scan with per-block top-P (the shared candidate
// pool), Reindex re-scoring of the pool, and the exact Top-k selection.
//
// "DeepSeek-V4.1-Flash deep dive", section 3.1: Indexer Q x Indexer K -> score -> Top-K.
// Section 3.3: the first Full indexer scans the whole causally visible range and keeps
// the best positions of every block (2,048 blocks x 8 = a 16,384-entry shared pool);
// Reindex layers score only the pool; the search range stays 16,384.
//
// Scoring runs on the tensor cores with mma.sync m16n8k16 (bf16 in, fp32 accumulate):
// M = 16 cache rows, N = 8 indexer heads, K = 16 dims.  Each thread loads its own
// 16-byte slices of a row straight from HBM into registers (no shared-memory staging):
// the contraction over dims is invariant under any permutation applied to both
// operands, so the k-slots of the fragment are mapped to the dims each thread loads
// contiguously (32j + 8c + [0, 8) for lane c of a row quad).  The indexer Q of the query
// is loaded with the same mapping once per warp.
#include <algorithm>
#include <mutex>

#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace csa2 {

CSA2_DEFINE_ERROR_WORD(g_err_index);

constexpr unsigned FULL_MASK = 0xffffffffu;

// A thread's slices of one indexer-K row: bf16 (uint4 j = dims 32j + 8c + [0, 8) of lane c of a
// row quad) or, in the FP8 form, the bytes [DK/4 c, DK/4 (c + 1)) with the row's scale.
template <int DK, bool F8>
struct KRow {
  uint4 v[F8 ? DK / 64 : DK / 32];
  float s;
};

// The query's indexer Q in the same dim mapping (head g of lane (g, c), one head group per
// entry of v) and the head weights of the lane's two accumulator columns.  FP8 form: the Q
// bytes and the weights w_h * sq_h quantised by k_quant_q8.
template <int DK, int NHG, bool F8>
struct QFrag {
  uint4 v[NHG][DK / 32];         // bf16 pairs, or (FP8 form) the E4M3 bytes as f16 pairs: byte
                                 // pair (2i, 2i + 1) of the lane's 4-byte word w in word 2w + i
  float w[NHG][2];
};

template <int DK, int NHG, bool F8>
__device__ __forceinline__ void load_qfrag(const void* __restrict__ qv, const float* __restrict__ w, int H_i,
                                           QFrag<DK, NHG, F8>& f) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int hg = 0; hg < NHG; ++hg) {
    const int head = hg * 8 + g;
    if constexpr (F8) {
      const uint8_t* q = static_cast<const uint8_t*>(qv);
#pragma unroll
      for (int j = 0; j < DK / 64; ++j) {
        const uint4 b = (head < H_i) ? __ldg(reinterpret_cast<const uint4*>(q + head * DK + (DK / 4) * c + 16 * j))
                                     : make_uint4(0, 0, 0, 0);
        f.v[hg][2 * j] = make_uint4(e4m3x2_lo_f16x2(b.x), e4m3x2_hi_f16x2(b.x), e4m3x2_lo_f16x2(b.y),
                                    e4m3x2_hi_f16x2(b.y));
        f.v[hg][2 * j + 1] = make_uint4(e4m3x2_lo_f16x2(b.z), e4m3x2_hi_f16x2(b.z), e4m3x2_lo_f16x2(b.w),
                                        e4m3x2_hi_f16x2(b.w));
      }
    } else {
      const uint16_t* q = static_cast<const uint16_t*>(qv);
#pragma unroll
      for (int j = 0; j < DK / 32; ++j)
        f.v[hg][j] = (head < H_i) ? __ldg(reinterpret_cast<const uint4*>(q + head * DK + 32 * j + 8 * c))
                                  : make_uint4(0, 0, 0, 0);
    }
    const int h0 = hg * 8 + 2 * c;
    f.w[hg][0] = (h0 < H_i) ? __ldg(w + h0) : 0.f;
    f.w[hg][1] = (h0 + 1 < H_i) ? __ldg(w + h0 + 1) : 0.f;
  }
}

// Load the thread's slices of one cache row (zeros when row < 0).  SEQ: rows of a sequential
// run (the scan: the 256-byte L2 prefetch serves the next row too); otherwise scattered rows
// (Reindex), whose FP8 rows are 128 bytes: no prefetch past the row.
// In the FP8 form the row's scale is given (loaded once by the lane that resolved the row);
// a negative `scale` asks for the load here.
template <int DK, bool F8, bool SEQ = true>
__device__ __forceinline__ void load_row(const csa2_cache& cache, long long row, KRow<DK, F8>& a,
                                         float scale = -1.f) {
  const int c = threadIdx.x & 3;
  if constexpr (F8) {
    const uint8_t* p = cache.idx_k8 + row * DK + (DK / 4) * c;
#pragma unroll
    for (int j = 0; j < DK / 64; ++j)
      a.v[j] = (row >= 0) ? (SEQ ? ldg_stream_v4(p + 16 * j) : ldg_gather_v4(p + 16 * j)) : make_uint4(0, 0, 0, 0);
    a.s = (row < 0) ? 0.f : (scale >= 0.f ? scale : __ldg(cache.idx_k8_scale + row));
  } else {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j)
      a.v[j] = (row >= 0) ? ldg_stream_v4(cache.idx_k + row * DK + 32 * j + 8 * c) : make_uint4(0, 0, 0, 0);
    a.s = 1.f;
  }
}

__device__ __forceinline__ uint32_t word_of(const uint4* v, int w) {
  const uint4 x = v[w >> 2];
  return (w & 3) == 0 ? x.x : (w & 3) == 1 ? x.y : (w & 3) == 2 ? x.z : x.w;
}

// Scores of rows (g) and (g + 8) of a 16-row tile; identical in the 4 lanes of a quad.
// bf16: m16n8k16 products over dims.  FP8: the E4M3 bytes converted to f16 pairs (exact) and
// multiplied by m16n8k16 f16 products (exact in float32): the k-slots 2c, 2c + 1 / 8 + 2c,
// 9 + 2c of the product for the lane's row word w take its bytes 0, 1 / 2, 3 (Q's bytes in the
// same places, converted once when the fragment is loaded; the tensor cores here run E4M3
// mma.sync as f16 products anyway, converting both operands at every product), and the row
// scale is applied after the weighted ReLU sum (both scales are >= 0).
template <int DK, int NHG, bool F8>
__device__ __forceinline__ void tile_scores(const QFrag<DK, NHG, F8>& f, const KRow<DK, F8>& A0,
                                            const KRow<DK, F8>& A1, bool relu, float& s0, float& s1) {
  float acc[NHG][4];
#pragma unroll
  for (int hg = 0; hg < NHG; ++hg) acc[hg][0] = acc[hg][1] = acc[hg][2] = acc[hg][3] = 0.f;
  if constexpr (F8) {
    // each row word (4 E4M3 bytes) becomes two f16 pairs, paired with Q's pre-converted pairs
    // of the same bytes: m16n8k16 f16 products (exact, float32 accumulation)
#pragma unroll
    for (int j = 0; j < DK / 32; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t r0 = word_of(A0.v, 2 * j + h), r1 = word_of(A1.v, 2 * j + h);
        const uint32_t a0 = e4m3x2_lo_f16x2(r0), a1 = e4m3x2_lo_f16x2(r1);
        const uint32_t a2 = e4m3x2_hi_f16x2(r0), a3 = e4m3x2_hi_f16x2(r1);
#pragma unroll
        for (int hg = 0; hg < NHG; ++hg)
          mma_f16_16816(acc[hg], a0, a1, a2, a3, word_of(f.v[hg], 2 * (2 * j + h)),
                        word_of(f.v[hg], 2 * (2 * j + h) + 1));
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < DK / 32; ++j) {
#pragma unroll
      for (int hg = 0; hg < NHG; ++hg) {
        mma_bf16_16816(acc[hg], A0.v[j].x, A1.v[j].x, A0.v[j].y, A1.v[j].y, f.v[hg][j].x, f.v[hg][j].y);
        mma_bf16_16816(acc[hg], A0.v[j].z, A1.v[j].z, A0.v[j].w, A1.v[j].w, f.v[hg][j].z, f.v[hg][j].w);
      }
    }
  }
  float p0 = 0.f, p1 = 0.f;
#pragma unroll
  for (int hg = 0; hg < NHG; ++hg) {
    float a0 = acc[hg][0], a1 = acc[hg][1], a2 = acc[hg][2], a3 = acc[hg][3];
    if (relu) { a0 = fmaxf(a0, 0.f); a1 = fmaxf(a1, 0.f); a2 = fmaxf(a2, 0.f); a3 = fmaxf(a3, 0.f); }
    p0 = fmaf(f.w[hg][0], a0, p0);
    p0 = fmaf(f.w[hg][1], a1, p0);
    p1 = fmaf(f.w[hg][0], a2, p1);
    p1 = fmaf(f.w[hg][1], a3, p1);
  }
  p0 += __shfl_xor_sync(FULL_MASK, p0, 1);
  p1 += __shfl_xor_sync(FULL_MASK, p1, 1);
  p0 += __shfl_xor_sync(FULL_MASK, p0, 2);
  p1 += __shfl_xor_sync(FULL_MASK, p1, 2);
  if constexpr (F8) {
    p0 *= A0.s;
    p1 *= A1.s;
  }
  s0 = p0;
  s1 = p1;
}

// The FP8 form's indexer Q: each (query, head) row of q_idx (bf16) quantised as the
// compressed indexer K is (s = amax / 448, E4M3 bytes; zero row -> zero bytes), into q8,
// and the head weight times that scale into w8.  One warp per row.
template <int DK>
__global__ void __launch_bounds__(256) k_quant_q8(const uint16_t* __restrict__ q, const float* __restrict__ w, int rows,
                                                  uint8_t* __restrict__ q8, float* __restrict__ w8) {
  pdl_wait();
  pdl_trigger();
  constexpr int N = DK / 32;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  float v[N];
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] = bf16_bits_to_f32(__ldg(q + (long long)r * DK + lane * N + j));
  float sq;
  const float s = fp8_row_store<N>(v, q8 + (long long)r * DK + lane * N, &sq);
  if (lane == 0) w8[r] = __ldg(w + r) * s;
}

__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// ---------------------------------------------------------------------------------
// Full scan: one warp per pool block.  The warp keeps the block's best P entries in
// lanes 0..P-1 (sorted best first) and inserts candidates that beat the P-th.
// ---------------------------------------------------------------------------------
struct ScanParams {
  const uint16_t* q;      // [B][H_i][DK]
  const float* w;         // [B][H_i]
  const uint8_t* q8;      // FP8 form: [B][H_i][DK] quantised indexer Q (workspace)
  const float* w8;        // FP8 form: [B][H_i] weights times the Q scales (workspace)
  csa2_cache cache;
  const int* seq_of;
  const int* n_vis;
  int max_n;
  int H_i, NB, P;
  int relu;
  int* pool;              // [B][NB*P]
  float* pool_score;      // [B][NB*P]
  int B;
};

// Offer the warp's 32 candidates (cv, ci: one per lane) to a block's best-P list (tv, ti in
// lanes 0..P-1, best first; thv, thi: its P-th entry in every lane).
__device__ __forceinline__ void topp_offer(float cv, int ci, int P, float& tv, int& ti, float& thv, int& thi) {
  const int lane = threadIdx.x & 31;
  const unsigned m = __ballot_sync(FULL_MASK, better(cv, ci, thv, thi));
  if (m == 0) return;
  if (__popc(m) <= 3 || P > 16) {
    // few candidates (or a long list): insert them one by one
    unsigned mm = m;
    while (mm) {
      const int src = __ffs(mm) - 1;
      mm &= mm - 1;
      const float xv = __shfl_sync(FULL_MASK, cv, src);
      const int xi = __shfl_sync(FULL_MASK, ci, src);
      const unsigned bm = __ballot_sync(FULL_MASK, lane < P && better(xv, xi, tv, ti));
      if (bm) {
        const int at = __ffs(bm) - 1;
        const float upv = __shfl_up_sync(FULL_MASK, tv, 1);
        const int upi = __shfl_up_sync(FULL_MASK, ti, 1);
        if (lane > at && lane < P) { tv = upv; ti = upi; }
        if (lane == at) { tv = xv; ti = xi; }
      }
    }
  } else {
    // many candidates: bitonic sort of the 32 (best first), then a bitonic merge of
    // the best Pp of them with the list (Pp = P rounded up to a power of two <= 16)
#pragma unroll
    for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        const float ov = __shfl_xor_sync(FULL_MASK, cv, jj);
        const int oi = __shfl_xor_sync(FULL_MASK, ci, jj);
        const bool want_better = (((lane & jj) == 0) == ((lane & kk) == 0));
        const bool ob = better(ov, oi, cv, ci);
        if (want_better == ob) { cv = ov; ci = oi; }
      }
    }
    int Pp = 1;
    while (Pp < P) Pp <<= 1;
    const float nv = __shfl_sync(FULL_MASK, cv, (2 * Pp - 1 - lane) & 31);
    const int ni = __shfl_sync(FULL_MASK, ci, (2 * Pp - 1 - lane) & 31);
    float mv = (lane < Pp) ? tv : nv;
    int mi = (lane < Pp) ? ti : ni;
    for (int jj = Pp; jj > 0; jj >>= 1) {
      const float ov = __shfl_xor_sync(FULL_MASK, mv, jj);
      const int oi = __shfl_xor_sync(FULL_MASK, mi, jj);
      const bool want_better = (lane & jj) == 0;
      const bool ob = better(ov, oi, mv, mi);
      if (want_better == ob) { mv = ov; mi = oi; }
    }
    if (lane < P) { tv = mv; ti = mi; }
  }
  thv = __shfl_sync(FULL_MASK, tv, P - 1);
  thi = __shfl_sync(FULL_MASK, ti, P - 1);
}

// Write a block's kept entries (the list of lanes 0..kept-1) to the pool, ascending by entry.
__device__ __forceinline__ void topp_write(const ScanParams& p, int b, int j, int n, long long lo, long long hi,
                                           float tv, int ti) {
  const int lane = threadIdx.x & 31, P = p.P;
  const int kept = (int)((hi - lo) < (long long)P ? (hi - lo) : (long long)P);
  int rank = 0;
  for (int l = 0; l < P; ++l) {
    int oi = __shfl_sync(FULL_MASK, ti, l);
    rank += (l < kept && oi < ti) ? 1 : 0;
  }
  const long long off = ((long long)n >= (long long)P * p.NB) ? (long long)P * j : lo;
  if (lane < kept) {
    long long o = (long long)b * p.NB * P + off + rank;
    p.pool[o] = ti;
    p.pool_score[o] = tv;
  }
}

template <int DK, int NHG, bool F8>
__global__ void __launch_bounds__(256, 2) k_full_scan(ScanParams p) {
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  // persistent: warp w of CTA x takes pool blocks u = 8 x + w, + 8 gridDim.x, ... of all
  // queries (u = b NB + j)
  const long long total = (long long)p.B * p.NB;
  for (long long u = (long long)blockIdx.x * 8 + warp; u < total; u += (long long)gridDim.x * 8) {
  const int b = (int)(u / p.NB);
  const int j = (int)(u % p.NB);
  int n = __ldg(p.n_vis + b);
  if (n < 0 || n > p.max_n) {
    if (lane == 0 && j == 0) raise_error(&g_err_index, CSA2_DEVERR_N_VIS);
    n = max(0, min(n, p.max_n));
  }
  const int s = __ldg(p.seq_of + b);
  const long long lo = ((long long)j * n) / p.NB;
  const long long hi = ((long long)(j + 1) * n) / p.NB;
  const int P = p.P;

  // up to two head groups keep their Q fragments in registers; more are streamed from L1
  // one group at a time (registers for two resident CTAs per SM)
  constexpr bool STREAM_Q = NHG > 2;
  constexpr int NHG_REG = STREAM_Q ? 1 : NHG;
  constexpr int QB = F8 ? 1 : 2;                 // bytes per indexer-Q element
  const uint8_t* qb = reinterpret_cast<const uint8_t*>(F8 ? (const void*)p.q8 : (const void*)p.q) +
                      (long long)b * p.H_i * DK * QB;
  const float* wb = (F8 ? p.w8 : p.w) + (long long)b * p.H_i;
  QFrag<DK, NHG_REG, F8> f;
  if (!STREAM_Q) load_qfrag<DK, NHG_REG, F8>(qb, wb, p.H_i, f);

  float tv = -INFINITY;
  int ti = 0x7fffffff;
  float thv = -INFINITY;
  int thi = 0x7fffffff;

  // rows of TPI tiles of 32 are loaded per iteration: the FP8 form's rows are half the
  // bytes, so it takes two tiles to keep as many bytes in flight as the bf16 form
  constexpr int TPI = F8 ? 2 : 1;
  constexpr int ROWB = F8 ? DK : 2 * DK;          // bytes of one indexer-K row
  for (long long base = lo; base < hi; base += 32 * TPI) {
    // FP8 form: the next iteration's rows (their run within one page, up to the block's end)
    // are requested into L2 now, so that their DRAM reads overlap this iteration's loads and
    // products (1.64 -> 1.61 ms at 1M x 64).  The bf16 form measured slower with it (2.45 ->
    // 2.63 ms): its register loads already keep the DRAM busy.
    if (F8 && lane == 0 && base + 32 * TPI < hi) {
      const long long nb = base + 32 * TPI;
      const long long nrow = entry_row(p.cache, s, nb, &g_err_index);
      if (nrow >= 0) {
        long long rows = kPage - (nb & (kPage - 1));
        rows = rows < 32 * TPI ? rows : 32 * TPI;
        rows = rows < hi - nb ? rows : hi - nb;
        const uint8_t* src = F8 ? p.cache.idx_k8 : reinterpret_cast<const uint8_t*>(p.cache.idx_k);
        prefetch_l2_bulk(src + nrow * ROWB, (uint32_t)(rows * ROWB));
      }
    }
    long long r[TPI][4];
    KRow<DK, F8> A[TPI][4];
    // lane (g, c) resolves row 8c + g of each tile through the page table; the four lanes of
    // a quad then share their rows (each row is loaded in slices by a whole quad)
    int mine[TPI];
    float msc[TPI];                                // FP8 form: the resolved row's scale
#pragma unroll
    for (int tt = 0; tt < TPI; ++tt) {
      const long long rr = base + 32 * tt + 8 * c + g;
      mine[tt] = (rr < hi) ? (int)entry_row(p.cache, s, rr, &g_err_index) : -1;
      msc[tt] = (F8 && mine[tt] >= 0) ? __ldg(p.cache.idx_k8_scale + mine[tt]) : 0.f;
    }
#pragma unroll
    for (int tt = 0; tt < TPI; ++tt)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        r[tt][t] = base + 32 * tt + 8 * t + g;
        const int src = (lane & ~3) | t;
        const int row = __shfl_sync(FULL_MASK, mine[tt], src);
        load_row<DK, F8>(p.cache, row, A[tt][t], F8 ? __shfl_sync(FULL_MASK, msc[tt], src) : -1.f);
      }
#pragma unroll
    for (int tt = 0; tt < TPI; ++tt) {
      float sc[4];
      if (STREAM_Q) {
        sc[0] = sc[1] = sc[2] = sc[3] = 0.f;
#pragma unroll 1
        for (int hg = 0; hg < NHG; ++hg) {
          load_qfrag<DK, NHG_REG, F8>(qb + hg * 8 * DK * QB, wb + hg * 8, p.H_i - hg * 8, f);
          float x0, x1, x2, x3;
          tile_scores<DK, NHG_REG, F8>(f, A[tt][0], A[tt][1], p.relu != 0, x0, x1);
          tile_scores<DK, NHG_REG, F8>(f, A[tt][2], A[tt][3], p.relu != 0, x2, x3);
          sc[0] += x0;
          sc[1] += x1;
          sc[2] += x2;
          sc[3] += x3;
        }
      } else {
        tile_scores<DK, NHG_REG, F8>(f, A[tt][0], A[tt][1], p.relu != 0, sc[0], sc[1]);
        tile_scores<DK, NHG_REG, F8>(f, A[tt][2], A[tt][3], p.relu != 0, sc[2], sc[3]);
      }
      // lane (g, c) owns candidate row r[c] = base + g + 8c (a permutation of the 32 rows)
      float cv = sc[0];
      int ci = (int)r[tt][0];
#pragma unroll
      for (int t = 1; t < 4; ++t)
        if (c == t) { cv = sc[t]; ci = (int)r[tt][t]; }
      if ((long long)ci >= hi) { cv = -INFINITY; ci = 0x7fffffff; }
      topp_offer(cv, ci, P, tv, ti, thv, thi);
    }
  }
  topp_write(p, b, j, n, lo, hi, tv, ti);
  }
}

// Full scan of short blocks (at most 64 entries each, e.g. N = 131,072 over 2,048 blocks) with
// one head group and P = 8: a warp scores the rows of SEG consecutive blocks of one query into
// shared memory, then lane j < SEG keeps block j's best P by a min/max bubble down a sorted list
// of values (the selection of k_block_topp).  k_full_scan keeps each block's list warp-wide and
// offers it every 32-row tile, which costs a 32-wide sort whenever most of a tile beats the
// list -- always, for a block of two tiles.  Same pool, pool scores and order as k_full_scan.
// Used for the FP8 form, whose scan is bound by instruction issue (N = 131,072 x 32 queries:
// 167 -> 129 us a call).  The bf16 form, bound by bytes, keeps k_full_scan: with SEG = 32 or 4
// it measured 212 and 216 us against 203 (whole segments balance the persistent warps' shares
// worse than single blocks).
constexpr int SS_P = 8;                                   // per_block of this path
constexpr int SS_MAXB = 64;                               // entries per block at most
__host__ __device__ constexpr int ss_wfloats(int seg) { return seg * SS_MAXB + SS_MAXB; }   // a pad word per 32
__host__ __device__ constexpr int ss_warp_words(int seg) { return ss_wfloats(seg) + 2 * seg * SS_P; }
__host__ __device__ constexpr size_t ss_smem(int seg) { return (size_t)8 * ss_warp_words(seg) * sizeof(float); }

__device__ __forceinline__ int ss_pad(int i) { return i + (i >> 5); }

template <int DK, bool F8, int SEG>
__global__ void __launch_bounds__(256, 2) k_full_scan_short(ScanParams p) {
  pdl_wait();
  extern __shared__ float ss_sh[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  float* wsc = ss_sh + warp * ss_warp_words(SEG);
  int* oid = reinterpret_cast<int*>(wsc + ss_wfloats(SEG));
  float* osc = wsc + ss_wfloats(SEG) + SEG * SS_P;
  constexpr int QB = F8 ? 1 : 2;                 // bytes per indexer-Q element
  constexpr int TPI = F8 ? 2 : 1;                // 32-row tiles per iteration, as in k_full_scan
  constexpr int ROWB = F8 ? DK : 2 * DK;
  const int segs = (p.NB + SEG - 1) / SEG;
  const long long total = (long long)p.B * segs;
  QFrag<DK, 1, F8> f;
  int fb = -1;                                   // the query whose fragment f holds
  // persistent: warp w of CTA x takes units u = 8 x + w, + 8 gridDim.x, ... (u = b segs + seg)
  for (long long u = (long long)blockIdx.x * 8 + warp; u < total; u += (long long)gridDim.x * 8) {
    const int b = (int)(u / segs), j0 = (int)(u % segs) * SEG;
    int n = __ldg(p.n_vis + b);
    if (n < 0 || n > p.max_n) {
      if (lane == 0 && j0 == 0) raise_error(&g_err_index, CSA2_DEVERR_N_VIS);
      n = max(0, min(n, p.max_n));
    }
    const int s = __ldg(p.seq_of + b);
    if (b != fb) {
      const uint8_t* qb = reinterpret_cast<const uint8_t*>(F8 ? (const void*)p.q8 : (const void*)p.q) +
                          (long long)b * p.H_i * DK * QB;
      load_qfrag<DK, 1, F8>(qb, (F8 ? p.w8 : p.w) + (long long)b * p.H_i, p.H_i, f);
      fb = b;
    }
    // lane j < SEG: block j0 + j = [lo, hi) (the other lanes: empty); the warp's rows [e0, e1)
    const int j = j0 + min(lane, SEG);
    const long long lo = ((long long)min(j, p.NB) * n) / p.NB;
    const long long hi = ((long long)min(j0 + min(lane + 1, SEG), p.NB) * n) / p.NB;
    const long long e0 = __shfl_sync(FULL_MASK, lo, 0);
    const long long e1 = ((long long)min(j0 + SEG, p.NB) * n) / p.NB;
    for (long long base = e0; base < e1; base += 32 * TPI) {
      if (F8 && lane == 0 && base + 32 * TPI < e1) {       // the next iteration's rows into L2
        const long long nb = base + 32 * TPI;
        const long long nrow = entry_row(p.cache, s, nb, &g_err_index);
        if (nrow >= 0) {
          long long rows = kPage - (nb & (kPage - 1));
          rows = rows < 32 * TPI ? rows : 32 * TPI;
          rows = rows < e1 - nb ? rows : e1 - nb;
          const uint8_t* src = F8 ? p.cache.idx_k8 : reinterpret_cast<const uint8_t*>(p.cache.idx_k);
          prefetch_l2_bulk(src + nrow * ROWB, (uint32_t)(rows * ROWB));
        }
      }
      KRow<DK, F8> A[TPI][4];
      int mine[TPI];
      float msc[TPI];
#pragma unroll
      for (int tt = 0; tt < TPI; ++tt) {
        const long long rr = base + 32 * tt + 8 * c + g;
        mine[tt] = (rr < e1) ? (int)entry_row(p.cache, s, rr, &g_err_index) : -1;
        msc[tt] = (F8 && mine[tt] >= 0) ? __ldg(p.cache.idx_k8_scale + mine[tt]) : 0.f;
      }
#pragma unroll
      for (int tt = 0; tt < TPI; ++tt)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int src = (lane & ~3) | t;
          load_row<DK, F8>(p.cache, __shfl_sync(FULL_MASK, mine[tt], src), A[tt][t],
                           F8 ? __shfl_sync(FULL_MASK, msc[tt], src) : -1.f);
        }
#pragma unroll
      for (int tt = 0; tt < TPI; ++tt) {
        float sc[4];
        tile_scores<DK, 1, F8>(f, A[tt][0], A[tt][1], p.relu != 0, sc[0], sc[1]);
        tile_scores<DK, 1, F8>(f, A[tt][2], A[tt][3], p.relu != 0, sc[2], sc[3]);
        if (c == 0) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const long long r = base + 32 * tt + 8 * t + g;
            if (r < e1) wsc[ss_pad((int)(r - e0))] = sc[t];
          }
        }
      }
    }
    __syncwarp();
    // lane j keeps its block's best P: every entry above the P-th best value tv, then the first
    // entries equal to it in ascending order (all of a block of fewer than P entries)
    const int cnt = (lane < SEG && j < p.NB) ? (int)(hi - lo) : 0;
    const int b0 = (int)(lo - e0);
    float kv[SS_P];
#pragma unroll
    for (int i = 0; i < SS_P; ++i) kv[i] = -INFINITY;
    for (int e = 0; e < cnt; ++e) {
      float v = wsc[ss_pad(b0 + e)];
#pragma unroll
      for (int i = 0; i < SS_P; ++i) {
        const float t = fmaxf(v, kv[i]);
        v = fminf(v, kv[i]);
        kv[i] = t;
      }
    }
    const float tv = (cnt >= SS_P) ? kv[SS_P - 1] : -INFINITY;
    int quota = SS_P;
#pragma unroll
    for (int i = 0; i < SS_P; ++i) quota -= (kv[i] > tv) ? 1 : 0;
    // the SEG blocks' kept entries are one contiguous run of the pool: staged, then stored
    const long long off = ((long long)n >= (long long)SS_P * p.NB) ? (long long)SS_P * j : lo;
    const long long off0 = __shfl_sync(FULL_MASK, off, 0);
    const int loc = (int)(off - off0);
    int kept = 0;
    for (int e = 0; e < cnt; ++e) {
      const float v = wsc[ss_pad(b0 + e)];
      if (v > tv || (v == tv && quota-- > 0)) {
        oid[loc + kept] = (int)(lo + e);
        osc[loc + kept] = v;
        ++kept;
      }
    }
    const int tot = __reduce_max_sync(FULL_MASK, cnt > 0 ? loc + kept : 0);
    __syncwarp();
    const long long o = (long long)b * p.NB * SS_P + off0;
    for (int i = lane; i < tot; i += 32) {
      p.pool[o + i] = oid[i];
      p.pool_score[o + i] = osc[i];
    }
    __syncwarp();                                 // before the next unit reuses the buffers
  }
}

// Full scan of G queries of one sequence at once (G consecutive queries sharing seq_of, e.g.
// the positions of a speculative-decoding verification step): each indexer-K row is read
// once and scored against every query (H_i <= 8).  Query q keeps its own blocks of its own
// n_vis: the warp of block j reads rows [min_q lo_q, max_q hi_q) and offers each query only
// its rows, so every query's pool and scores equal those of scanning it alone.
template <int DK, int G, bool F8>
__global__ void __launch_bounds__(256, 2) k_full_scan_g(ScanParams p) {
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const long long total = (long long)(p.B / G) * p.NB;
  for (long long u = (long long)blockIdx.x * 8 + warp; u < total; u += (long long)gridDim.x * 8) {
    const int grp = (int)(u / p.NB), j = (int)(u % p.NB);
    const int b0 = grp * G;
    const int s = __ldg(p.seq_of + b0);
    int n[G], lo[G], hi[G];
    int rlo = 0x7fffffff, rhi = 0;
#pragma unroll
    for (int q = 0; q < G; ++q) {
      int nq = __ldg(p.n_vis + b0 + q);
      if (nq < 0 || nq > p.max_n) {
        if (lane == 0 && j == 0) raise_error(&g_err_index, CSA2_DEVERR_N_VIS);
        nq = max(0, min(nq, p.max_n));
      }
      if (q > 0 && __ldg(p.seq_of + b0 + q) != s && lane == 0 && j == 0) raise_error(&g_err_index, CSA2_DEVERR_SEQ);
      n[q] = nq;
      lo[q] = (int)(((long long)j * nq) / p.NB);
      hi[q] = (int)(((long long)(j + 1) * nq) / p.NB);
      if (lo[q] < hi[q]) {
        rlo = min(rlo, lo[q]);
        rhi = max(rhi, hi[q]);
      }
    }
    float tv[G], thv[G];
    int ti[G], thi[G];
#pragma unroll
    for (int q = 0; q < G; ++q) {
      tv[q] = -INFINITY;
      ti[q] = 0x7fffffff;
      thv[q] = -INFINITY;
      thi[q] = 0x7fffffff;
    }
    constexpr int TPI = 1;                       // each row is scored G times: compute, not bytes, bounds it
    for (int base0 = rlo; base0 < rhi; base0 += 32 * TPI) {
      int rr[TPI][4];
      KRow<DK, F8> AA[TPI][4];
#pragma unroll
      for (int tt = 0; tt < TPI; ++tt)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          rr[tt][t] = base0 + 32 * tt + 8 * t + g;
          const long long row = (rr[tt][t] < rhi) ? entry_row(p.cache, s, rr[tt][t], &g_err_index) : -1;
          load_row<DK, F8>(p.cache, row, AA[tt][t]);
        }
#pragma unroll
      for (int tt = 0; tt < TPI; ++tt) {
      const int* r = rr[tt];
      const KRow<DK, F8>* A = AA[tt];
      // lane (g, c) owns candidate row base + g + 8c (a permutation of the 32 rows)
      int ci = r[0];
#pragma unroll
      for (int t = 1; t < 4; ++t)
        if (c == t) ci = r[t];
#pragma unroll
      for (int q = 0; q < G; ++q) {
        QFrag<DK, 1, F8> f;
        if constexpr (F8)
          load_qfrag<DK, 1, F8>(p.q8 + (long long)(b0 + q) * p.H_i * DK, p.w8 + (long long)(b0 + q) * p.H_i, p.H_i, f);
        else
          load_qfrag<DK, 1, F8>(p.q + (long long)(b0 + q) * p.H_i * DK, p.w + (long long)(b0 + q) * p.H_i, p.H_i, f);
        float sc[4];
        tile_scores<DK, 1, F8>(f, A[0], A[1], p.relu != 0, sc[0], sc[1]);
        tile_scores<DK, 1, F8>(f, A[2], A[3], p.relu != 0, sc[2], sc[3]);
        float cv = sc[0];
#pragma unroll
        for (int t = 1; t < 4; ++t)
          if (c == t) cv = sc[t];
        const bool mine = ci >= lo[q] && ci < hi[q];
        topp_offer(mine ? cv : -INFINITY, mine ? ci : 0x7fffffff, p.P, tv[q], ti[q], thv[q], thi[q]);
      }
      }
    }
#pragma unroll
    for (int q = 0; q < G; ++q) topp_write(p, b0 + q, j, n[q], lo[q], hi[q], tv[q], ti[q]);
  }
}

// ---------------------------------------------------------------------------------
// Reindex scoring parameters (the scoring itself runs inside k_select_cl).
// ---------------------------------------------------------------------------------
struct PoolScoreParams {
  const uint16_t* q;
  const float* w;
  const uint8_t* q8;      // FP8 form (workspace), as in ScanParams
  const float* w8;
  csa2_cache cache;
  const int* seq_of;
  const int* pool;
  const int* pool_len;
  int stride;
  int H_i;
  int relu;
  float* score;           // [B][stride]
};

// ---------------------------------------------------------------------------------
// Exact Top-k of up to 16,384 scored candidates per query: 4-pass radix select of the
// k-th largest key, then ties at that key taken in ascending position, output in
// ascending position (= ascending entry, the pool being ascending).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(FULL_MASK, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = (lane < nw) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(FULL_MASK, t, o);
      if (lane >= o) t += y;
    }
    sh[lane] = t;
  }
  __syncthreads();
  int base = warp ? sh[warp - 1] : 0;
  total = sh[nw - 1];
  __syncthreads();
  return base + x - v;
}

struct SelectParams {
  const float* score;     // [B][stride]
  const int* pool;        // [B][stride]
  int stride;
  // candidate count: full mode -> min(n_vis[b], stride); reindex -> pool_len[b]
  const int* n_vis;
  int max_n;
  const int* pool_len_in;
  int* pool_len_out;      // full mode: written
  int* pool_out;          // full mode: tail filled with -1
  int k;
  int* topk;
  int* topk_len;
};

// ---------------------------------------------------------------------------------
// Cluster Top-k: the candidates of one query are split over a cluster of NCL CTAs
// (2,048 each at most).  Radix-select histograms and the compaction offsets are
// combined through distributed shared memory, so every pass runs on NCL SMs at once.
// With SCORE the CTAs first score their slice of the pool (Reindex) into shared
// memory; otherwise they read the scores the Full scan wrote (and finish the pool).
// ---------------------------------------------------------------------------------
constexpr int NCL = 8;
constexpr int CL_SLICE = 16384 / NCL;                 // 2048
// Threads per CTA (CT): 256, or 128 when a batch's clusters would not fit the GPU at once with
// 256 (two CTAs an SM by registers, four at 128), so that they run in one wave.

// Histogram increment of `cnt` at `bin` for a warp: the lanes sharing the first active
// lane's bin add once (in the leading digits most keys share one); the others add their
// own.  Called by all 32 lanes of the warp.
__device__ __forceinline__ void hist_add_warp(int* hist, int bin, int cnt) {
  const bool active = cnt > 0;
  const unsigned act = __ballot_sync(FULL_MASK, active);
  if (!act) return;
  const int lane = threadIdx.x & 31, leader = __ffs(act) - 1;
  const int b0 = __shfl_sync(FULL_MASK, bin, leader);
  const bool same = active && bin == b0;
  const int tot = __reduce_add_sync(FULL_MASK, same ? cnt : 0);
  if (lane == leader) atomicAdd(&hist[b0], tot);
  if (active && !same) atomicAdd(&hist[bin], cnt);
}

// The cluster radix select's digits, from the top of the 32-bit key: 11, 11 and 10 bits.  A
// histogram is summed over the cluster in two steps, so that the distributed-shared-memory
// traffic stays at one word per thread and CTA: its CL_THREADS super-bins first, then the bins
// of the one super-bin that holds the wanted key.
__host__ __device__ constexpr int radix_shift(int pass) { return pass == 0 ? 21 : pass == 1 ? 10 : 0; }
__host__ __device__ constexpr int radix_bins(int pass) { return pass == 2 ? 1024 : 2048; }

// One pass of the cluster's radix select: count the live keys (those whose resolved bits equal
// `prefix`) by this pass's digit into `hb` (zeroed), sum the NCL CTAs' histograms through
// distributed shared memory and find the digit of the `remaining`-th largest live key.  `sup`
// receives this CTA's super-bin sums, `tot` is scratch for CL_THREADS sums.
// Returns true when every live key with that digit is selected (the digit's count equals what
// remains): the bits below it then decide nothing and the later passes are skipped.  Every CTA
// of the cluster computes the same totals, so all take the same decision.
template <int PASS, int CT>
__device__ __forceinline__ bool radix_pass(int* hb, int* sup, int* tot, const uint32_t (&key)[CL_SLICE / CT], int q0,
                                           int e1, uint32_t& prefix, uint32_t& mask, int& remaining, int* pick) {
  constexpr int CL_THREADS = CT, CL_PER_T = CL_SLICE / CT;
  constexpr int SHIFT = radix_shift(PASS), NB = radix_bins(PASS), SB = NB / CL_THREADS;   // bins per super-bin
  const int tid = threadIdx.x;
  {
    // this thread's keys in the digit of its first live key are counted once; the rest one by one
    int b0 = 0, c0 = 0;
    bool any = false;
#pragma unroll
    for (int i = 0; i < CL_PER_T; ++i) {
      const bool live = q0 + i < e1 && (key[i] & mask) == prefix;
      const int bi = (int)((key[i] >> SHIFT) & (NB - 1));
      if (live && !any) { b0 = bi; any = true; }
      c0 += (live && bi == b0) ? 1 : 0;
    }
    hist_add_warp(hb, b0, c0);
#pragma unroll
    for (int i = 0; i < CL_PER_T; ++i) {
      const int bi = (int)((key[i] >> SHIFT) & (NB - 1));
      if (q0 + i < e1 && (key[i] & mask) == prefix && bi != b0) atomicAdd(&hb[bi], 1);
    }
  }
  // super-bin t (thread t's) = bins [NB - SB (t + 1), NB - SB t): thread 0 has the top bins
  __syncthreads();                                        // this CTA's histogram is complete
  {
    const int4* h4 = reinterpret_cast<const int4*>(hb + NB - SB * (tid + 1));
    int sum = 0;
#pragma unroll
    for (int j = 0; j < SB / 4; ++j) {
      const int4 v = h4[j];
      sum += v.x + v.y + v.z + v.w;
    }
    sup[tid] = sum;
  }
  tc::cluster_sync();                                     // every CTA's counts are complete
  {
    const uint32_t a = smem_u32(sup + tid);
    int sum = 0;
#pragma unroll
    for (int cc = 0; cc < NCL; ++cc) sum += tc::ld_dsmem_s32(tc::mapa(a, cc));
    tot[tid] = sum;
  }
  __syncthreads();
  if (tid < 32) {
    // warp 0 scans the super-bin totals from the top, SPL a lane
    constexpr int SPL = CL_THREADS / 32;
    int c8[SPL], local = 0;
#pragma unroll
    for (int i = 0; i < SPL; ++i) { c8[i] = tot[SPL * tid + i]; local += c8[i]; }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, incl, o);
      if (tid >= o) incl += y;
    }
    int sstar = -1, before = 0;
    if (incl - local < remaining && remaining <= incl) {
      int cum = incl - local;
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        if (cum < remaining && cum + c8[i] >= remaining) { sstar = SPL * tid + i; before = cum; }
        cum += c8[i];
      }
    }
    const int src = __ffs(__ballot_sync(FULL_MASK, sstar >= 0)) - 1;   // exactly one lane
    sstar = __shfl_sync(FULL_MASK, sstar, src);
    before = __shfl_sync(FULL_MASK, before, src);
    // the SB bins of super-bin s*, summed over the cluster: lane l < NJ * NCL loads 4 bins
    // (4 j .. 4 j + 3, j = l % NJ) of CTA l / NJ, and the lanes with the same j are summed
    constexpr int NJ = SB / 4;
    static_assert(SB % 4 == 0 && NJ * NCL <= 32, "one 4-bin load a lane");
    const int lo = NB - SB * (sstar + 1), j = tid % NJ;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (tid < NJ * NCL) v = tc::ld_dsmem_v4(tc::mapa(smem_u32(hb + lo + 4 * j), (uint32_t)(tid / NJ)));
    int x[4] = {(int)v.x, (int)v.y, (int)v.z, (int)v.w};
#pragma unroll
    for (int o = NJ; o < 32; o <<= 1)
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] += __shfl_xor_sync(FULL_MASK, x[i], o);
    int bin[SB];
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj)
#pragma unroll
      for (int i = 0; i < 4; ++i) bin[4 * jj + i] = __shfl_sync(FULL_MASK, x[i], jj);
    if (tid == 0) {
      int cum = before;
#pragma unroll
      for (int i = SB - 1; i >= 0; --i) {
        if (cum < remaining && cum + bin[i] >= remaining) {
          pick[0] = lo + i;
          pick[1] = remaining - cum;
          pick[2] = bin[i];
        }
        cum += bin[i];
      }
    }
  }
  __syncthreads();
  prefix |= ((uint32_t)pick[0]) << SHIFT;
  mask |= (uint32_t)(NB - 1) << SHIFT;
  remaining = pick[1];
  // (pick and tot are next written after the next pass's cluster barrier, once every thread
  //  of this CTA has read them)
  return pick[2] == remaining;
}

template <int DK, int NHG, bool SCORE, bool F8, int CT>
__global__ void __cluster_dims__(NCL, 1, 1) __launch_bounds__(CT, 512 / CT) k_select_cl(SelectParams p, PoolScoreParams sp) {
  constexpr int CL_THREADS = CT, CL_WARPS = CT / 32, CL_PER_T = CL_SLICE / CT;
  pdl_wait();
  pdl_trigger();
  // Reindex: the slice's scores and pool entries (2,048 each); once they are in registers,
  // the histograms of the first two passes (2,048 bins each)
  __shared__ __align__(16) int sbuf[2 * CL_SLICE];
  float* sscore = reinterpret_cast<float*>(sbuf);
  int* sent = sbuf + CL_SLICE;
  __shared__ __align__(16) int hist2[1024];         // the third pass's histogram
  __shared__ int sup[3][CL_THREADS];                // each pass's super-bin sums
  __shared__ int tot[CL_THREADS];                   // scratch of the passes
  __shared__ int scan_sh[32];
  __shared__ int pick[3];
  __shared__ int xfer;                              // this CTA's packed (above, equal) count
  __shared__ int base_sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.y;
  const int rank = (int)tc::cluster_ctarank();
  int P;
  if (p.n_vis) {
    int n = __ldg(p.n_vis + b);
    n = max(0, min(n, p.max_n));
    P = min(n, p.stride);
  } else {
    P = __ldg(p.pool_len_in + b);
    if (P < 0 || P > p.stride) {
      if (tid == 0 && rank == 0) raise_error(&g_err_index, CSA2_DEVERR_POOL_ENTRY);
      P = max(0, min(P, p.stride));
    }
  }
  const long long rowb = (long long)b * p.stride;
  const int S = (p.stride + NCL - 1) / NCL;
  const int s0 = rank * S, s1 = min(p.stride, s0 + S);
  const int k = p.k;
  int* out = p.topk + (long long)b * k;
  if (p.pool_len_out && tid == 0 && rank == 0) p.pool_len_out[b] = P;
  if (p.pool_out)
    for (int i = max(P, s0) + tid; i < s1; i += CL_THREADS) p.pool_out[rowb + i] = -1;
  if (P <= k) {                                           // every candidate is selected
    for (int i = s0 + tid; i < min(s1, P); i += CL_THREADS) out[i] = p.pool[rowb + i];
    for (int i = P + rank * CL_THREADS + tid; i < k; i += NCL * CL_THREADS) out[i] = -1;
    if (tid == 0 && rank == 0) p.topk_len[b] = P;
    return;                                               // the same in every CTA of the cluster
  }
  const int e1 = min(s1, P);                              // valid positions [s0, e1)
  for (int i = tid; i < 1024; i += CL_THREADS) hist2[i] = 0;
  if constexpr (SCORE) {
    // ---- score this CTA's slice of the pool (Reindex).  Warp w owns tiles w, w + CL_WARPS, ...
    //      of 32 positions; lane (g, c) owns rows g + 8u of a tile.  While a tile's rows
    //      are loading, the next tile's rows are resolved (pool id -> page table) and the
    //      pool ids of the tile after that are fetched.
    // tiles of 32 positions per iteration: two for the FP8 form's half-size rows (as in the
    // scan), one when several head groups need the registers
    constexpr int TPI = (F8 && NHG == 1) ? 2 : 1;
    constexpr int U = 4 * TPI;                     // rows per lane per iteration
    constexpr int NT = CL_SLICE / (32 * TPI) / (CL_THREADS / 32);   // iterations per warp: 8 (bf16), 4 (FP8)
    const int g = lane >> 2, c = lane & 3;
    const int sq = __ldg(sp.seq_of + b);
    // as in the Full scan: more than two head groups stream their Q fragments from L1
    constexpr bool STREAM_Q = NHG > 2;
    constexpr int NHG_REG = STREAM_Q ? 1 : NHG;
    constexpr int QB = F8 ? 1 : 2;               // bytes per indexer-Q element
    const uint8_t* qb = reinterpret_cast<const uint8_t*>(F8 ? (const void*)sp.q8 : (const void*)sp.q) +
                        (long long)b * sp.H_i * DK * QB;
    const float* wb = (F8 ? sp.w8 : sp.w) + (long long)b * sp.H_i;
    QFrag<DK, NHG_REG, F8> f;
    if (!STREAM_Q) load_qfrag<DK, NHG_REG, F8>(qb, wb, sp.H_i, f);
    auto pos_of = [&](int it, int u) { return s0 + 32 * TPI * (warp + CL_WARPS * it) + g + 8 * u; };
    // lane (g, c) fetches the pool ids of rows u = c + 4v (v < TPI) and resolves them; the
    // four lanes of a quad share the rows (each row is loaded in slices by a whole quad)
    auto fetch_ent = [&](int it, int* e) {
#pragma unroll
      for (int v = 0; v < TPI; ++v) {
        const int pos = pos_of(it, c + 4 * v);
        e[v] = (it < NT && pos < e1) ? __ldg(sp.pool + rowb + pos) : -1;
      }
    };
    auto resolve = [&](int it, const int* e, int* rw, float* rs) {
#pragma unroll
      for (int v = 0; v < TPI; ++v) {
        const int pos = pos_of(it, c + 4 * v);
        if (it < NT && pos < e1) sent[pos - s0] = e[v];
        rw[v] = (e[v] >= 0) ? (int)entry_row(sp.cache, sq, e[v], &g_err_index) : -1;
        rs[v] = (F8 && rw[v] >= 0) ? __ldg(sp.cache.idx_k8_scale + rw[v]) : 0.f;
      }
    };
    int en[TPI];
    int rw[TPI];
    float rs[TPI];                                 // FP8 form: the resolved rows' scales
    fetch_ent(0, en);
    resolve(0, en, rw, rs);
    fetch_ent(1, en);
#pragma unroll 1
    for (int it = 0; it < NT && s0 + 32 * TPI * (warp + CL_WARPS * it) < e1; ++it) {
      KRow<DK, F8> A[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int src = (lane & ~3) | (u & 3);
        load_row<DK, F8, false>(sp.cache, __shfl_sync(FULL_MASK, rw[u >> 2], src), A[u],
                                F8 ? __shfl_sync(FULL_MASK, rs[u >> 2], src) : -1.f);
      }
      resolve(it + 1, en, rw, rs);                        // next tile, while these rows load
      fetch_ent(it + 2, en);
      float sc[U];
#pragma unroll
      for (int tt = 0; tt < TPI; ++tt) {
        float* st = sc + 4 * tt;
        const KRow<DK, F8>* At = A + 4 * tt;
        if (STREAM_Q) {
          st[0] = st[1] = st[2] = st[3] = 0.f;
#pragma unroll 1
          for (int hg = 0; hg < NHG; ++hg) {
            load_qfrag<DK, NHG_REG, F8>(qb + hg * 8 * DK * QB, wb + hg * 8, sp.H_i - hg * 8, f);
            float x0, x1, x2, x3;
            tile_scores<DK, NHG_REG, F8>(f, At[0], At[1], sp.relu != 0, x0, x1);
            tile_scores<DK, NHG_REG, F8>(f, At[2], At[3], sp.relu != 0, x2, x3);
            st[0] += x0;
            st[1] += x1;
            st[2] += x2;
            st[3] += x3;
          }
        } else {
          tile_scores<DK, NHG_REG, F8>(f, At[0], At[1], sp.relu != 0, st[0], st[1]);
          tile_scores<DK, NHG_REG, F8>(f, At[2], At[3], sp.relu != 0, st[2], st[3]);
        }
      }
      if (c == 0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int pos = pos_of(it, u);
          if (pos < e1) sscore[pos - s0] = sc[u];
        }
      }
    }
  }
  __syncthreads();                                        // scores and zeroed histograms
  // ---- keys (and pool entries): 8 consecutive positions per thread ---------------------
  uint32_t key[CL_PER_T];
  int ent[CL_PER_T];
  const int q0 = s0 + tid * CL_PER_T;
  {
    // Reindex: the slice's positions q0 - s0 .. + CL_PER_T - 1 in 16-byte loads of each array
    float sv[CL_PER_T];
    if constexpr (SCORE) {
      const float4* s4 = reinterpret_cast<const float4*>(sscore + (q0 - s0));
      const int4* e4 = reinterpret_cast<const int4*>(sent + (q0 - s0));
#pragma unroll
      for (int h = 0; h < CL_PER_T / 4; ++h) {
        const float4 a = s4[h];
        const int4 c = e4[h];
        sv[4 * h] = a.x; sv[4 * h + 1] = a.y; sv[4 * h + 2] = a.z; sv[4 * h + 3] = a.w;
        ent[4 * h] = c.x; ent[4 * h + 1] = c.y; ent[4 * h + 2] = c.z; ent[4 * h + 3] = c.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < CL_PER_T; ++i) {
        sv[i] = q0 + i < e1 ? __ldg(p.score + rowb + q0 + i) : 0.f;
        ent[i] = q0 + i < e1 ? __ldg(p.pool + rowb + q0 + i) : -1;
      }
    }
#pragma unroll
    for (int i = 0; i < CL_PER_T; ++i) {
      if (q0 + i >= e1) ent[i] = -1;
      key[i] = (q0 + i < e1) ? float_key(sv[i]) : 0u;
    }
  }
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  __syncthreads();                                        // every key is in registers: sbuf
  for (int i = tid; i < 2 * CL_SLICE; i += CL_THREADS) sbuf[i] = 0;   // becomes two histograms
  __syncthreads();
  bool done = radix_pass<0, CT>(sbuf, sup[0], tot, key, q0, e1, prefix, mask, remaining, pick);
  if (!done) done = radix_pass<1, CT>(sbuf + 2048, sup[1], tot, key, q0, e1, prefix, mask, remaining, pick);
  if (!done) radix_pass<2, CT>(hist2, sup[2], tot, key, q0, e1, prefix, mask, remaining, pick);
  // ---- output slots from one scan of (keys above the threshold, keys equal to it), keys
  //      compared on the bits the passes resolved: ties at the threshold go to the lowest
  //      positions, cluster-wide (when the passes stopped early, every key equal on those
  //      bits is taken) ---------------------------------------------------------------------
  int gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < CL_PER_T; ++i) {
    if (q0 + i < e1) {
      gt += (key[i] & mask) > prefix ? 1 : 0;
      eq += (key[i] & mask) == prefix ? 1 : 0;
    }
  }
  int packed;
  const int ex = block_exclusive_scan(gt | (eq << 16), scan_sh, packed);   // counts < 2^15
  if (tid == 0) xfer = packed;
  tc::cluster_sync();
  if (tid == 0) {
    int bsum = 0;
    for (int cc = 0; cc < rank; ++cc) bsum += tc::ld_dsmem_s32(tc::mapa(smem_u32(&xfer), cc));
    base_sh = bsum;
  }
  __syncthreads();
  const int before = base_sh + ex;
  int er = before >> 16;                                  // equal keys before this thread
  int o = (before & 0xffff) + min(er, remaining);
#pragma unroll
  for (int i = 0; i < CL_PER_T; ++i) {
    const uint32_t km = key[i] & mask;
    if (q0 + i < e1 && (km > prefix || (km == prefix && er++ < remaining))) {
      if (o < k) out[o] = ent[i];
      ++o;
    }
  }
  if (tid == 0 && rank == 0) p.topk_len[b] = k;
  tc::cluster_sync();                                   // no CTA leaves while others read it
}

// ---------------------------------------------------------------------------------
// Top-k of one query's pool by one CTA, for many queries at once (a prefill chunk): an MSB
// radix select of 8-bit digits with block barriers instead of the cluster's, the same tie rule
// and early stop as k_select_cl (so the same output).  Full mode (scores written by the scan)
// only.
// ---------------------------------------------------------------------------------
constexpr int C1_THREADS = 512;
constexpr int C1_PER_T = 16384 / C1_THREADS;          // 32 consecutive positions per thread
constexpr int C1_ROW = C1_THREADS + 1;                // padded row of the key array
constexpr size_t C1_SMEM = (size_t)C1_PER_T * C1_ROW * sizeof(uint32_t);

// The keys live in shared memory (skey[i * C1_ROW + t] = key of position 32 t + i; the pad
// word keeps both the coalesced fill and the per-thread reads free of bank conflicts), so
// that several CTAs share an SM and one's loads overlap the others' passes.  Registers are
// held to 40 a thread for three CTAs an SM (at two, the 8,192 prefill selects took 9 % longer).
__global__ void __launch_bounds__(C1_THREADS, 3) k_select_cta(SelectParams p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t skey[];
  __shared__ int hist[4][256];                      // one per radix pass, zeroed at entry
  __shared__ int scan_sh[32];
  __shared__ int pick[3];
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  for (int i = tid; i < 4 * 256; i += C1_THREADS) (&hist[0][0])[i] = 0;
  const int n = max(0, min(__ldg(p.n_vis + b), p.max_n));
  const int P = min(n, p.stride);
  const long long rowb = (long long)b * p.stride;
  const int k = p.k;
  int* out = p.topk + (long long)b * k;
  if (p.pool_len_out && tid == 0) p.pool_len_out[b] = P;
  if (p.pool_out)
    for (int i = P + tid; i < p.stride; i += C1_THREADS) p.pool_out[rowb + i] = -1;
  if (P <= k) {                                    // every candidate is selected
    for (int i = tid; i < P; i += C1_THREADS) out[i] = p.pool[rowb + i];
    for (int i = P + tid; i < k; i += C1_THREADS) out[i] = -1;
    if (tid == 0) p.topk_len[b] = P;
    return;
  }
  // coalesced fill, eight loads in flight per thread: position q = c * 512 + tid
#pragma unroll 1
  for (int c0 = 0; c0 < C1_PER_T; c0 += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = (c0 + u) * C1_THREADS + tid;
      v[u] = q < P ? __ldg(p.score + rowb + q) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = (c0 + u) * C1_THREADS + tid;
      skey[(q & 31) * C1_ROW + (q >> 5)] = q < P ? float_key(v[u]) : 0u;
    }
  }
  __syncthreads();                                 // keys and zeroed histograms
  const int q0 = tid * C1_PER_T;
  const int nv = min(C1_PER_T, max(0, P - q0));   // this thread's valid positions
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int* hb = hist[pass];
    // the keys in the digit of this thread's first live key are counted once; the rest
    // (rare in the leading digits) one by one
    int b0 = -1, c0 = 0;
#pragma unroll 8
    for (int i = 0; i < nv; ++i) {
      const uint32_t key = skey[i * C1_ROW + tid];
      if ((key & mask) == prefix) {
        const int bi = (int)((key >> shift) & 255u);
        if (b0 < 0) b0 = bi;
        if (bi == b0) ++c0;
        else atomicAdd(&hb[bi], 1);
      }
    }
    hist_add_warp(hb, max(b0, 0), c0);
    __syncthreads();
    if (tid < 32) {
      int cnt[8], local = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { cnt[i] = hb[255 - 8 * tid - i]; local += cnt[i]; }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL_MASK, incl, o);
        if (tid >= o) incl += y;
      }
      const int excl = incl - local;
      if (excl < remaining && remaining <= incl) {
        int cum = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum + cnt[i] >= remaining) {
            pick[0] = 255 - 8 * tid - i;
            pick[1] = remaining - cum;
            pick[2] = cnt[i];
            break;
          }
          cum += cnt[i];
        }
      }
    }
    __syncthreads();
    prefix |= ((uint32_t)pick[0]) << shift;
    mask |= 0xFFu << shift;
    remaining = pick[1];
    // every key with the picked digit is selected: the bits below decide nothing (the same
    // value in every thread, so the whole CTA leaves the loop together)
    if (pick[2] == remaining) break;
  }
  // output slots from one scan of (keys above the threshold, keys equal to it, both on the
  // resolved bits): ties at the threshold go to the lowest positions
  int gt = 0, eq = 0;
#pragma unroll 8
  for (int i = 0; i < nv; ++i) {
    const uint32_t key = skey[i * C1_ROW + tid] & mask;
    gt += key > prefix ? 1 : 0;
    eq += key == prefix ? 1 : 0;
  }
  int tot;
  const int ex = block_exclusive_scan(gt | (eq << 16), scan_sh, tot);   // counts < 2^15
  int er = ex >> 16;                                // equal keys before this thread
  int o = (ex & 0xffff) + min(er, remaining);
#pragma unroll 8
  for (int i = 0; i < nv; ++i) {
    const uint32_t key = skey[i * C1_ROW + tid] & mask;
    if (key > prefix || (key == prefix && er++ < remaining)) {
      if (o < k) out[o] = __ldg(p.pool + rowb + q0 + i);
      ++o;
    }
  }
  if (tid == 0) p.topk_len[b] = k;
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
// persistent grid: as many CTAs as can be resident at once (the register use differs with
// the variant), capped by the work
template <typename K>
static void launch_persistent(K kernel, const ScanParams& sp, long long units, cudaStream_t st) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  const dim3 grid((unsigned)std::min<long long>(units, (long long)per_sm * (sms > 0 ? sms : 1)));
  // not a programmatic launch: a persistent grid sized to fill the GPU must start on an empty
  // GPU -- launched early, next to the previous kernel's CTAs, the 1M scan ran 1.2-1.8x slower
  launch_k_late(kernel, grid, 256, 0, st, sp);
}

template <int DK, bool F8>
static void launch_scan_group(const ScanParams& sp, int group, long long units, cudaStream_t st) {
  switch (group) {
    case 2: launch_persistent(k_full_scan_g<DK, 2, F8>, sp, units, st); break;
    case 3: launch_persistent(k_full_scan_g<DK, 3, F8>, sp, units, st); break;
    case 4: launch_persistent(k_full_scan_g<DK, 4, F8>, sp, units, st); break;
    case 5: launch_persistent(k_full_scan_g<DK, 5, F8>, sp, units, st); break;
    case 6: launch_persistent(k_full_scan_g<DK, 6, F8>, sp, units, st); break;
    case 7: launch_persistent(k_full_scan_g<DK, 7, F8>, sp, units, st); break;
    default: launch_persistent(k_full_scan_g<DK, 8, F8>, sp, units, st); break;
  }
}

// The short-block scan, whose score buffers are dynamic shared memory.
static cudaError_t launch_scan_short(const ScanParams& sp, cudaStream_t st) {
  constexpr int SEG = 32;
  auto kernel = k_full_scan_short<128, true, SEG>;
  constexpr size_t smem = ss_smem(SEG);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const long long units = ((long long)sp.B * ((sp.NB + SEG - 1) / SEG) + 7) / 8;
  const dim3 grid((unsigned)std::min<long long>(units, (long long)per_sm * (sms > 0 ? sms : 1)));
  launch_k_late(kernel, grid, 256, smem, st, sp);   // persistent: see launch_persistent
  return cudaGetLastError();
}

// the short-block scan serves the FP8 form with one head group, P = 8, d_ik = 128 and blocks
// of at most 64 entries
static bool scan_short_chosen(const csa2_index_full_args& a, int nhg, int group) {
  return a.cache.idx_k_dtype == CSA2_FP8E4M3 && nhg == 1 && group == 1 && a.per_block == SS_P &&
         a.cache.d_ik == 128 && ((long long)a.max_n + a.num_blocks - 1) / a.num_blocks <= SS_MAXB;
}

template <int DK, bool F8>
static void launch_scan_dk(const ScanParams& sp, int nhg, long long units, cudaStream_t st) {
  switch (nhg) {
    case 1: launch_persistent(k_full_scan<DK, 1, F8>, sp, units, st); break;
    case 2: launch_persistent(k_full_scan<DK, 2, F8>, sp, units, st); break;
    case 3: launch_persistent(k_full_scan<DK, 3, F8>, sp, units, st); break;
    default: launch_persistent(k_full_scan<DK, 4, F8>, sp, units, st); break;
  }
}

// The FP8 form's quantised indexer Q and weights, after `at` bytes of the workspace.
static size_t q8_bytes(int B, int H_i, int DK) { return (((size_t)B * H_i * DK + 255) & ~(size_t)255); }
static size_t q8_total(int B, int H_i, int DK) { return q8_bytes(B, H_i, DK) + (size_t)B * H_i * sizeof(float); }

static cudaError_t launch_quant_q8(const uint16_t* q, const float* w, int B, int H_i, int DK, uint8_t* q8, float* w8,
                                   cudaStream_t st) {
  const int rows = B * H_i;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  if (DK == 128) return launch_k(k_quant_q8<128>, grid, 256, 0, st, q, w, rows, q8, w8);
  return launch_k(k_quant_q8<64>, grid, 256, 0, st, q, w, rows, q8, w8);
}

// The tensor-core scoring streams every row once per group of queries and scores it against
// all of their heads; a single query with 8 heads keeps the scan, whose mma.sync scoring
// already runs at the memory rate (and writes no score matrix).  CSA2_INDEX_FULL=scan or
// =tc overrides the choice (for comparison measurements).
bool full_scores_tc_chosen(const csa2_index_full_args& a) {
  static int force = -2;
  if (force == -2) {
    const char* e = getenv("CSA2_INDEX_FULL");
    force = (e && e[0] == 't') ? 1 : (e && e[0] == 's') ? 0 : -1;
  }
  if (force == 0 || !full_scores_tc_supported(a)) return false;
  const int G = a.group > 1 ? a.group : 1;
  return force == 1 || G * a.H_i >= 16;
}

static size_t pool_score_bytes(const csa2_index_full_args& a) {
  return (((size_t)a.B * a.num_blocks * a.per_block * sizeof(float)) + 255) & ~(size_t)255;
}

size_t index_full_workspace_bytes(const csa2_index_full_args& a) {
  // pool scores, then (tensor-core scoring) the score matrix, or (FP8 form) the quantised
  // indexer Q and weights
  // (the score matrix starts 256-byte aligned: its rows are read in 16-byte loads)
  if (a.cache.idx_k_dtype == CSA2_FP8E4M3) return pool_score_bytes(a) + q8_total(a.B, a.H_i, a.cache.d_ik);
  if (full_scores_tc_chosen(a)) return pool_score_bytes(a) + full_scores_tc_bytes(a);
  return (size_t)a.B * a.num_blocks * a.per_block * sizeof(float);
}

cudaError_t launch_index_full(const csa2_index_full_args& a, void* ws, cudaStream_t st, bool allow_tc) {
  if (a.B == 0) return cudaSuccess;
  const int stride = a.num_blocks * a.per_block;
  ScanParams sp{};
  sp.q = a.q_idx;
  sp.w = a.w;
  sp.cache = a.cache;
  sp.seq_of = a.seq_of;
  sp.n_vis = a.n_vis;
  sp.max_n = a.max_n;
  sp.H_i = a.H_i;
  sp.NB = a.num_blocks;
  sp.P = a.per_block;
  sp.relu = a.relu;
  sp.pool = a.pool;
  sp.pool_score = static_cast<float*>(ws);
  sp.B = a.B;
  const int nhg = (a.H_i + 7) / 8;
  const int group = a.group > 1 ? a.group : 1;
  // CTAs of 8 blocks' work: per group of queries (grouped scan) or per query
  const long long units_g = ((long long)(a.B / group) * a.num_blocks + 7) / 8;
  const long long units = ((long long)a.B * a.num_blocks + 7) / 8;
  const bool f8 = a.cache.idx_k_dtype == CSA2_FP8E4M3;
  if (f8) {                                        // the indexer Q quantised like the compressed K
    uint8_t* q8 = static_cast<uint8_t*>(ws) + pool_score_bytes(a);
    float* w8 = reinterpret_cast<float*>(q8 + q8_bytes(a.B, a.H_i, a.cache.d_ik));
    cudaError_t e = launch_quant_q8(a.q_idx, a.w, a.B, a.H_i, a.cache.d_ik, q8, w8, st);
    if (e != cudaSuccess) return e;
    sp.q8 = q8;
    sp.w8 = w8;
    if (group > 1 && group <= 8 && a.H_i <= 8) {
      if (a.cache.d_ik == 128) launch_scan_group<128, true>(sp, group, units_g, st);
      else launch_scan_group<64, true>(sp, group, units_g, st);
    } else if (scan_short_chosen(a, nhg, group)) {
      cudaError_t e = launch_scan_short(sp, st);
      if (e != cudaSuccess) return e;
    } else if (a.cache.d_ik == 128) {
      launch_scan_dk<128, true>(sp, nhg, units, st);
    } else {
      launch_scan_dk<64, true>(sp, nhg, units, st);
    }
  } else if (allow_tc && full_scores_tc_chosen(a)) {     // groups of queries of one sequence: a dense product
    float* S = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pool_score_bytes(a));
    cudaError_t e = launch_full_scores_tc(a, S, static_cast<float*>(ws), st);
    if (e != cudaSuccess) return e;
  } else if (group > 1 && group <= 8 && a.H_i <= 8) {
    if (a.cache.d_ik == 128) launch_scan_group<128, false>(sp, group, units_g, st);
    else launch_scan_group<64, false>(sp, group, units_g, st);
  } else if (a.cache.d_ik == 128) {
    launch_scan_dk<128, false>(sp, nhg, units, st);
  } else {
    launch_scan_dk<64, false>(sp, nhg, units, st);
  }
  SelectParams sel{};
  sel.score = static_cast<const float*>(ws);
  sel.pool = a.pool;
  sel.stride = stride;
  sel.n_vis = a.n_vis;
  sel.max_n = a.max_n;
  sel.pool_len_out = a.pool_len;
  sel.pool_out = a.pool;
  sel.k = a.k;
  sel.topk = a.topk;
  sel.topk_len = a.topk_len;
  if (a.B >= 256) {                                // many queries: a CTA each, no cluster barriers
    static bool attr_set = false;
    if (!attr_set) {
      cudaError_t e = cudaFuncSetAttribute(k_select_cta, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C1_SMEM);
      if (e != cudaSuccess) return e;
      attr_set = true;
    }
    launch_k(k_select_cta, a.B, C1_THREADS, C1_SMEM, st, sel);
  } else {
    PoolScoreParams none{};
    launch_k_late(k_select_cl<128, 1, false, false, 256>, dim3(NCL, a.B), 256, 0, st, sel, none);
  }
  return cudaGetLastError();
}

// Reindex keeps its scores in shared memory; the FP8 form needs the quantised indexer Q
size_t index_reindex_workspace_bytes(const csa2_index_reindex_args& a) {
  return a.cache.idx_k_dtype == CSA2_FP8E4M3 ? q8_total(a.B, a.H_i, a.cache.d_ik) : 0;
}

template <int DK, bool F8>
static void launch_reindex_dk(const SelectParams& sel, const PoolScoreParams& pp, int nhg, int B, cudaStream_t st) {
  const dim3 grid(NCL, B);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // one head group: 128-thread CTAs once the clusters of 256-thread CTAs (two an SM) would need
  // a second wave (at 1M x 64, 56 against 63 us a call; at 32 queries 256 threads are faster:
  // 32 against 43 us)
  if (nhg == 1 && (long long)B * NCL > 2LL * sms) {
    launch_k_late(k_select_cl<DK, 1, true, F8, 128>, grid, 128, 0, st, sel, pp);
    return;
  }
  switch (nhg) {
    case 1: launch_k_late(k_select_cl<DK, 1, true, F8, 256>, grid, 256, 0, st, sel, pp); break;
    case 2: launch_k_late(k_select_cl<DK, 2, true, F8, 256>, grid, 256, 0, st, sel, pp); break;
    case 3: launch_k_late(k_select_cl<DK, 3, true, F8, 256>, grid, 256, 0, st, sel, pp); break;
    default: launch_k_late(k_select_cl<DK, 4, true, F8, 256>, grid, 256, 0, st, sel, pp); break;
  }
}

cudaError_t launch_index_reindex(const csa2_index_reindex_args& a, void* ws, cudaStream_t st) {
  if (a.B == 0) return cudaSuccess;
  PoolScoreParams pp{};
  pp.q = a.q_idx;
  pp.w = a.w;
  pp.cache = a.cache;
  pp.seq_of = a.seq_of;
  pp.pool = a.pool;
  pp.pool_len = a.pool_len;
  pp.stride = a.pool_stride;
  pp.H_i = a.H_i;
  pp.relu = a.relu;
  SelectParams sel{};
  sel.pool = a.pool;
  sel.stride = a.pool_stride;
  sel.pool_len_in = a.pool_len;
  sel.k = a.k;
  sel.topk = a.topk;
  sel.topk_len = a.topk_len;
  const int nhg = (a.H_i + 7) / 8;
  if (a.cache.idx_k_dtype == CSA2_FP8E4M3) {
    uint8_t* q8 = static_cast<uint8_t*>(ws);
    float* w8 = reinterpret_cast<float*>(q8 + q8_bytes(a.B, a.H_i, a.cache.d_ik));
    cudaError_t e = launch_quant_q8(a.q_idx, a.w, a.B, a.H_i, a.cache.d_ik, q8, w8, st);
    if (e != cudaSuccess) return e;
    pp.q8 = q8;
    pp.w8 = w8;
    if (a.cache.d_ik == 128) launch_reindex_dk<128, true>(sel, pp, nhg, a.B, st);
    else launch_reindex_dk<64, true>(sel, pp, nhg, a.B, st);
  } else if (a.cache.d_ik == 128) {
    launch_reindex_dk<128, false>(sel, pp, nhg, a.B, st);
  } else {
    launch_reindex_dk<64, false>(sel, pp, nhg, a.B, st);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// Fixed scratch for csa2_index_full_noalloc: the pool scores live in this array
// instead of a caller workspace.  Host code cannot use the symbol as a device address,
// so the address is looked up with the device current, once per CUDA context: the
// array's address belongs to the context the library's module is loaded in, so the cache
// is keyed by the context's unique id (a new context after cudaDeviceReset, or a second
// context on the same device, gets its own lookup).
// ---------------------------------------------------------------------------------
static __device__ __align__(256) float g_noalloc_scores[CSA2_NOALLOC_MAX_SCORES];

namespace {
constexpr int kMaxContexts = 64;
std::mutex g_noalloc_mu;
unsigned long long g_noalloc_ctx[kMaxContexts] = {};
void* g_noalloc_addr[kMaxContexts] = {};
int g_noalloc_n = 0;

typedef CUresult (*PFN_ctx_current)(CUcontext*);
typedef CUresult (*PFN_ctx_id)(CUcontext, unsigned long long*);

// unique id of the calling thread's current context; false when the driver cannot say
bool current_context_id(unsigned long long* id) {
  static PFN_ctx_current get_current = nullptr;
  static PFN_ctx_id get_id = nullptr;
  static bool tried = false;
  if (!tried) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_ctx_current>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_ctx_id>(fn);
    tried = true;
  }
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t index_noalloc_scratch(void** ptr, size_t* bytes) {
  *bytes = sizeof(g_noalloc_scores);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  if (have_id)
    for (int i = 0; i < g_noalloc_n; ++i)
      if (g_noalloc_ctx[i] == id) {
        *ptr = g_noalloc_addr[i];
        return cudaSuccess;
      }
  // no context current yet (the lookup below creates the primary one) or a new context
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scores);
  if (e != cudaSuccess) return e;
  if (have_id && g_noalloc_n < kMaxContexts) {      // remembered; past 64 contexts looked up each call
    g_noalloc_ctx[g_noalloc_n] = id;
    g_noalloc_addr[g_noalloc_n] = p;
    ++g_noalloc_n;
  }
  *ptr = p;
  return cudaSuccess;
}

uint32_t read_clear_error_index() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_index, sizeof(v));
  cudaMemcpyToSymbol(g_err_index, &z, sizeof(z));
  return v;
}

}  // namespace csa2
