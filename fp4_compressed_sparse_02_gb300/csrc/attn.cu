// Sparse MQA attention of each decode query over its selected FP4 Main KV entries plus
// its FP8 SWA window, in one softmax.
//
// "DeepSeek-V4.1-Flash deep dive", section 3.1: Main Q attends to (selected Main KV +
// layer-local SWA KV); section 6.3: 64 query heads x 512 dims, Top-K 512, n_win 128.
//
// Split over keys: CTA (query b, chunk c) takes key slots [c*128, c*128+128) of the
// list [topk slots 0..k) ++ [window rows 0..swa_max), gathers and dequantises them into
// shared memory as fp16 (FP4 x E4M3 and E4M3 values are exact in fp16), runs
// S = Q K^T and O = P V on the tensor cores (mma.sync m16n8k16, fp16 in, fp32
// accumulate) and writes an unnormalised partial (O, row max, row sum).  k_combine
// merges the chunks of a query.  The entry vector is both K and V, so one shared-memory
// tile serves both products (row-major for S, transposed ldmatrix for O).
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

#include <cstdlib>

namespace csa2 {

CSA2_DEFINE_ERROR_WORD(g_err_attn);

constexpr unsigned AFULL = 0xffffffffu;
constexpr int KC = 128;          // keys per CTA
constexpr int ATHREADS = 512;    // 16 warps
constexpr float LOG2E = 1.4426950408889634f;

struct AttnParams {
  const uint16_t* q;
  csa2_cache cache;
  const int* seq_of;
  const int* topk;
  const int* topk_len;
  int k;
  const uint8_t* swa;
  const float* swa_scale;
  int swa_rows;
  const int* swa_start;
  const int* swa_len;
  int swa_max;
  int Hq;
  int nchunk;
  float scale_log2;               // softmax_scale * log2(e)
  float* opart;                   // [B][nchunk][Hq][DIM]
  float2* ml;                     // [B][nchunk][Hq]  (row max in log2 units, row sum)
  // tcgen05 path: normalised fp16 partials, per-query arrival counters, final outputs
  __half* opart16;                // [B][nchunk][Hq][DIM]
  int* counter;                   // [B], zero on entry
  void* out;
  int out_f32;
  float* lse;
  int early;                      // inputs_ready: read and compute before waiting on the
                                  // previous kernel, wait only before the first write.  The
                                  // wait returns once that kernel (and so, transitively, every
                                  // earlier one) has completed, so all writes stay ordered.
};

// byte offset of 16-byte chunk `ch` of row `row` in a swizzled tile of `rowbytes`
__device__ __forceinline__ uint32_t swz(int row, int ch, int rowbytes) {
  return (uint32_t)(row * rowbytes + ((ch ^ (row & 7)) << 4));
}

// ---- operand ranges ---------------------------------------------------------------------
// The products run on fp16 operands.  fp16 holds every FP4 x E4M3 value and every E4M3 value
// exactly, so the key tile holds the FP4 rows dequantised and the window rows as their raw
// E4M3 values: the keys are exact.  A window row's float32 scale c_r is applied in float32
// instead, to its logit (S column r times c_r) and to its probability in the P.V product
// (p_r c_r 2^-G, G a per-CTA power of two that keeps every p_r c_r 2^-G <= 1; undone on the
// partial output).  So the logits carry no rounding of the keys, which their size would
// amplify.  q (bf16) is scaled per head by a power of two that puts its largest magnitude in
// [2^14, 2^15) before the fp16 rounding (exact; undone on the logits).

// 2^e as float32, e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// the shift F with (nonnegative float bits `mx`) * 2^-F in [2^14, 2^15); 0 for mx == 0.
// Clamped to [-100, 100]: beyond that the values are far below (or the logits far beyond)
// anything the float32 softmax resolves.
__device__ __forceinline__ int pow2_shift(uint32_t mx) {
  if (mx == 0u) return 0;
  const int e = (int)((mx >> 23) & 0xffu) - 127 - 14;
  return max(-100, min(100, e));
}

// the G with (positive float bits `mx`) * 2^-G in [0.5, 1); 0 for mx == 0.  Clamped to
// [-126, 126] (2^-G stays a normal float32).
__device__ __forceinline__ int pfactor_shift(uint32_t mx) {
  if (mx == 0u) return 0;
  return max(-126, min(126, (int)((mx >> 23) & 0xffu) - 126));
}

// largest |x| of eight bf16 values, as a bf16 magnitude bit pattern
__device__ __forceinline__ uint32_t bf16x8_absmax(uint4 v) {
  const uint32_t M = 0x7fff7fffu;
  const uint32_t m = __vmaxu2(__vmaxu2(v.x & M, v.y & M), __vmaxu2(v.z & M, v.w & M));
  return max(m & 0xffffu, m >> 16);
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t v, float s) {
  const float lo = __uint_as_float(v << 16) * s, hi = __uint_as_float(v & 0xffff0000u) * s;
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int DIM, int MT>
struct ACfg {
  static constexpr int HP = 16 * MT;                  // padded heads
  static constexpr int ROWB = DIM * 2;                // bytes per f16 row of Q / KV
  static constexpr int PROWB = KC * 2;                // bytes per f16 row of P
  static constexpr int KG = 16 / MT;                  // key groups in S
  static constexpr int KPW = KC / KG;                 // keys per warp in S (= 8*MT)
  static constexpr int DPW = DIM * MT / 16;           // dims per warp in O
  static constexpr int NTO = DPW / 8;                 // n-tiles per warp in O
  static constexpr int SMEM_Q = HP * ROWB;
  static constexpr int SMEM_KV = KC * ROWB;
  static constexpr int SMEM_P = HP * PROWB;
  static constexpr int SMEM_RED = 2 * HP * KG * 4;
  static constexpr int SMEM = SMEM_Q + SMEM_KV + SMEM_P + SMEM_RED;
};

template <int DIM, int MT>
__global__ void __launch_bounds__(ATHREADS, 1) k_attn_chunk(AttnParams p) {
  if (!p.early) pdl_wait();         // otherwise the wait comes before the first write (below)
  pdl_trigger();
  using C = ACfg<DIM, MT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sKV = sQ + C::SMEM_Q;
  uint8_t* sP = sKV + C::SMEM_KV;
  float* sMax = reinterpret_cast<float*>(sP + C::SMEM_P);   // [HP][KG]
  float* sSum = sMax + C::HP * C::KG;                         // [HP][KG]
  __shared__ long long keyrow[KC];
  __shared__ float keyscale[KC];
  __shared__ int keykind[KC];       // 0 none, 1 FP4 entry, 2 SWA row
  __shared__ float qf[C::HP];       // 2^F of each head's Q normalisation
  __shared__ uint32_t kvmax[ATHREADS / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.y, chunk = blockIdx.x;
  const uint32_t qs = smem_u32(sQ), kvs = smem_u32(sKV), ps = smem_u32(sP);

  // ---- 1. resolve this chunk's key slots --------------------------------------
  if (tid < KC) {
    const int j = chunk * KC + tid;
    int kind = 0;
    long long row = -1;
    float sc = 0.f;
    if (j < p.k) {
      int tl = p.topk_len ? __ldg(p.topk_len + b) : p.k;
      if (j < tl) {
        int e = __ldg(p.topk + (long long)b * p.k + j);
        if (e >= 0) {
          row = entry_row(p.cache, __ldg(p.seq_of + b), e, &g_err_attn);
          kind = row >= 0 ? 1 : 0;
          sc = kind ? 1.f : 0.f;
        }
      }
    } else if (j - p.k < p.swa_max) {
      int w = j - p.k;
      if (w < __ldg(p.swa_len + b)) {
        long long r = (long long)__ldg(p.swa_start + b) + w;
        if (r >= 0 && r < p.swa_rows) {
          row = r;
          kind = 2;
          sc = __ldg(p.swa_scale + r);
        } else {
          raise_error(&g_err_attn, CSA2_DEVERR_SWA_RANGE);
        }
      }
    }
    keyrow[tid] = row;
    keykind[tid] = kind;
    keyscale[tid] = sc;
  }
  // ---- 2. Q (bf16 -> fp16, scaled per head), rows >= Hq are zero: warp w converts heads
  //      w, w + 16, ..., lane l the head's 16-byte chunks l and l + 32 ---------------------
  {
    constexpr int CH = DIM / 8, CPL = (CH + 31) / 32;
    for (int h = warp; h < C::HP; h += ATHREADS / 32) {
      uint4 v[CPL];
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int ch = lane + 32 * j;
        v[j] = make_uint4(0, 0, 0, 0);
        if (h < p.Hq && ch < CH) v[j] = __ldg(reinterpret_cast<const uint4*>(p.q + ((long long)b * p.Hq + h) * DIM) + ch);
        m = max(m, bf16x8_absmax(v[j]));
      }
      const int F = pow2_shift(__reduce_max_sync(AFULL, m) << 16);
      const float sc = exp2i(-F);
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int ch = lane + 32 * j;
        if (ch < CH)
          *reinterpret_cast<uint4*>(sQ + swz(h, ch, C::ROWB)) =
              make_uint4(bf16x2_to_f16x2_scaled(v[j].x, sc), bf16x2_to_f16x2_scaled(v[j].y, sc),
                         bf16x2_to_f16x2_scaled(v[j].z, sc), bf16x2_to_f16x2_scaled(v[j].w, sc));
      }
      if (lane == 0) qf[h] = exp2i(F);
    }
  }
  __syncthreads();
  // ---- 3. the chunk's probability factor 2^-G: every key's float32 factor c (FP4 entry 1,
  //      window row its scale), maximised over the CTA ---------------------------------------
  const int key = tid >> 2, qtr = tid & 3;
  const int kind = keykind[key];
  const long long row = keyrow[key];
  constexpr int DQ = DIM / 4;                   // dims per thread
  {
    uint32_t mloc = kind == 0 ? 0u : __float_as_uint(fabsf(keyscale[key]));
    mloc = __reduce_max_sync(AFULL, mloc);
    if (lane == 0) kvmax[warp] = mloc;
  }
  __syncthreads();
  uint32_t kvm = 0;
#pragma unroll
  for (int w = 0; w < ATHREADS / 32; ++w) kvm = max(kvm, kvmax[w]);
  const int G = pfactor_shift(kvm);
  const float sG = exp2i(-G), fG = exp2i(G);
  // ---- 4. gather + dequantise the 128 keys (4 threads per key): FP4 rows exactly, window
  //      rows as their E4M3 values (both exact in fp16) ---------------------------------------
  {
    if (kind == 1) {
      const uint8_t* cp = p.cache.codes + row * (DIM / 2) + qtr * (DQ / 2);
      const uint8_t* sp = p.cache.scales + row * (DIM / 16) + qtr * (DQ / 16);
#pragma unroll
      for (int cc = 0; cc < DQ / 32; ++cc) {      // 16 code bytes = 32 dims = 2 scale groups
        uint4 cw = ldg_stream_v4(cp + cc * 16);
        uint16_t s2 = (uint16_t)sp[cc * 2] | ((uint16_t)sp[cc * 2 + 1] << 8);
        uint32_t sh = e4m3x2_to_f16x2(s2);
        uint32_t s0 = (sh & 0xffffu) * 0x10001u, s1 = (sh >> 16) * 0x10001u;
        uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
        uint32_t outw[16];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi)
#pragma unroll
          for (int bi = 0; bi < 4; ++bi) {
            uint32_t h2 = e2m1x2_to_f16x2((words[wi] >> (8 * bi)) & 0xffu);
            outw[wi * 4 + bi] = hmul2_u32(h2, wi < 2 ? s0 : s1);
          }
        const int ch0 = (qtr * DQ + cc * 32) / 8;
#pragma unroll
        for (int t = 0; t < 4; ++t)
          *reinterpret_cast<uint4*>(sKV + swz(key, ch0 + t, C::ROWB)) =
              make_uint4(outw[4 * t], outw[4 * t + 1], outw[4 * t + 2], outw[4 * t + 3]);
      }
    } else if (kind == 2) {
      const uint8_t* rp = p.swa + row * DIM + qtr * DQ;
#pragma unroll
      for (int cc = 0; cc < DQ / 16; ++cc) {      // 16 bytes = 16 dims = 2 smem chunks
        uint4 v = __ldg(reinterpret_cast<const uint4*>(rp + cc * 16));
        uint32_t words[4] = {v.x, v.y, v.z, v.w};
        uint32_t outw[8];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi)
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) outw[wi * 2 + hi] = e4m3x2_to_f16x2((uint16_t)(words[wi] >> (16 * hi)));
        const int ch0 = (qtr * DQ + cc * 16) / 8;
        *reinterpret_cast<uint4*>(sKV + swz(key, ch0, C::ROWB)) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
        *reinterpret_cast<uint4*>(sKV + swz(key, ch0 + 1, C::ROWB)) = make_uint4(outw[4], outw[5], outw[6], outw[7]);
      }
    } else {
      const int ch0 = qtr * DQ / 8;
#pragma unroll
      for (int t = 0; t < DQ / 8; ++t)
        *reinterpret_cast<uint4*>(sKV + swz(key, ch0 + t, C::ROWB)) = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  // ---- 4. S = Q K^T: warp -> (m-tile mt, key group kg of 8*MT keys) ------------
  const int mt = warp % MT, kg = warp / MT;
  const int kbase = kg * C::KPW;
  float sacc[MT][4];
#pragma unroll
  for (int t = 0; t < MT; ++t) sacc[t][0] = sacc[t][1] = sacc[t][2] = sacc[t][3] = 0.f;
  {
    const int arow = mt * 16 + (lane & 15);
    const int mi = lane >> 3, r8 = lane & 7;
    if constexpr (MT == 1) {
#pragma unroll 4
      for (int ks = 0; ks < DIM / 16; ks += 2) {
        uint32_t a[2][4];
        ldmatrix_x4(a[0][0], a[0][1], a[0][2], a[0][3], qs + swz(arow, 2 * ks + (lane >> 4), C::ROWB));
        ldmatrix_x4(a[1][0], a[1][1], a[1][2], a[1][3], qs + swz(arow, 2 * ks + 2 + (lane >> 4), C::ROWB));
        uint32_t bb[4];
        ldmatrix_x4(bb[0], bb[1], bb[2], bb[3], kvs + swz(kbase + r8, 2 * ks + mi, C::ROWB));
        mma_f16_16816(sacc[0], a[0][0], a[0][1], a[0][2], a[0][3], bb[0], bb[1]);
        mma_f16_16816(sacc[0], a[1][0], a[1][1], a[1][2], a[1][3], bb[2], bb[3]);
      }
    } else {
#pragma unroll 2
      for (int ks = 0; ks < DIM / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(a0, a1, a2, a3, qs + swz(arow, 2 * ks + (lane >> 4), C::ROWB));
#pragma unroll
        for (int np = 0; np < MT / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          const int key = kbase + np * 16 + (mi >> 1) * 8 + r8;
          ldmatrix_x4(b0, b1, b2, b3, kvs + swz(key, 2 * ks + (mi & 1), C::ROWB));
          mma_f16_16816(sacc[2 * np], a0, a1, a2, a3, b0, b1);
          mma_f16_16816(sacc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
  }
  // ---- 5. chunk-local softmax (logits in log2 units: the head's Q factor and the key's c
  //      applied) ----------------------------------------------------------------------------
  // thread holds rows r0 = mt*16+g, r1 = r0+8; keys kbase + 8t + 2c + {0,1}
  const int r0 = mt * 16 + g, r1 = r0 + 8;
  const float lsc0 = p.scale_log2 * qf[r0], lsc1 = p.scale_log2 * qf[r1];
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int t = 0; t < MT; ++t) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int kk = kbase + 8 * t + 2 * c + e;
      const bool valid = keykind[kk] != 0;
      const float ck = keyscale[kk];
      float v0 = valid ? sacc[t][e] * lsc0 * ck : -INFINITY;
      float v1 = valid ? sacc[t][2 + e] * lsc1 * ck : -INFINITY;
      sacc[t][e] = v0;
      sacc[t][2 + e] = v1;
      mx0 = fmaxf(mx0, v0);
      mx1 = fmaxf(mx1, v1);
    }
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(AFULL, mx0, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(AFULL, mx1, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(AFULL, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(AFULL, mx1, 2));
  if (c == 0) {
    sMax[r0 * C::KG + kg] = mx0;
    sMax[r1 * C::KG + kg] = mx1;
  }
  __syncthreads();
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int q = 0; q < C::KG; ++q) {
    m0 = fmaxf(m0, sMax[r0 * C::KG + q]);
    m1 = fmaxf(m1, sMax[r1 * C::KG + q]);
  }
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    const int kk = kbase + 8 * t + 2 * c;
    float e00 = (m0 == -INFINITY) ? 0.f : exp2f(sacc[t][0] - m0);
    float e01 = (m0 == -INFINITY) ? 0.f : exp2f(sacc[t][1] - m0);
    float e10 = (m1 == -INFINITY) ? 0.f : exp2f(sacc[t][2] - m1);
    float e11 = (m1 == -INFINITY) ? 0.f : exp2f(sacc[t][3] - m1);
    l0 += e00 + e01;
    l1 += e10 + e11;
    // the P.V weights p c 2^-G (<= 1; an invalid key has p = 0 and c = 0)
    const float c0 = keyscale[kk] * sG, c1 = keyscale[kk + 1] * sG;
    __half2 h0 = __floats2half2_rn(e00 * c0, e01 * c1);
    __half2 h1 = __floats2half2_rn(e10 * c0, e11 * c1);
    // P[row][key..key+1]: chunk key/8, element offset (key%8)*2 bytes
    *reinterpret_cast<__half2*>(sP + swz(r0, kk >> 3, C::PROWB) + (kk & 7) * 2) = h0;
    *reinterpret_cast<__half2*>(sP + swz(r1, kk >> 3, C::PROWB) + (kk & 7) * 2) = h1;
  }
  l0 += __shfl_xor_sync(AFULL, l0, 1);
  l1 += __shfl_xor_sync(AFULL, l1, 1);
  l0 += __shfl_xor_sync(AFULL, l0, 2);
  l1 += __shfl_xor_sync(AFULL, l1, 2);
  if (c == 0) {
    sSum[r0 * C::KG + kg] = l0;
    sSum[r1 * C::KG + kg] = l1;
  }
  __syncthreads();
  // ---- 6. O = P V: warp -> (m-tile mt, dims [dg*DPW, +DPW)) --------------------
  const int dg = warp / MT;
  const int dbase = dg * C::DPW;
  float oacc[C::NTO][4];
#pragma unroll
  for (int t = 0; t < C::NTO; ++t) oacc[t][0] = oacc[t][1] = oacc[t][2] = oacc[t][3] = 0.f;
  {
    const int arow = mt * 16 + (lane & 15);
    const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
    for (int ks = 0; ks < KC / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(a0, a1, a2, a3, ps + swz(arow, 2 * ks + (lane >> 4), C::PROWB));
      if constexpr (C::NTO == 1) {
        // two k-steps' worth is not needed: one n-tile, keys 16ks..16ks+15
        uint32_t b0, b1, b2, b3;
        const int kk = 16 * ks + (mi & 1) * 8 + r8;
        ldmatrix_x4_trans(b0, b1, b2, b3, kvs + swz(kk, dbase / 8, C::ROWB));
        mma_f16_16816(oacc[0], a0, a1, a2, a3, b0, b1);
      } else {
#pragma unroll
        for (int np = 0; np < C::NTO / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          const int kk = 16 * ks + (mi & 1) * 8 + r8;
          ldmatrix_x4_trans(b0, b1, b2, b3, kvs + swz(kk, (dbase + 16 * np) / 8 + (mi >> 1), C::ROWB));
          mma_f16_16816(oacc[2 * np], a0, a1, a2, a3, b0, b1);
          mma_f16_16816(oacc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
  }
  // ---- 7. partial outputs (the probability factor 2^-G undone) ------------------------
  if (p.early) pdl_wait();          // the workspace may still be read by the previous kernel
  const long long pbase = ((long long)b * p.nchunk + chunk) * p.Hq;
  if (r0 < p.Hq) {
    float* o = p.opart + (pbase + r0) * DIM + dbase + 2 * c;
#pragma unroll
    for (int t = 0; t < C::NTO; ++t)
      *reinterpret_cast<float2*>(o + 8 * t) = make_float2(oacc[t][0] * fG, oacc[t][1] * fG);
  }
  if (r1 < p.Hq) {
    float* o = p.opart + (pbase + r1) * DIM + dbase + 2 * c;
#pragma unroll
    for (int t = 0; t < C::NTO; ++t)
      *reinterpret_cast<float2*>(o + 8 * t) = make_float2(oacc[t][2] * fG, oacc[t][3] * fG);
  }
  if (dg == 0 && c == 0) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int q = 0; q < C::KG; ++q) { s0 += sSum[r0 * C::KG + q]; s1 += sSum[r1 * C::KG + q]; }
    if (r0 < p.Hq) p.ml[pbase + r0] = make_float2(m0, s0);
    if (r1 < p.Hq) p.ml[pbase + r1] = make_float2(m1, s1);
  }
}

// ---------------------------------------------------------------------------------
// tcgen05 path for d = 512, Hq = 64, k <= 512, swa_max <= 128 (the model's shape).
// CTA (chunk c of 4, query b), 256 threads.  The chunk's keys are the selected-entry
// slots [128c, 128c+128) and the window rows [32c, 32c+32): 160 keys, so a query needs
// 4 CTAs and a decode batch of 32 fills the GPU in one wave.  The 4 CTAs of a query form
// a thread-block cluster.
//   shared : KV tile 160 keys x 512 dims fp16 (K-major, 128-byte swizzle)      160 KB
//            Q 64 heads x 512 dims fp16 (K-major, 128-byte swizzle)               64 KB
//            Q arrives by TMA (bf16, eight 64-dim x 64-head boxes, every CTA loading the
//            query's whole Q for itself; L2 serves the other three CTAs' reads) issued at
//            kernel start; the data threads convert it to fp16 in place while their
//            gathers are in flight.
//   TMEM   : S = Q K^T (fp32, 160 columns)                              cols   0..159
//            P = softmax numerators (fp16 pairs, A operand)             cols   0..79
//            O quarter q = P V[:, 128q..] (fp32)      q0: 256..383, q1: 384..511,
//                                                     q2: 128..255, q3: 256..383
//   MMA1  S[64 x 160] = Q[smem] . KV^T        (A, B K-major)
//   MMA2  O[64 x 128] = P[tmem] . KV[:, quarter] (B MN-major: the same tile read along
//         the other axis); quarters 0..2 are issued back to back, quarter 3 once the
//         epilogue has read quarter 0, so the epilogues overlap the products.
// With M = 64 the 64 heads occupy lanes 0..15 of each of the four TMEM lane quarters, so
// all eight warps (two per quarter, each taking half of the keys or dims) share the
// softmax and the epilogue; the 16x32bx2 access shape gives lanes 0..15 and 16..31 of a
// warp two column ranges of the same 16 heads, so every thread carries data.
// CTA r owns the merge of heads [16 r, 16 r + 16).  Once every CTA of the cluster has
// finished MMA1 (a cluster barrier), the epilogue writes o = O / l (fp16) of each head and
// its (max, l) pair straight into the owning CTA's Q space (slot = this chunk, 1 KB rows)
// with distributed-shared-memory stores; a second cluster barrier (release / acquire)
// makes them visible, and the owner combines the 4 chunks from its own shared memory.
// ---------------------------------------------------------------------------------
namespace tca {
constexpr int NW = 256;                         // data threads: warps 0..7
constexpr int THREADS = NW + 32;                // + warp 8, whose lane 0 issues the MMAs
constexpr int ISSUER = NW;
constexpr int HQ = 64;
constexpr int DIM = 512;
constexpr int NCH = 4;                          // chunks per query
constexpr int KT = 128;                         // selected-entry slots per chunk
constexpr int KW = 32;                          // window rows per chunk
constexpr int NK = KT + KW;                     // keys per chunk
constexpr int ATOM = NK / 8 * 1024;             // bytes per 64-dim K-atom of the KV tile
constexpr int QATOM = HQ / 8 * 1024;            // bytes per 64-dim K-atom of the Q tile
constexpr int SM_KV = NK * DIM * 2;             // 163840
constexpr int SM_Q = HQ * DIM * 2;              // 65536
struct Misc {                                   // small per-CTA state, after the tiles
  alignas(16) float kc[NK];      // each key's logit factor c: 1 (FP4 entry), the row scale
                                 // (window row), NaN (no key)
  int8_t qfe[HQ];                // F of each head's Q normalisation (q scaled by 2^-F)
  float pmax[2][HQ];
  float psum[2][HQ];
  alignas(16) float2 rml[NCH][HQ / NCH];   // (row max in log2 units, row sum) of each chunk
                                           // for this CTA's 16 heads
  alignas(16) float2 rml_out[NCH][HQ / NCH];   // this chunk's pairs for each owner's heads
  alignas(16) float ecs[NCH][4];          // [c][0]: 2^G of chunk c (its P.V weights carry 2^-G)
  alignas(16) float ec_out[4];            // [0]: this chunk's 2^G, sent to the other owners
  uint32_t kvmax[NW / 32];                // each data warp's largest key factor c (float bits)
  uint64_t mbar[10];              // 0: MMA1, 1..4: MMA2 quarters, 5: dims 0..255 of every key
                                  // written (by the 8 data warps), 6: quarter 0's columns read
                                  // by the 8 data warps, 7: Q landed, 8: the other chunks'
                                  // blocks of this CTA's heads landed, 9: the raw rows landed
  uint32_t tslot;
  int ok_flag;
};
constexpr int SMEM = SM_KV + SM_Q + (int)sizeof(Misc);   // no static shared memory
static_assert(SMEM <= 232448, "shared memory per CTA");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0;                   // S, then P over its first 80 columns
constexpr uint32_t MAX_POLL = 1u << 22;
constexpr int BLK = HQ / NCH * DIM * 2;         // one chunk's block of 16 heads x 512 dims fp16
// raw rows land by TMA in the tail of the KV tile (read into registers before any
// dequantised row is written): FP4 codes [128][256 B], scales [128][32 B], window rows as
// two 256-byte halves [2][32][256 B]
constexpr int STG_CODES = 32768, STG_SCALES = 4096, STG_SWA = 16384;
constexpr int STG = SM_KV - (STG_CODES + STG_SCALES + STG_SWA);
static_assert(STG % 1024 == 0, "staging alignment");
constexpr int QBLK = BLK / 4;                   // its part of one O quarter (128 dims), 4 KB
constexpr uint32_t RECV_BYTES = (NCH - 1) * (4 * QBLK + HQ / NCH * 8 + 16);   // from the 3 other chunks

__device__ __forceinline__ uint32_t col_o(int q) { return q == 0 ? 256u : q == 1 ? 384u : q == 2 ? 128u : 256u; }

// byte offset of 16-byte chunk ch (8 fp16) of row r in a K-major swizzled tile whose
// 64-dim atoms are `atom` bytes apart
__device__ __forceinline__ uint32_t tileoff(int r, int ch, int atom) {
  return (uint32_t)((ch >> 3) * atom + (r >> 3) * 1024 + (r & 7) * 128 + (((ch & 7) ^ (r & 7)) << 4));
}
__device__ __forceinline__ uint32_t kvoff(int r, int ch) { return tileoff(r, ch, ATOM); }

__device__ __forceinline__ bool wait_mma(uint64_t* mbar, uint32_t parity) {
  const bool ok = tc::mbar_wait(mbar, parity, MAX_POLL);
  if (!ok) raise_error(&g_err_attn, CSA2_DEVERR_TIMEOUT);
  return ok;
}
}  // namespace tca

__global__ void __cluster_dims__(tca::NCH, 1, 1) __launch_bounds__(tca::THREADS, 1)
    k_attn_tc(AttnParams p, const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap cmap,
              const __grid_constant__ CUtensorMap smap, const __grid_constant__ CUtensorMap wmap) {
  if (!p.early) pdl_wait();         // otherwise the wait comes before the merge's writes
  pdl_trigger();
  using namespace tca;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sKV = smem;
  uint8_t* sQ = smem + SM_KV;
  Misc& ms = *reinterpret_cast<Misc*>(smem + SM_KV + SM_Q);
  float (*pmax)[HQ] = ms.pmax;
  float (*psum)[HQ] = ms.psum;
  uint64_t* mbar = ms.mbar;
  int& ok_flag = ms.ok_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.y, chunk = blockIdx.x;
  if ((smem_u32(smem) & 1023) != 0) {           // the same in every CTA: all return together
    if (tid == 0) raise_error(&g_err_attn, CSA2_DEVERR_SMEM_ALIGN);
    return;
  }
  const uint32_t kv_a = smem_u32(sKV), q_a = smem_u32(sQ);
  // M = 64 tensor-memory layout: head h sits in lane 32 * (h / 16) + h % 16, so warp w
  // (lane quarter w % 4) owns heads [16 (w % 4), 16 (w % 4) + 16) and warp >> 2 picks a
  // half of the columns; threads t and t + 16 of a warp hold the same head.
  const bool lv = lane < 16;
  const int head = 16 * (warp & 3) + (lane & 15);
  const int kh = warp >> 2;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

  // Warp 8 allocates TMEM (and frees it at the end); its lane 0 initialises the mbarriers and
  // at once issues this CTA's own load of Q.  The start-up cluster barrier orders every CTA's
  // mbarrier initialisation before the bulk copies other CTAs later complete on them (the
  // merge blocks): warp 8 arrives after initialising and waits at once; the data warps arrive
  // at once and wait for that phase only before issuing their gathers.
  const bool worker = tid < NW;
  float sG = 1.f;                               // 2^-G: this chunk's P.V weights are p c 2^-G
  if (worker) {
    tc::cluster_arrive_relaxed();
  } else {
    tc::tmem_alloc(&ms.tslot, TMEM_COLS);
    if (tid == ISSUER) {
#pragma unroll
      for (int i = 0; i < 5; ++i) tc::mbar_init(&mbar[i], 1);
      tc::mbar_init(&mbar[5], NW / 32);
      tc::mbar_init(&mbar[6], NW / 32);
      tc::mbar_init(&mbar[7], 1);
      tc::mbar_init(&mbar[8], 1);
      tc::mbar_arrive_expect_tx(&mbar[8], RECV_BYTES);
      tc::mbar_init(&mbar[9], 1);
      tc::mbar_arrive_expect_tx(&mbar[9], STG_CODES + STG_SCALES + (p.swa_max > 0 ? STG_SWA : 0));
      tc::fence_proxy_async_smem();             // the initialised barriers, seen by the TMA unit
      ok_flag = 1;
      tc::mbar_arrive_expect_tx(&mbar[7], SM_Q);
#pragma unroll
      for (int a = 0; a < DIM / 64; ++a) tc::tma_load_2d(sQ + a * QATOM, &qmap, 64 * a, b * HQ, &mbar[7]);
    }
    __syncwarp();
    tc::cluster_arrive_relaxed();               // after fence.mbarrier_init (in mbar_init)
    tc::cluster_wait();
  }
  if (worker) {
  // ---- each thread resolves the keys it dequantises: FP4 slot fkey (2 threads per key)
  //      and window row skey (8 threads per key) -------------------------------------------
  const int fkey = tid >> 1, half = tid & 1;
  const int skey = KT + (tid >> 3), part = tid & 7;
  long long frow = -1, srow = -1;
  float ssc = 0.f;
  int wrow0 = 0;                                // first window row of this chunk
  {
    // two rounds of loads: first every index that depends on nothing, then the page-table
    // entry and the window row's scale together
    const int j = chunk * KT + fkey, w = chunk * KW + (tid >> 3);
    const int tl = p.topk_len ? __ldg(p.topk_len + b) : p.k;
    const int e = (j < p.k) ? __ldg(p.topk + (long long)b * p.k + j) : -1;
    const int sq = __ldg(p.seq_of + b);
    const int wl = p.swa_max > 0 ? __ldg(p.swa_len + b) : 0;
    const long long r0 = p.swa_max > 0 ? (long long)__ldg(p.swa_start + b) + chunk * KW : 0;
    int page = -1;
    bool fslot = false;
    if (j < p.k && j < tl && e >= 0) page = entry_page_load(p.cache, sq, e, &g_err_attn, fslot);
    if (p.swa_max > 0) {
      wrow0 = (int)max(-(long long)KW, min(r0, (long long)p.swa_rows));   // TMA fills rows outside
      const long long r = r0 + (tid >> 3);
      if (w < p.swa_max && w < wl) {
        if (r >= 0 && r < p.swa_rows) {
          srow = r;
          ssc = __ldg(p.swa_scale + r);
        } else if (part == 0) {
          raise_error(&g_err_attn, CSA2_DEVERR_SWA_RANGE);
        }
      }
    }
    if (fslot) frow = entry_row_of_page(p.cache, page, e, &g_err_attn);
  }
  const bool fok = frow >= 0, sok = srow >= 0;
  // ---- the raw rows come by TMA into the staging area, off the load/store path: per warp,
  //      lanes 0, 8, 16, 24 gather the code and scale rows of 4 keys (held by lanes l, l+2,
  //      l+4, l+6; a key without a row reads row 0, unused), thread 0 the chunk's 32
  //      consecutive window rows (rows outside the array read as zero).  The start-up
  //      cluster phase (complete by now) orders warp 8's initialisation of mbarrier 9 (and
  //      7) before these copies and the waits below. ------------------------------------------
  tc::cluster_wait();
  {
    const int rowc = fok ? (int)frow : 0, base = lane & ~7;
    const int r0 = __shfl_sync(0xffffffffu, rowc, base), r1 = __shfl_sync(0xffffffffu, rowc, base + 2);
    const int r2 = __shfl_sync(0xffffffffu, rowc, base + 4), r3 = __shfl_sync(0xffffffffu, rowc, base + 6);
    if ((lane & 7) == 0) {
      const int g = warp * 4 + (lane >> 3);
      tc::tma_gather4(sKV + STG + g * 1024, &cmap, 0, r0, r1, r2, r3, &mbar[9]);
      tc::tma_gather4(sKV + STG + STG_CODES + g * 128, &smap, 0, r0, r1, r2, r3, &mbar[9]);
    }
    if (tid == 0 && p.swa_max > 0) {
      tc::tma_load_2d(sKV + STG + STG_CODES + STG_SCALES, &wmap, 0, wrow0, &mbar[9]);
      tc::tma_load_2d(sKV + STG + STG_CODES + STG_SCALES + STG_SWA / 2, &wmap, 256, wrow0, &mbar[9]);
    }
  }
  if (half == 0) ms.kc[fkey] = fok ? 1.f : __int_as_float(0x7fc00000);
  if (part == 0) ms.kc[skey] = sok ? ssc : __int_as_float(0x7fc00000);
  // ---- Q -> fp16 in place, scaled per head, while the rows are in flight.  Warp w converts
  //      heads w, w + 8, ..., lane l the head's 16-byte chunks l and l + 32. ------------------
  if (tc::mbar_wait_warp(&mbar[7], 0, MAX_POLL)) {
#pragma unroll
    for (int i = 0; i < HQ / (NW / 32); ++i) {
      const int h = warp + (NW / 32) * i;
      uint4* q0 = reinterpret_cast<uint4*>(sQ + tileoff(h, lane, QATOM));
      uint4* q1 = reinterpret_cast<uint4*>(sQ + tileoff(h, lane + 32, QATOM));
      const uint4 v0 = *q0, v1 = *q1;
      const int F = pow2_shift(__reduce_max_sync(0xffffffffu, max(bf16x8_absmax(v0), bf16x8_absmax(v1))) << 16);
      const float sc = exp2i(-F);
      *q0 = make_uint4(bf16x2_to_f16x2_scaled(v0.x, sc), bf16x2_to_f16x2_scaled(v0.y, sc),
                       bf16x2_to_f16x2_scaled(v0.z, sc), bf16x2_to_f16x2_scaled(v0.w, sc));
      *q1 = make_uint4(bf16x2_to_f16x2_scaled(v1.x, sc), bf16x2_to_f16x2_scaled(v1.y, sc),
                       bf16x2_to_f16x2_scaled(v1.z, sc), bf16x2_to_f16x2_scaled(v1.w, sc));
      if (lane == 0) ms.qfe[h] = (int8_t)F;
    }
  } else {
    raise_error(&g_err_attn, CSA2_DEVERR_TIMEOUT);
    ok_flag = 0;
  }
  // ---- raw rows into registers.  Thread (fkey, half) dequantises, in phase ph, dims
  //      [256 ph + 128 half, + 128) of its key: four 16-byte pieces of codes (32 dims each)
  //      and 8 scale bytes.  Step i reads piece (i + key) mod 4, which spreads a quarter warp
  //      over the banks.  Every thread has its bytes before any dequantised row overwrites
  //      the staging area. ------------------------------------------------------------------
  uint4 cw[8], wv[4];
  uint2 sv[2];
  const int rot_f = (lane >> 1) & 3, rot_s = part >> 1;
  if (!tc::mbar_wait_warp(&mbar[9], 0, MAX_POLL)) {
    if (lane == 0) raise_error(&g_err_attn, CSA2_DEVERR_TIMEOUT);
    ok_flag = 0;
  }
  {
    const uint8_t* cs = sKV + STG + fkey * 256 + half * 64;
#pragma unroll
    for (int ph = 0; ph < 2; ++ph) {
#pragma unroll
      for (int i = 0; i < 4; ++i) cw[4 * ph + i] = *reinterpret_cast<const uint4*>(cs + 128 * ph + 16 * ((i + rot_f) & 3));
      sv[ph] = *reinterpret_cast<const uint2*>(sKV + STG + STG_CODES + fkey * 32 + 16 * ph + 8 * half);
    }
    const uint8_t* ws = sKV + STG + STG_CODES + STG_SCALES + (part >> 2) * (STG_SWA / 2) + (tid >> 3) * 256 +
                        (part & 3) * 64;
#pragma unroll
    for (int i = 0; i < 4; ++i) wv[i] = *reinterpret_cast<const uint4*>(ws + 16 * ((i + rot_s) & 3));
  }
  // the chunk's P.V factor 2^-G: the largest key factor c of its keys (1 for an FP4 entry,
  // the row scale for a window row), maximised over the data warps
  {
    uint32_t mloc = fok ? __float_as_uint(1.f) : 0u;
    if (sok) mloc = max(mloc, __float_as_uint(fabsf(ssc)));
    mloc = __reduce_max_sync(0xffffffffu, mloc);
    if (lane == 0) ms.kvmax[warp] = mloc;
  }
  asm volatile("bar.sync 5, %0;" :: "n"(NW) : "memory");
  {
    uint32_t kvm = 0;
#pragma unroll
    for (int w = 0; w < NW / 32; ++w) kvm = max(kvm, ms.kvmax[w]);
    const int G = pfactor_shift(kvm);
    sG = exp2i(-G);
    if (tid == 0) {
      ms.ec_out[0] = exp2i(G);
      ms.ecs[tc::cluster_ctarank()][0] = exp2i(G);
      tc::fence_proxy_async_smem();             // ec_out is read by a bulk copy later
    }
  }
  // ---- dequantise into the K-major KV tile: the window rows (every dim), then the FP4 rows
  //      in two phases of 256 dims.  Once every warp has written phase 0 (mbarrier 5), the
  //      products over those dims start while phase 1 is written. ----------------------------
  if (sok) {
    // the row's E4M3 values, exact in fp16 (its scale is applied in float32 to its logit and
    // to its P.V weight)
#pragma unroll
    for (int i = 0; i < 4; ++i) {               // 16 bytes = 16 dims = 2 chunks
      const int c = (i + rot_s) & 3;
      const uint32_t words[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
      uint32_t o[8];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi)
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) o[wi * 2 + hi] = e4m3x2_to_f16x2((uint16_t)(words[wi] >> (16 * hi)));
      const int ch0 = part * 8 + c * 2;
      *reinterpret_cast<uint4*>(sKV + kvoff(skey, ch0)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(sKV + kvoff(skey, ch0 + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t) *reinterpret_cast<uint4*>(sKV + kvoff(skey, part * 8 + t)) = make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int ph = 0; ph < 2; ++ph) {
    const uint32_t sw[2] = {sv[ph].x, sv[ph].y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {               // 16 code bytes = 32 dims = scale groups 2j, 2j+1
      const int j = (i + rot_f) & 3;
      const int ch0 = 32 * ph + 16 * half + 4 * j;
      if (fok) {
        const uint32_t sc2 = j < 2 ? sw[0] : sw[1];
        const uint32_t sh = e4m3x2_to_f16x2((uint16_t)(sc2 >> (16 * (j & 1))));
        const uint32_t s0 = (sh & 0xffffu) * 0x10001u, s1 = (sh >> 16) * 0x10001u;
        const uint32_t words[4] = {cw[4 * ph + i].x, cw[4 * ph + i].y, cw[4 * ph + i].z, cw[4 * ph + i].w};
        uint32_t o[16];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi)
#pragma unroll
          for (int bi = 0; bi < 4; ++bi)
            o[wi * 4 + bi] = hmul2_u32(e2m1x2_to_f16x2((words[wi] >> (8 * bi)) & 0xffu), wi < 2 ? s0 : s1);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          *reinterpret_cast<uint4*>(sKV + kvoff(fkey, ch0 + t)) = make_uint4(o[4 * t], o[4 * t + 1], o[4 * t + 2], o[4 * t + 3]);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) *reinterpret_cast<uint4*>(sKV + kvoff(fkey, ch0 + t)) = make_uint4(0, 0, 0, 0);
      }
    }
    if (ph == 0) {                              // dims 0..255 of every key (and Q) are written
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&mbar[5]);
    }
  }
  }  // worker
  // ---- MMA1: S = Q K^T, the K steps over dims 0..255 once phase 0 is written, the rest
  //      after the block barrier below ---------------------------------------------------
  constexpr uint32_t id1 = tc::idesc_f16(64, NK, 0, 0, 0);
  auto issue_s = [&](uint32_t tmem_s, int ks0, int ks1) {
#pragma unroll 4
    for (int ks = ks0; ks < ks1; ++ks) {
      const uint64_t ad = tc::smem_desc_sw128(q_a + (ks >> 2) * QATOM + (ks & 3) * 32, 16, 1024);
      const uint64_t bd = tc::smem_desc_sw128(kv_a + (ks >> 2) * ATOM + (ks & 3) * 32, 16, 1024);
      tc::mma_f16_ss(tmem_s, ad, bd, id1, ks > 0);
    }
  };
  if (tid == ISSUER) {
    if (tc::mbar_wait(&mbar[5], 0, MAX_POLL)) {
      tc::fence_after_sync();
      if (ok_flag) issue_s(ms.tslot + COL_S, 0, DIM / 32);
    } else {
      raise_error(&g_err_attn, CSA2_DEVERR_TIMEOUT);
      ok_flag = 0;
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = ms.tslot;
  if (tid == ISSUER && ok_flag) {
    issue_s(tb + COL_S, DIM / 32, DIM / 16);
    tc::mma_commit(&mbar[0]);
    ok_flag = wait_mma(&mbar[0], 0) ? 1 : 0;
  }
  __syncthreads();
  tc::fence_after_sync();
  // Q is no longer read: the cluster may write merge blocks into this CTA's Q space.  Nothing
  // written before this point is read by another CTA, so the arrive need not release.
  tc::cluster_arrive_relaxed();
  // ---- softmax: a head's 160 keys are split over four threads: warps w and w ^ 4 take
  //      halves of 80, and within a warp threads t and t + 16 take 40 each -------------------
  const int sub = lane >> 4;                    // which 40-key (or 32-column) sub-range
  if (worker) {
  float e[40];
  if (ok_flag) {
    uint32_t r[40];
    tc::tmem_ld16x2_32<40>(tb + lane_base + COL_S + 80 * kh, r);
    tc::tmem_ld16x2_8<40>(tb + lane_base + COL_S + 80 * kh + 32, r + 32);
    tc::tmem_ld_wait();
    // logits in log2 units: the head's Q factor 2^F and each key's factor c applied
    const float4* kc4 = reinterpret_cast<const float4*>(ms.kc + 80 * kh + 40 * sub);
    const float lsc = p.scale_log2 * exp2i(ms.qfe[head]);
    float mx = -INFINITY;
#pragma unroll
    for (int j4 = 0; j4 < 10; ++j4) {
      const float4 v = kc4[j4];
      const float cv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int j = 4 * j4 + t;
        e[j] = cv[t] == cv[t] ? __uint_as_float(r[j]) * lsc * cv[t] : -INFINITY;
        mx = fmaxf(mx, e[j]);
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    if (lv) pmax[kh][head] = mx;
  }
  // the two warps of a lane quarter exchange their halves' maxima; both have read S, so
  // P may now overwrite it
  tc::fence_before_sync();
  asm volatile("bar.sync %0, 64;" :: "r"(1 + (warp & 3)) : "memory");
  tc::fence_after_sync();
  if (ok_flag) {
    const float m = fmaxf(pmax[0][head], pmax[1][head]);
    const float4* kc4 = reinterpret_cast<const float4*>(ms.kc + 80 * kh + 40 * sub);
    float l = 0.f;
    uint32_t pk[20];
#pragma unroll
    for (int j4 = 0; j4 < 10; ++j4) {
      const float4 v = kc4[j4];
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (m != -INFINITY) {
#pragma unroll
        for (int t = 0; t < 4; ++t) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(x[t]) : "f"(e[4 * j4 + t] - m));
      }
      l += (x[0] + x[1]) + (x[2] + x[3]);
      // the P.V weights p c 2^-G (<= 1); no key: 0
      const float w0 = v.x == v.x ? x[0] * v.x * sG : 0.f, w1 = v.y == v.y ? x[1] * v.y * sG : 0.f;
      const float w2 = v.z == v.z ? x[2] * v.z * sG : 0.f, w3 = v.w == v.w ? x[3] * v.w * sG : 0.f;
      const __half2 h01 = __floats2half2_rn(w0, w1), h23 = __floats2half2_rn(w2, w3);
      pk[2 * j4] = *reinterpret_cast<const uint32_t*>(&h01);
      pk[2 * j4 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
    }
    // P column = key / 2: this thread's 40 keys are columns [40 kh + 20 sub, + 20)
    tc::tmem_st16x2_16<20>(tb + lane_base + COL_S + 40 * kh, pk);
    tc::tmem_st16x2_4<20>(tb + lane_base + COL_S + 40 * kh + 16, pk + 16);
    tc::tmem_st_wait();
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    if (lv) psum[kh][head] = l;
  }
  }  // worker
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // ---- MMA2 quarters 0..2 back to back.  The epilogue of quarter q turns O / l into fp16 and
  //      places each owner's 16 heads x 128 dims as a 4 KB block (head row hh: 256 bytes,
  //      16-byte chunk cq at cq ^ hh): this CTA's own heads straight into its Q space (slot
  //      `rank`, block q), another owner's into the KV atoms that quarter q has finished
  //      reading, from where one thread sends it with a bulk copy into the owner's slot
  //      `rank` (completing on the owner's mbarrier 8).  Bulk copies keep the data off the
  //      load/store path the products share. ------------------------------------------------
  auto issue_quarter = [&](int q) {
    constexpr uint32_t id2 = tc::idesc_f16(64, 128, 0, 0, 1);
#pragma unroll
    for (int ks = 0; ks < NK / 16; ++ks) {
      const uint64_t bd = tc::smem_desc_sw128(kv_a + (2 * q) * ATOM + (2 * ks) * 1024, ATOM, 1024);
      tc::mma_f16_ts(tb + col_o(q), tb + COL_S + ks * 8, bd, id2, ks > 0);
    }
    tc::mma_commit(&mbar[1 + q]);
  };
  const int rank = (int)tc::cluster_ctarank();
  if (!worker) {                                // warp 8
    if (lane == 0 && ok_flag) {
      issue_quarter(0);
      issue_quarter(1);
      issue_quarter(2);
      // quarter 3 reuses quarter 0's columns once every data warp has read them
      if (tc::mbar_wait(&mbar[6], 0, MAX_POLL)) {
        tc::fence_after_sync();
        issue_quarter(3);
      } else {
        raise_error(&g_err_attn, CSA2_DEVERR_TIMEOUT);
      }
    }
    __syncwarp();
    tc::cluster_wait();                         // (every CTA has finished MMA1)
  }
  if (worker) {
    const float lh = psum[0][head] + psum[1][head];
    const bool anyh = ok_flag && lh > 0.f;
    const float li = anyh ? 1.f / lh : 0.f;
    bool ok = ok_flag != 0;
    const int owner = warp & 3, hh = head & 15;
    const bool remote = owner != rank;
    tc::cluster_wait();                         // every CTA has finished MMA1: Q spaces free
    if (lv && kh == 0) {
      const float2 v = anyh ? make_float2(fmaxf(pmax[0][head], pmax[1][head]), lh) : make_float2(-INFINITY, 0.f);
      if (remote) ms.rml_out[owner][hh] = v;
      else ms.rml[rank][hh] = v;
    }
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      if (ok) {
        ok = tc::mbar_wait_warp(&mbar[1 + q], 0, MAX_POLL);
        if (!ok && lane == 0) raise_error(&g_err_attn, CSA2_DEVERR_TIMEOUT);
      }
      tc::fence_after_sync();
      uint8_t* blk = remote ? sKV + (2 * q) * ATOM + owner * QBLK : sQ + rank * BLK + q * QBLK;
      uint32_t r[32];
      if (ok) {                                   // 16 heads x 64 columns per warp
        tc::tmem_ld16x2_32<32>(tb + lane_base + col_o(q) + 64 * kh, r);
        tc::tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t pk[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const __half2 hv = __floats2half2_rn(__uint_as_float(r[8 * i + 2 * t]) * li,
                                               __uint_as_float(r[8 * i + 2 * t + 1]) * li);
          pk[t] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        const int cq = 8 * kh + 4 * sub + i;
        *reinterpret_cast<uint4*>(blk + hh * 256 + ((cq ^ hh) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      if (q == 0) {
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&mbar[6]);
      }
      if (remote) {                               // warps owner and owner + 4 fill the block
        tc::fence_proxy_async_smem();
        asm volatile("bar.sync %0, 64;" :: "r"(1 + owner) : "memory");
        if (kh == 0 && lane == 0) {
          const uint32_t dmb = tc::mapa(smem_u32(&mbar[8]), owner);
          tc::bulk_copy_to_cluster(tc::mapa(q_a + rank * BLK + q * QBLK, owner), blk, QBLK, dmb);
          if (q == 0) {
            tc::bulk_copy_to_cluster(tc::mapa(smem_u32(&ms.rml[rank][0]), owner), &ms.rml_out[owner][0],
                                     HQ / NCH * 8, dmb);
            tc::bulk_copy_to_cluster(tc::mapa(smem_u32(&ms.ecs[rank][0]), owner), &ms.ec_out[0], 16, dmb);
          }
        }
      }
    }
    if (!ok && lane == 0) ok_flag = 0;
  }
  // the other chunks' blocks of this CTA's heads have landed once mbarrier 8 completes; its
  // own were written by its own warps before the barrier below.  Every CTA arrives on the
  // cluster's last phase only after that, so when the phase completes every bulk copy out of
  // every CTA's shared memory has finished and the CTAs may exit.
  if (!tc::mbar_wait_warp(&mbar[8], 0, MAX_POLL) && lane == 0) raise_error(&g_err_attn, CSA2_DEVERR_TIMEOUT);
  tc::cluster_arrive_relaxed();
  __syncthreads();
  // ---- merge: CTA r combines the 4 chunks of heads [16 r, 16 r + 16) from its Q space
  //      (slot c = chunk c) -------------------------------------------------------------
  if (p.early) pdl_wait();          // the first global write of the kernel comes next
  {
    float* wts = reinterpret_cast<float*>(&pmax[0][0]);       // [16][NCH] merge weights
    if (tid < 16) {
      const int h = 16 * rank + tid;
      float2 mv[NCH];
      float M = -INFINITY, L = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        mv[c] = ms.rml[c][tid];
        M = fmaxf(M, mv[c].x);
      }
      float w4[NCH];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        w4[c] = (mv[c].x == -INFINITY) ? 0.f : mv[c].y * exp2f(mv[c].x - M);
        L += w4[c];
      }
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) wts[tid * NCH + c] = w4[c] * inv * ms.ecs[c][0];   // x 2^G of chunk c
      if (p.lse) p.lse[(long long)b * HQ + h] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    // item = (head, 16-byte chunk); a warp covers 32 consecutive chunks of one head, two
    // 256-byte rows of quarter blocks
#pragma unroll
    for (int it = 0; it < 4 && worker; ++it) {
      const int idx = tid + it * NW;
      const int hh = idx >> 6, ch = idx & 63;
      const int h = 16 * rank + hh;
      const int off = (ch >> 4) * QBLK + hh * 256 + (((ch & 15) ^ hh) << 4);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const float wgt = wts[hh * NCH + c];
        const uint8_t* src = sQ + c * BLK;
        const uint4 u = *reinterpret_cast<const uint4*>(src + off);
        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&uw[t]));
          acc[2 * t] = fmaf(wgt, f.x, acc[2 * t]);
          acc[2 * t + 1] = fmaf(wgt, f.y, acc[2 * t + 1]);
        }
      }
      const long long ob = ((long long)b * HQ + h) * DIM + 8 * ch;
      if (p.out_f32) {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out) + ob);
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
        uint32_t pk[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          __nv_bfloat162 v2 = __floats2bfloat162_rn(acc[2 * t], acc[2 * t + 1]);
          pk[t] = *reinterpret_cast<uint32_t*>(&v2);
        }
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + ob) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
  }
  tc::cluster_wait();                           // every CTA has all of its blocks
  tc::fence_before_sync();
  __syncthreads();
  if (warp == NW / 32) tc::tmem_dealloc(tb, TMEM_COLS);
}

// Merge the chunk partials of (query b, head h).  Thread -> 4 dims.
template <int DIM>
__global__ void __launch_bounds__(DIM / 4) k_combine(const float* __restrict__ opart, const float2* __restrict__ ml,
                                                     int Hq, int nchunk, void* out, int out_f32, float* lse) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
  float M = -INFINITY;
  for (int c = 0; c < nchunk; ++c) M = fmaxf(M, ml[((long long)b * nchunk + c) * Hq + h].x);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int c = 0; c < nchunk; ++c) {
      const long long pi = ((long long)b * nchunk + c) * Hq + h;
      float2 v = ml[pi];
      if (v.x == -INFINITY) continue;
      float wgt = exp2f(v.x - M);
      L += v.y * wgt;
      float4 o = *reinterpret_cast<const float4*>(opart + pi * DIM + 4 * t);
      acc.x += o.x * wgt; acc.y += o.y * wgt; acc.z += o.z * wgt; acc.w += o.w * wgt;
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
  const long long ob = ((long long)b * Hq + h) * DIM + 4 * t;
  if (out_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + ob) = acc;
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 v = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + ob) = v;
  }
  if (lse && t == 0) lse[(long long)b * Hq + h] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
// CSA2_ATTN_LEGACY=1 selects the mma.sync kernel for every shape (kept for comparison
// measurements of the two tensor-core paths).
static bool attn_force_legacy() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("CSA2_ATTN_LEGACY");
    v = (e && e[0] == '1') ? 1 : 0;
  }
  return v == 1;
}

static int attn_nchunk(const csa2_attn_args& a) { return (a.k + a.swa_max + KC - 1) / KC; }

// chunks the workspace is laid out for: enough for either kernel
static int ws_chunks(const csa2_attn_args& a) { return attn_nchunk(a) > tca::NCH ? attn_nchunk(a) : tca::NCH; }

// partials (float32 for the mma.sync path; the tcgen05 path uses the first half as
// fp16), then (m, l) per chunk and head, then one arrival counter per query.
static size_t attn_counter_offset(const csa2_attn_args& a) {
  size_t n = (size_t)a.B * ws_chunks(a) * a.Hq;
  return ((n * a.cache.d * sizeof(float) + n * sizeof(float2)) + 255) & ~(size_t)255;
}

size_t attn_workspace_bytes(const csa2_attn_args& a) {
  return attn_counter_offset(a) + (size_t)a.B * sizeof(int);
}

template <int DIM, int MT>
static cudaError_t run_attn(const csa2_attn_args& a, AttnParams& ap, cudaStream_t st) {
  using C = ACfg<DIM, MT>;
  static bool attr_set = false;   // per instantiation; harmless to repeat
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_chunk<DIM, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(ap.nchunk, a.B);
  launch_k(k_attn_chunk<DIM, MT>, grid, ATHREADS, C::SMEM, st, ap);
  launch_k(k_combine<DIM>, dim3(a.B, a.Hq), DIM / 4, 0, st, ap.opart, ap.ml, a.Hq, ap.nchunk, a.out,
                                                     a.out_dtype == CSA2_F32, a.lse);
  return cudaGetLastError();
}

static cudaError_t run_attn_tc(const csa2_attn_args& a, AttnParams& ap, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, tca::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  ap.nchunk = tca::NCH;
  CUtensorMap qmap, cmap, smap, wmap;            // q as [B * 64 heads][512] bf16, 64 heads x 64 dims boxes;
                                                // code / scale rows (one-row boxes, gathered 4 at a time);
                                                // window rows (32 rows x 256 bytes)
  const long long rows = (long long)a.cache.num_pages * 64;
  if (!bf16_map(&qmap, a.q, (long long)a.B * tca::HQ, tca::DIM, tca::HQ) ||
      !u8_map(&cmap, a.cache.codes, rows, tca::DIM / 2, tca::DIM / 2, 1) ||
      !u8_map(&smap, a.cache.scales, rows, tca::DIM / 16, tca::DIM / 16, 1))
    return cudaErrorInvalidValue;
  if (a.swa_max > 0) {
    if (!u8_map(&wmap, a.swa, a.swa_rows, tca::DIM, 256, tca::KW)) return cudaErrorInvalidValue;
  } else {
    wmap = cmap;                                // not read
  }
  launch_k(k_attn_tc, dim3(tca::NCH, a.B), tca::THREADS, tca::SMEM, st, ap, qmap, cmap, smap, wmap);
  return cudaGetLastError();
}

// One CTA waiting on an mbarrier that nothing arrives on, for at most `polls` polls: the
// failure path of every bounded wait (error bit, no trap, the kernel returns).
__global__ void k_selftest_wait(int polls) {
  pdl_wait();
  __shared__ uint64_t mb;
  if (threadIdx.x == 0) tc::mbar_init(&mb, 1);
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&mb, 0, (uint32_t)polls)) raise_error(&g_err_attn, CSA2_DEVERR_TIMEOUT);
}

cudaError_t launch_selftest_wait(int polls, cudaStream_t st) {
  return launch_k(k_selftest_wait, 1, 32, 0, st, polls);
}

cudaError_t launch_attn(const csa2_attn_args& a, void* ws, cudaStream_t st) {
  if (a.B == 0) return cudaSuccess;
  AttnParams ap{};
  ap.q = a.q;
  ap.cache = a.cache;
  ap.seq_of = a.seq_of;
  ap.topk = a.topk;
  ap.topk_len = a.topk_len;
  ap.k = a.k;
  ap.swa = a.swa;
  ap.swa_scale = a.swa_scale;
  ap.swa_rows = a.swa_rows;
  ap.swa_start = a.swa_start;
  ap.swa_len = a.swa_len;
  ap.swa_max = a.swa_max;
  ap.Hq = a.Hq;
  ap.nchunk = attn_nchunk(a);
  ap.scale_log2 = a.softmax_scale * LOG2E;
  size_t n = (size_t)a.B * ws_chunks(a) * a.Hq;
  ap.opart = static_cast<float*>(ws);
  ap.ml = reinterpret_cast<float2*>(static_cast<float*>(ws) + n * a.cache.d);
  ap.opart16 = static_cast<__half*>(ws);
  ap.counter = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + attn_counter_offset(a));
  ap.out = a.out;
  ap.out_f32 = a.out_dtype == CSA2_F32;
  ap.lse = a.lse;
  ap.early = a.inputs_ready != 0;
  const int mt = (a.Hq + 15) / 16;
  if (a.cache.d == 512 && a.Hq == 64 && a.k <= tca::NCH * tca::KT && a.swa_max <= tca::NCH * tca::KW &&
      (long long)a.cache.num_pages * 64 < (1ll << 31) && tensor_map_encoder() != nullptr && !attn_force_legacy())
    return run_attn_tc(a, ap, st);
  if (a.cache.d == 512) {
    if (mt == 4) return run_attn<512, 4>(a, ap, st);
    if (mt == 2) return run_attn<512, 2>(a, ap, st);
    return run_attn<512, 1>(a, ap, st);
  }
  if (mt == 4) return run_attn<128, 4>(a, ap, st);
  if (mt == 2) return run_attn<128, 2>(a, ap, st);
  return run_attn<128, 1>(a, ap, st);
}

uint32_t read_clear_error_attn() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_attn, sizeof(v));
  cudaMemcpyToSymbol(g_err_attn, &z, sizeof(z));
  return v;
}

}  // namespace csa2
