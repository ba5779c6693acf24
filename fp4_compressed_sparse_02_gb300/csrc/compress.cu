// Non-overlapping compressor + RoPE + FP4 (E2M1, E4M3 per 16 channels) quantiser and
// the indexer-K projection.
//
// "DeepSeek-V4.1-Flash deep dive", section 2: C = H.W_KV, Z = H.W_Z.
// Section 3.1: every m tokens -> one Main KV entry, no overlap, no absolute PE; Indexer
// K is projected from Main KV.  Section 3.4: RoPE before quantisation; E2M1 values with
// one E4M3 scale per 16 channels.
//
// Kernels
//   k_project     C|Z = H . [W_kv | W_z] in float32 (split-K partials, no atomics)
//   k_quant       per group of m rows: sum the split-K partials, per-channel softmax
//                 pooling, RoPE, amax/6 -> E4M3 scale, E2M1 codes, paged store
//   k_index_k     idx_k = bf16(dequant(entry) . W_ik), re-reading the stored entry
#include "common.cuh"
#include "internal.h"

namespace csa2 {

CSA2_DEFINE_ERROR_WORD(g_err_compress);

// ---------------------------------------------------------------------------------
// Projection GEMM: out[s][t][n] = sum_{k in split s} H[t][k] * W[k][n]
//   n <  d : W = W_kv,   n >= d : W = W_z (column n - d)
// 64x64 tile, 32-deep K slices, 256 threads, 4x4 outputs per thread, float32 FMA.
// ---------------------------------------------------------------------------------
constexpr int PBM = 64, PBN = 64, PBK = 32;

template <typename HT>
__device__ __forceinline__ float load_h(const HT* p);
template <>
__device__ __forceinline__ float load_h<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_h<uint16_t>(const uint16_t* p) {
  return bf16_bits_to_f32(__ldg(p));
}

template <typename HT>
__global__ void __launch_bounds__(256) k_project(const HT* __restrict__ H,
                                                 const uint16_t* __restrict__ Wkv,
                                                 const uint16_t* __restrict__ Wz, float* __restrict__ out,
                                                 int T, int d_model, int d, int N, int k_per_split) {
  pdl_wait();
  __shared__ float As[PBK][PBM + 4];
  __shared__ float Bs[PBK][PBN + 4];
  const int tid = threadIdx.x;
  const int n0 = blockIdx.x * PBN;
  const int t0 = blockIdx.y * PBM;
  const int s = blockIdx.z;
  const int kbeg = s * k_per_split;
  const int kend = min(d_model, kbeg + k_per_split);
  const uint16_t* W = (n0 < d) ? Wkv : Wz;
  const int wn0 = (n0 < d) ? n0 : n0 - d;
  const int tx = tid % 16, ty = tid / 16;
  float acc[4][4] = {};
  for (int k0 = kbeg; k0 < kend; k0 += PBK) {
    // H tile: 64 rows x 32 k -> As[k][row]
    for (int i = tid; i < PBM * PBK; i += 256) {
      int r = i / PBK, kk = i % PBK;
      int t = t0 + r, kg = k0 + kk;
      As[kk][r] = (t < T && kg < kend) ? load_h<HT>(H + (long long)t * d_model + kg) : 0.0f;
    }
    // W tile: 32 k x 64 n -> Bs[k][n]
    for (int i = tid; i < PBK * PBN; i += 256) {
      int kk = i / PBN, nn = i % PBN;
      int kg = k0 + kk;
      Bs[kk][nn] = (kg < kend) ? bf16_bits_to_f32(__ldg(W + (long long)kg * d + wn0 + nn)) : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < PBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* o = out + (long long)s * T * N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int t = t0 + ty * 4 + i;
    if (t >= T) continue;
    float4 v = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4*>(o + (long long)t * N + n0 + tx * 4) = v;
  }
}

// ---------------------------------------------------------------------------------
// Projection for few rows (decode append, T <= 64): CTA = (64 output columns, one K
// slice of ks rows).  The whole W slice and H slice are loaded with 16-byte loads in
// one go (no K loop), then each thread accumulates T/4 rows of one column.
// ---------------------------------------------------------------------------------
constexpr int SMALL_T = 64;

template <typename HT>
__device__ __forceinline__ void load_h8(const HT* p, float* v);
template <>
__device__ __forceinline__ void load_h8<uint16_t>(const uint16_t* p, float* v) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { v[2 * i] = __uint_as_float(w[i] << 16); v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u); }
}
template <>
__device__ __forceinline__ void load_h8<float>(const float* p, float* v) {
  float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename HT>
__global__ void __launch_bounds__(256) k_project_small(const HT* __restrict__ H, const uint16_t* __restrict__ Wkv,
                                                       const uint16_t* __restrict__ Wz, float* __restrict__ out,
                                                       int T, int d_model, int d, int N, int ks) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t psm[];
  uint16_t* Ws = reinterpret_cast<uint16_t*>(psm);                 // [ks][64] bf16
  float* Hs = reinterpret_cast<float*>(psm + (size_t)ks * 128);      // [T][ks]
  const int tid = threadIdx.x;
  const int n0 = blockIdx.x * 64, s = blockIdx.y;
  const int k0 = s * ks;
  const uint16_t* W = (n0 < d) ? Wkv : Wz;
  const int wn0 = (n0 < d) ? n0 : n0 - d;
  for (int i = tid; i < ks * 8; i += 256) {
    const int r = i >> 3, c8 = i & 7;
    *reinterpret_cast<uint4*>(Ws + r * 64 + c8 * 8) =
        __ldg(reinterpret_cast<const uint4*>(W + (long long)(k0 + r) * d + wn0 + c8 * 8));
  }
  for (int i = tid; i < T * (ks / 8); i += 256) {
    const int t = i / (ks / 8), c8 = i % (ks / 8);
    float v[8];
    load_h8<HT>(H + (long long)t * d_model + k0 + c8 * 8, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) Hs[t * ks + c8 * 8 + j] = v[j];
  }
  __syncthreads();
  const int c = tid & 63, rg = tid >> 6;
  float acc[SMALL_T / 4];
#pragma unroll
  for (int i = 0; i < SMALL_T / 4; ++i) acc[i] = 0.f;
  for (int k = 0; k < ks; ++k) {
    const float w = bf16_bits_to_f32(Ws[k * 64 + c]);
#pragma unroll
    for (int i = 0; i < SMALL_T / 4; ++i)
      if (rg + 4 * i < T) acc[i] = fmaf(Hs[(rg + 4 * i) * ks + k], w, acc[i]);
  }
  float* o = out + (long long)s * T * N + n0 + c;
#pragma unroll
  for (int i = 0; i < SMALL_T / 4; ++i)
    if (rg + 4 * i < T) o[(long long)(rg + 4 * i) * N] = acc[i];
}

// Few-row projection on the tensor cores (bf16 H): mma.sync m16n8k16, fp32 accumulate.
// CTA = (64 output columns, one K slice of ks rows, ks % 16 == 0), 4 warps; warp w owns
// rows [16w, 16w + 16).  Shared rows are padded to an odd number of 16-byte chunks so the
// ldmatrix row addresses fall in distinct banks.
__global__ void __launch_bounds__(128) k_project_mma(const uint16_t* __restrict__ H, const uint16_t* __restrict__ Wkv,
                                                     const uint16_t* __restrict__ Wz, float* __restrict__ out, int T,
                                                     int d_model, int d, int N, int ks) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t psm[];
  const int HS = ks * 2 + 16, WS = 64 * 2 + 16;
  uint8_t* Hs = psm;                       // [64][HS]
  uint8_t* Ws = psm + 64 * HS;             // [ks][WS]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n0 = blockIdx.x * 64, s = blockIdx.y, k0 = s * ks;
  const uint16_t* W = (n0 < d) ? Wkv : Wz;
  const int wn0 = (n0 < d) ? n0 : n0 - d;
  for (int i = tid; i < ks * 8; i += 128) {
    const int r = i >> 3, c8 = i & 7;
    *reinterpret_cast<uint4*>(Ws + r * WS + c8 * 16) =
        __ldg(reinterpret_cast<const uint4*>(W + (long long)(k0 + r) * d + wn0 + c8 * 8));
  }
  const int kc = ks / 8;
  for (int i = tid; i < 64 * kc; i += 128) {
    const int t = i / kc, c8 = i % kc;
    *reinterpret_cast<uint4*>(Hs + t * HS + c8 * 16) =
        (t < T) ? __ldg(reinterpret_cast<const uint4*>(H + (long long)t * d_model + k0 + c8 * 8)) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (16 * warp >= T) return;
  float acc[8][4];
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  const int mi = lane >> 3, r8 = lane & 7;
  const uint32_t hs = smem_u32(Hs), ws = smem_u32(Ws);
  for (int kk = 0; kk < ks; kk += 16) {
    uint32_t a0, a1, a2, a3;
    ldmatrix_x4(a0, a1, a2, a3, hs + (16 * warp + (lane & 15)) * HS + (kk + (lane >> 4) * 8) * 2);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(b0, b1, b2, b3, ws + (kk + (mi & 1) * 8 + r8) * WS + (np * 16 + (mi >> 1) * 8) * 2);
      mma_bf16_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
    }
  }
  const int g = lane >> 2, c = lane & 3;
  const int r0 = 16 * warp + g, r1 = r0 + 8;
  float* o = out + (long long)s * T * N + n0 + 2 * c;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    if (r0 < T) *reinterpret_cast<float2*>(o + (long long)r0 * N + 8 * t) = make_float2(acc[t][0], acc[t][1]);
    if (r1 < T) *reinterpret_cast<float2*>(o + (long long)r1 * N + 8 * t) = make_float2(acc[t][2], acc[t][3]);
  }
}

// K slices for the tensor-core few-row projection: multiples of 16 rows, ~128 CTAs.
static int mma_splits(int d_model, int N) {
  int best = 1;
  for (int s = 1; s <= 64; ++s) {
    if (d_model % s || (d_model / s) % 16) continue;
    const size_t smem = (size_t)64 * ((d_model / s) * 2 + 16) + (size_t)(d_model / s) * 144;
    if (smem > 160 * 1024) continue;
    best = s;
    if ((N / 64) * s >= 128) break;
  }
  return best;
}

// ---------------------------------------------------------------------------------
// Pool + RoPE + quantise.  One thread per 16-channel group of one entry.
//   C row t, channel c: sum_{s < nsplit} Cp[s*split_stride + t*ldc + c]
//   Z likewise from Zp (m > 1 only).
// ---------------------------------------------------------------------------------
struct QuantParams {
  const float* Cp;
  const float* Zp;
  long long split_stride;
  int nsplit;
  int ldc;
  int G, m, d;
  int d_rope, rope_max_pos;
  const float* rope_cos;
  const float* rope_sin;
  const int* pos;
  const int* seq;
  const int* entry;
  csa2_cache cache;
  float* y_out;
};

__device__ __forceinline__ void load16(const float* p, float* v) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 x = q[i];
    v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
  }
}

__device__ __forceinline__ void load16_sum(const float* p, long long stride, int nsplit, float* v) {
  load16(p, v);
  int s = 1;
  for (; s + 3 < nsplit; s += 4) {   // four partial rows in flight
    float w0[16], w1[16], w2[16], w3[16];
    load16(p + s * stride, w0);
    load16(p + (s + 1) * stride, w1);
    load16(p + (s + 2) * stride, w2);
    load16(p + (s + 3) * stride, w3);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = (((v[i] + w0[i]) + w1[i]) + w2[i]) + w3[i];
  }
  for (; s < nsplit; ++s) {
    float w[16];
    load16(p + s * stride, w);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += w[i];
  }
}

// Group q (16 channels) of entry g: pooled row, RoPE at position ps, FP4 codes and scale into
// entry en of sequence sq; with deq, also the dequantised values (code x scale, float32) into
// deq[16 q ..].
__device__ __forceinline__ void quant_group_at(const QuantParams& p, long long g, int q, float* deq, int ps, int sq,
                                               int en) {
  const int c0 = q * 16;
  float y[16];
  if (p.m == 1) {
    load16_sum(p.Cp + g * p.ldc + c0, p.split_stride, p.nsplit, y);
  } else {
    // per-channel softmax over the m tokens of the group (float32)
    float zmax[16], den[16], num[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) { zmax[i] = -INFINITY; den[i] = 0.f; num[i] = 0.f; }
    for (int j = 0; j < p.m; ++j) {
      float z[16];
      load16_sum(p.Zp + (g * p.m + j) * p.ldc + c0, p.split_stride, p.nsplit, z);
#pragma unroll
      for (int i = 0; i < 16; ++i) zmax[i] = fmaxf(zmax[i], z[i]);
    }
    for (int j = 0; j < p.m; ++j) {
      float z[16], c[16];
      load16_sum(p.Zp + (g * p.m + j) * p.ldc + c0, p.split_stride, p.nsplit, z);
      load16_sum(p.Cp + (g * p.m + j) * p.ldc + c0, p.split_stride, p.nsplit, c);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float e = expf(z[i] - zmax[i]);
        den[i] += e;
        num[i] = fmaf(e, c[i], num[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = num[i] / den[i];
  }
  // RoPE on channels [d - d_rope, d): pairs (2i, 2i+1) of that slice
  const int rb = p.d - p.d_rope;
  if (p.d_rope > 0 && c0 >= rb) {
    if (ps < 0 || ps >= p.rope_max_pos) {
      raise_error(&g_err_compress, CSA2_DEVERR_POS);
    } else {
      const int half = p.d_rope / 2;
      const float* ct = p.rope_cos + (long long)ps * half + (c0 - rb) / 2;
      const float* st = p.rope_sin + (long long)ps * half + (c0 - rb) / 2;
#pragma unroll
      for (int i = 0; i < 8; ++i) rope_pair(y[2 * i], y[2 * i + 1], __ldg(ct + i), __ldg(st + i));
    }
  }
  if (p.y_out) {
    float4* yo = reinterpret_cast<float4*>(p.y_out + g * p.d + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) yo[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
  }
  uint32_t w0, w1, sbyte;
  fp4_group16(y, w0, w1, sbyte);
  if (deq) {                                          // as the indexer-K projection reads it back
    const float sc = e4m3_to_f32((uint8_t)sbyte);
    const uint32_t wd[2] = {w0, w1};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t h2 = e2m1x2_to_f16x2((wd[i >> 2] >> (8 * (i & 3))) & 0xffu);
      const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
      deq[c0 + 2 * i] = __low2float(hv) * sc;
      deq[c0 + 2 * i + 1] = __high2float(hv) * sc;
    }
  }
  long long row = entry_row(p.cache, sq, en, &g_err_compress);
  if (row < 0) return;
  uint2* cd = reinterpret_cast<uint2*>(p.cache.codes + row * (p.d / 2) + q * 8);
  *cd = make_uint2(w0, w1);
  p.cache.scales[row * (p.d / 16) + q] = (uint8_t)sbyte;
}

__device__ __forceinline__ void quant_group(const QuantParams& p, long long g, int q, float* deq) {
  const int ps = (p.d_rope > 0 && q * 16 >= p.d - p.d_rope) ? __ldg(p.pos + g) : 0;
  quant_group_at(p, g, q, deq, ps, __ldg(p.seq + g), __ldg(p.entry + g));
}

__global__ void __launch_bounds__(256) k_quant(QuantParams p) {
  pdl_wait();
  pdl_trigger();
  const int gpr = p.d / 16;                           // 16-channel groups per entry
  long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  long long g = gid / gpr;
  const int q = (int)(gid % gpr);
  if (g >= p.G) return;
  quant_group(p, g, q, nullptr);
}

// ---------------------------------------------------------------------------------
// Indexer K: idx_k[e][j] = bf16( sum_c dequant(e)[c] * W_ik[c][j] ).  CTA = E entries,
// 8 warps; warp w owns rows c in [w*d/8, (w+1)*d/8) of W_ik (loaded once, 16 rows at a
// time, for all E entries), lane l owns columns [l*cpl, l*cpl + cpl).  The 8 warp
// partials are summed in warp order, so the result does not depend on scheduling.
// ---------------------------------------------------------------------------------
template <int E, int DIK>
__device__ __forceinline__ void index_k_product(const csa2_cache& cache, const long long* rows, const float* deq,
                                                float* part, const uint16_t* __restrict__ Wik);

template <int E, int DIK>
__global__ void __launch_bounds__(256) k_index_k(csa2_cache cache, const int* __restrict__ seq,
                                                 const int* __restrict__ entry, int G,
                                                 const uint16_t* __restrict__ Wik) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float ik_sm[];
  const int d = cache.d;
  float* deq = ik_sm;                            // [E][d]
  float* part = ik_sm + E * d;                   // [8][E][DIK]
  __shared__ long long rows[E];
  const int tid = threadIdx.x;
  const int g0 = blockIdx.x * E;
  if (tid < E) {
    const int g = g0 + tid;
    rows[tid] = (g < G) ? entry_row(cache, __ldg(seq + g), __ldg(entry + g), &g_err_compress) : -1;
  }
  __syncthreads();
  for (int i = tid; i < E * d / 2; i += 256) {
    const int e = i / (d / 2), cb = i % (d / 2);
    const long long r = rows[e];
    float v0 = 0.f, v1 = 0.f;
    if (r >= 0) {
      const uint32_t byte = cache.codes[r * (d / 2) + cb];
      const float sc = e4m3_to_f32(cache.scales[r * (d / 16) + (2 * cb) / 16]);
      const uint32_t h2 = e2m1x2_to_f16x2(byte);
      const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
      v0 = __low2float(hv) * sc;
      v1 = __high2float(hv) * sc;
    }
    deq[e * d + 2 * cb] = v0;
    deq[e * d + 2 * cb + 1] = v1;
  }
  __syncthreads();
  index_k_product<E, DIK>(cache, rows, deq, part, Wik);
}

// idx_k of E entries from their dequantised rows deq[E][d] (shared memory), with `part`
// [8][E][DIK] floats of shared scratch; 256 threads.
template <int E, int DIK>
__device__ __forceinline__ void index_k_product(const csa2_cache& cache, const long long* rows, const float* deq,
                                                float* part, const uint16_t* __restrict__ Wik) {
  constexpr int CPL = DIK / 32;
  const int d = cache.d;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float acc[E][CPL];
#pragma unroll
  for (int e = 0; e < E; ++e)
#pragma unroll
    for (int j = 0; j < CPL; ++j) acc[e][j] = 0.f;
  const int rows_per_warp = d / 8;
  const int cbase = warp * rows_per_warp;
  for (int c0 = 0; c0 < rows_per_warp; c0 += 16) {
    float w[16][CPL];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
      const uint16_t* wp = Wik + (long long)(cbase + c0 + rr) * DIK + lane * CPL;
      if constexpr (CPL == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(wp));
        w[rr][0] = __uint_as_float(u.x << 16); w[rr][1] = __uint_as_float(u.x & 0xffff0000u);
        w[rr][2] = __uint_as_float(u.y << 16); w[rr][3] = __uint_as_float(u.y & 0xffff0000u);
      } else {
        const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(wp));
        w[rr][0] = __uint_as_float(u << 16); w[rr][1] = __uint_as_float(u & 0xffff0000u);
      }
    }
#pragma unroll
    for (int rr = 0; rr < 16; ++rr)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float x = deq[e * d + cbase + c0 + rr];
#pragma unroll
        for (int j = 0; j < CPL; ++j) acc[e][j] = fmaf(x, w[rr][j], acc[e][j]);
      }
  }
#pragma unroll
  for (int e = 0; e < E; ++e)
#pragma unroll
    for (int j = 0; j < CPL; ++j) part[(warp * E + e) * DIK + lane * CPL + j] = acc[e][j];
  __syncthreads();
  if (cache.idx_k_dtype == CSA2_FP8E4M3) {
    // the compressed form: warp e quantises entry e's bf16 row (lane l: columns l*CPL ..)
    for (int e = warp; e < E; e += 8) {
      const long long r = rows[e];
      if (r < 0) continue;
      float v[CPL];
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        float sum = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) sum += part[(w8 * E + e) * DIK + lane * CPL + j];
        v[j] = __bfloat162float(__float2bfloat16_rn(sum));
      }
      fp8_row_store<CPL>(v, cache.idx_k8 + r * DIK + lane * CPL, cache.idx_k8_scale + r);
    }
    return;
  }
  for (int i = tid; i < E * DIK; i += 256) {
    const int e = i / DIK, j = i % DIK;
    const long long r = rows[e];
    if (r < 0) continue;
    float sum = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) sum += part[(w8 * E + e) * DIK + j];
    const __nv_bfloat16 hb = __float2bfloat16_rn(sum);
    cache.idx_k[r * DIK + j] = *reinterpret_cast<const uint16_t*>(&hb);
  }
}

// The decode append's two steps in one launch, one CTA per entry: its 16-channel groups are
// quantised (as k_quant) by the first d/16 threads, which also leave the dequantised row in
// shared memory; then the indexer-K projection of that row (as k_index_k).
template <int DIK>
__global__ void __launch_bounds__(256) k_quant_index_k(QuantParams p, const uint16_t* __restrict__ Wik) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float qk_sm[];
  float* deq = qk_sm;                            // [d]
  float* part = qk_sm + p.d;                     // [8][DIK]
  __shared__ long long rows[1];
  const long long g = blockIdx.x;
  if (threadIdx.x < p.d / 16) quant_group(p, g, threadIdx.x, deq);
  if (threadIdx.x == 0) rows[0] = entry_row(p.cache, __ldg(p.seq + g), __ldg(p.entry + g), &g_err_compress);
  __syncthreads();
  index_k_product<1, DIK>(p.cache, rows, deq, part, Wik);
}

template <int DIK>
static cudaError_t launch_quant_index_k(const QuantParams& qp, const uint16_t* Wik, cudaStream_t st) {
  const size_t sm = ((size_t)qp.d + 8 * DIK) * sizeof(float);
  return launch_k(k_quant_index_k<DIK>, (unsigned)qp.G, 256, sm, st, qp, Wik);
}

// ---------------------------------------------------------------------------------
// The decode-time append at compression ratio m: one new token per CTA.  The token's C and
// Z rows (the summed projection partials) go to slot t % m of its sequence's pending group
// (pend[s]: C rows [m][d], then Z rows [m][d]); the token that completes the group (t % m
// == m - 1) then pools the group's m rows, applies RoPE at its own position t, quantises
// and writes entry t / m, and projects its indexer K.  At m = 1 every token completes its
// group and reads its row straight from the partials.
// ---------------------------------------------------------------------------------
struct AppendParams {
  QuantParams q;                                 // partials of the B tokens, RoPE, cache
  const int* tok_pos;
  float* pend;                                   // [num_seqs][2][m][d] (m > 1)
  float* y_out;                                  // [B][d] or null
};

template <int DIK>
__global__ void __launch_bounds__(256) k_append_quant_index_k(AppendParams ap, const uint16_t* __restrict__ Wik) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float qk_sm[];
  float* deq = qk_sm;                            // [d]
  float* part = qk_sm + ap.q.d;                  // [8][DIK]
  __shared__ long long rows[1];
  const int b = blockIdx.x, tid = threadIdx.x, d = ap.q.d, m = ap.q.m;
  const int s = __ldg(ap.q.seq + b), t = __ldg(ap.tok_pos + b);
  if (s < 0 || s >= ap.q.cache.num_seqs || t < 0) {           // the same for the whole CTA
    if (tid == 0) raise_error(&g_err_compress, t < 0 ? CSA2_DEVERR_POS : CSA2_DEVERR_SEQ);
    return;
  }
  const int j = t % m, g = t / m;
  QuantParams qp = ap.q;
  qp.y_out = ap.y_out ? ap.y_out + (long long)b * d : nullptr;
  if (m == 1) {
    qp.Cp = ap.q.Cp + (long long)b * ap.q.ldc;   // this token's partials (group 0 below)
  } else {
    float* grp = ap.pend + (long long)s * 2 * m * d;
    for (int i = tid; i < d; i += blockDim.x) {
      const float* cp = ap.q.Cp + (long long)b * ap.q.ldc + i;
      const float* zp = ap.q.Zp + (long long)b * ap.q.ldc + i;
      float c = cp[0], z = zp[0];
      for (int k = 1; k < ap.q.nsplit; ++k) {
        c += cp[k * ap.q.split_stride];
        z += zp[k * ap.q.split_stride];
      }
      grp[(long long)j * d + i] = c;
      grp[(long long)(m + j) * d + i] = z;
    }
    if (j < m - 1) return;                       // the group is not complete yet
    __syncthreads();                             // the group's rows, written by this CTA, are visible
    qp.Cp = grp;
    qp.Zp = grp + (long long)m * d;
    qp.split_stride = 0;
    qp.nsplit = 1;
    qp.ldc = d;
  }
  if (tid < d / 16) quant_group_at(qp, 0, tid, Wik ? deq : nullptr, t, s, g);
  if (Wik == nullptr) return;
  if (tid == 0) rows[0] = entry_row(qp.cache, s, g, &g_err_compress);
  __syncthreads();
  index_k_product<1, DIK>(qp.cache, rows, deq, part, Wik);
}

template <int E, int DIK>
static cudaError_t launch_index_k(const csa2_compress_args& a, int G, cudaStream_t st) {
  const size_t sm = ((size_t)E * a.cache.d + 8 * E * DIK) * sizeof(float);
  static size_t attr_bytes = 0;                 // opt-in above 48 KB, raised when needed
  if (sm > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(k_index_k<E, DIK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    attr_bytes = sm;
  }
  return launch_k(k_index_k<E, DIK>, (G + E - 1) / E, 256, sm, st, a.cache, a.seq, a.entry, G, a.W_ik);
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
// K slices for the few-row projection: aim at ~128 CTAs with slices that are a multiple of
// 8 rows and small enough for shared memory (ks * (128 + 4*T) bytes).
static int small_splits(int T, int d_model, int N) {
  int best = 1;
  for (int s = 1; s <= 64; ++s) {
    if (d_model % s || (d_model / s) % 8) continue;
    const size_t smem = (size_t)(d_model / s) * (128 + 4 * T);
    if (smem > 160 * 1024) continue;
    best = s;
    if ((N / 64) * s >= 128) break;
  }
  return best;
}

static bool use_small(const csa2_compress_args& a) { return a.T <= SMALL_T; }

static int pick_splits(int T, int d_model, int N) {
  // enough CTAs to cover the GPU when T is small (decode append): split K so that
  // (tiles x splits) >= ~2 waves of 152 SMs, keeping each split >= 128 deep.
  long long tiles = (long long)((T + PBM - 1) / PBM) * (N / PBN);
  int s = 1;
  while (tiles * s < 304 && d_model / (s * 2) >= 128) s *= 2;
  return s;
}

// The indexer-K projection of the G new entries (when W_ik is given) after k_quant: the
// tensor-core kernel, else 8 entries per CTA (fewer than 2,048 entries without the tensor-core
// kernel take k_quant_index_k instead).
static cudaError_t launch_index_k_any(const csa2_compress_args& a, int G, cudaStream_t st) {
  if (!a.W_ik || G <= 0) return cudaSuccess;
  if (index_k_tc_supported(a, G)) return launch_index_k_tc(a, G, st);
  return a.cache.d_ik == 128 ? launch_index_k<8, 128>(a, G, st) : launch_index_k<8, 64>(a, G, st);
}

// bytes of the unfused projection's output (its split-K partials)
static size_t project_ws_bytes(const csa2_compress_args& a) {
  int N = a.cache.d * (a.m > 1 ? 2 : 1);
  if (project_tc_supported(a)) return (size_t)a.T * N * sizeof(float);
  int s = !use_small(a) ? pick_splits(a.T, a.d_model, N)
          : (a.h_dtype == CSA2_BF16 ? mma_splits(a.d_model, N) : small_splits(a.T, a.d_model, N));
  return (size_t)s * a.T * N * sizeof(float);
}

size_t compress_workspace_bytes(const csa2_compress_args& a) {
  if (!a.W_kv) return 0;
  if (project_tc_fused(a)) return 0;
  return project_ws_bytes(a);
}

// C|Z = H.[W_kv|W_z] of the a.T rows into `out` (float32 split-K partials, no pooling); sets
// the partial layout of qp.
static cudaError_t project_rows(const csa2_compress_args& a, float* out, cudaStream_t st, QuantParams& qp) {
  const int d = a.cache.d;
  int N = d * (a.m > 1 ? 2 : 1);
  int s;
  if (project_tc_supported(a)) {
    s = 1;
    cudaError_t e = launch_project_tc(a, out, false, st);
    if (e != cudaSuccess) return e;
  } else if (use_small(a) && a.h_dtype == CSA2_BF16) {
    s = mma_splits(a.d_model, N);
    const int ks = a.d_model / s;
    const size_t sm = (size_t)64 * (ks * 2 + 16) + (size_t)ks * 144;
    cudaError_t e = cudaFuncSetAttribute(k_project_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    launch_k(k_project_mma, dim3(N / 64, s), 128, sm, st, static_cast<const uint16_t*>(a.H), a.W_kv, a.W_z, out, a.T,
                                                    a.d_model, d, N, ks);
  } else if (use_small(a)) {
    s = small_splits(a.T, a.d_model, N);
    const int ks = a.d_model / s;
    const size_t sm = (size_t)ks * (128 + 4 * a.T);
    cudaError_t e;
    if (a.h_dtype == CSA2_F32) {
      e = cudaFuncSetAttribute(k_project_small<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      if (e != cudaSuccess) return e;
      launch_k(k_project_small<float>, dim3(N / 64, s), 256, sm, st, static_cast<const float*>(a.H), a.W_kv, a.W_z,
                                                               out, a.T, a.d_model, d, N, ks);
    } else {
      e = cudaFuncSetAttribute(k_project_small<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      if (e != cudaSuccess) return e;
      launch_k(k_project_small<uint16_t>, dim3(N / 64, s), 256, sm, st, static_cast<const uint16_t*>(a.H), a.W_kv,
                                                                  a.W_z, out, a.T, a.d_model, d, N, ks);
    }
  } else {
    s = pick_splits(a.T, a.d_model, N);
    int kps = ((a.d_model / s + PBK - 1) / PBK) * PBK;
  dim3 grid(N / PBN, (a.T + PBM - 1) / PBM, s);
  if (a.h_dtype == CSA2_F32)
    launch_k(k_project<float>, grid, 256, 0, st, static_cast<const float*>(a.H), a.W_kv, a.W_z, out,
                                           a.T, a.d_model, d, N, kps);
  else
    launch_k(k_project<uint16_t>, grid, 256, 0, st, static_cast<const uint16_t*>(a.H), a.W_kv, a.W_z,
                                              out, a.T, a.d_model, d, N, kps);
  }
  qp.Cp = out;
  qp.Zp = out + d;
  qp.split_stride = (long long)a.T * N;
  qp.nsplit = s;
  qp.ldc = N;
  return cudaGetLastError();
}

cudaError_t launch_compress(const csa2_compress_args& a, void* ws, cudaStream_t st) {
  const int d = a.cache.d;
  const int G = a.T / a.m;
  QuantParams qp{};
  if (a.W_kv) {
    if (project_tc_fused(a)) {
      // projection, pooling, RoPE and FP4 in one kernel; then the indexer K
      cudaError_t e = launch_project_tc(a, nullptr, true, st);
      if (e != cudaSuccess) return e;
      return launch_index_k_any(a, G, st);
    }
    cudaError_t e = project_rows(a, static_cast<float*>(ws), st, qp);
    if (e != cudaSuccess) return e;
  } else {
    qp.Cp = a.C;
    qp.Zp = a.Z;
    qp.split_stride = 0;
    qp.nsplit = 1;
    qp.ldc = d;
  }
  qp.G = G;
  qp.m = a.m;
  qp.d = d;
  qp.d_rope = a.d_rope;
  qp.rope_max_pos = a.rope_max_pos;
  qp.rope_cos = a.rope_cos;
  qp.rope_sin = a.rope_sin;
  qp.pos = a.pos;
  qp.seq = a.seq;
  qp.entry = a.entry;
  qp.cache = a.cache;
  qp.y_out = a.y_out;
  long long threads = (long long)G * (d / 16);
  if (a.W_ik && G > 0 && G < 2048 && !index_k_tc_supported(a, G) && d / 16 <= 256) {
    // a few entries (the decode append): quantisation and indexer K in one launch
    cudaError_t e = a.cache.d_ik == 128 ? launch_quant_index_k<128>(qp, a.W_ik, st)
                                        : launch_quant_index_k<64>(qp, a.W_ik, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  if (threads > 0) launch_k(k_quant, (unsigned)((threads + 255) / 256), 256, 0, st, qp);
  cudaError_t e = launch_index_k_any(a, G, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// FP8 rows with one float32 scale per row (the SWA window rows a bounded replay rebuilds):
// s = amax / 448, byte = E4M3_RNE_satfinite(x / s), float32 divisions.  One warp per row,
// lane l holding the row's elements [l d/32, (l + 1) d/32).
// ---------------------------------------------------------------------------------
template <int D, typename XT>
__global__ void __launch_bounds__(256) k_swa_quant(const XT* __restrict__ x, const int* __restrict__ row_idx, int R,
                                                   uint8_t* __restrict__ swa, float* __restrict__ swa_scale,
                                                   int swa_rows) {
  pdl_wait();
  pdl_trigger();
  constexpr int PL = D / 32;                     // elements per lane: 16 (d = 512) or 4 (d = 128)
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= R) return;
  float v[PL];
  const XT* xp = x + r * D + lane * PL;
  if constexpr (sizeof(XT) == 4) {
#pragma unroll
    for (int i = 0; i < PL / 4; ++i) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(xp) + i);
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < PL / 4; ++i) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(xp) + i);
      v[4 * i] = __uint_as_float(u.x << 16); v[4 * i + 1] = __uint_as_float(u.x & 0xffff0000u);
      v[4 * i + 2] = __uint_as_float(u.y << 16); v[4 * i + 3] = __uint_as_float(u.y & 0xffff0000u);
    }
  }
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < PL; ++i) a = fmaxf(a, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float sc = __fdiv_rn(a, 448.0f);
  uint32_t w[PL / 4];
#pragma unroll
  for (int i = 0; i < PL / 4; ++i) {
    w[i] = 0u;
    if (sc > 0.f)
#pragma unroll
      for (int j = 0; j < 4; ++j) w[i] |= cvt_e4m3(__fdiv_rn(v[4 * i + j], sc)) << (8 * j);
  }
  const long long dst = row_idx ? (long long)__ldg(row_idx + r) : r;
  if (dst < 0 || dst >= swa_rows) {
    if (lane == 0) raise_error(&g_err_compress, CSA2_DEVERR_SWA_RANGE);
    return;
  }
  uint8_t* o = swa + dst * D + lane * PL;
  if constexpr (PL == 16) {
    *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    *reinterpret_cast<uint32_t*>(o) = w[0];
  }
  if (lane == 0) swa_scale[dst] = sc;
}

cudaError_t launch_swa_quant(const csa2_swa_quant_args& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((a.R + 7) / 8);
  if (a.d == 512) {
    if (a.x_dtype == CSA2_F32)
      return launch_k(k_swa_quant<512, float>, grid, 256, 0, st, static_cast<const float*>(a.x), a.row_idx, a.R,
                      a.swa, a.swa_scale, a.swa_rows);
    return launch_k(k_swa_quant<512, uint16_t>, grid, 256, 0, st, static_cast<const uint16_t*>(a.x), a.row_idx, a.R,
                    a.swa, a.swa_scale, a.swa_rows);
  }
  if (a.x_dtype == CSA2_F32)
    return launch_k(k_swa_quant<128, float>, grid, 256, 0, st, static_cast<const float*>(a.x), a.row_idx, a.R,
                    a.swa, a.swa_scale, a.swa_rows);
  return launch_k(k_swa_quant<128, uint16_t>, grid, 256, 0, st, static_cast<const uint16_t*>(a.x), a.row_idx, a.R,
                  a.swa, a.swa_scale, a.swa_rows);
}

// ---------------------------------------------------------------------------------
// The decode-time append (csa2_compress_append)
// ---------------------------------------------------------------------------------
static csa2_compress_args append_view(const csa2_append_args& a) {
  csa2_compress_args c{};
  c.struct_size = sizeof(c);
  c.T = a.B;
  c.m = a.m;
  c.d_model = a.d_model;
  c.h_dtype = a.h_dtype;
  c.H = a.H;
  c.W_kv = a.W_kv;
  c.W_z = a.W_z;
  c.d_rope = a.d_rope;
  c.rope_max_pos = a.rope_max_pos;
  c.rope_cos = a.rope_cos;
  c.rope_sin = a.rope_sin;
  c.seq = a.seq;
  c.W_ik = a.W_ik;
  c.cache = a.cache;
  return c;
}

size_t append_workspace_bytes(const csa2_append_args& a) { return a.B > 0 ? project_ws_bytes(append_view(a)) : 0; }

cudaError_t launch_append(const csa2_append_args& a, void* ws, cudaStream_t st) {
  if (a.B == 0) return cudaSuccess;
  const csa2_compress_args c = append_view(a);
  AppendParams ap{};
  cudaError_t e = project_rows(c, static_cast<float*>(ws), st, ap.q);
  if (e != cudaSuccess) return e;
  ap.q.G = a.B;
  ap.q.m = a.m;
  ap.q.d = a.cache.d;
  ap.q.d_rope = a.d_rope;
  ap.q.rope_max_pos = a.rope_max_pos;
  ap.q.rope_cos = a.rope_cos;
  ap.q.rope_sin = a.rope_sin;
  ap.q.seq = a.seq;
  ap.q.cache = a.cache;
  ap.tok_pos = a.tok_pos;
  ap.pend = a.pend;
  ap.y_out = a.y_out;
  if (a.W_ik && a.cache.d_ik == 64)
    return launch_k(k_append_quant_index_k<64>, (unsigned)a.B, 256, ((size_t)a.cache.d + 8 * 64) * sizeof(float), st,
                    ap, a.W_ik);
  return launch_k(k_append_quant_index_k<128>, (unsigned)a.B, 256, ((size_t)a.cache.d + 8 * 128) * sizeof(float), st,
                  ap, a.W_ik);
}

uint32_t read_clear_error_compress() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_compress, sizeof(v));
  cudaMemcpyToSymbol(g_err_compress, &z, sizeof(z));
  return v;
}

}  // namespace csa2
