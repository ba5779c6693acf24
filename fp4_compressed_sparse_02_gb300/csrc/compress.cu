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
  for (int s = 1; s < nsplit; ++s) {
    float w[16];
    load16(p + s * stride, w);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += w[i];
  }
}

__global__ void __launch_bounds__(256) k_quant(QuantParams p) {
  const int gpr = p.d / 16;                           // 16-channel groups per entry
  long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  long long g = gid / gpr;
  const int q = (int)(gid % gpr);
  if (g >= p.G) return;
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
    int ps = __ldg(p.pos + g);
    if (ps < 0 || ps >= p.rope_max_pos) {
      raise_error(&g_err_compress, CSA2_DEVERR_POS);
    } else {
      const int half = p.d_rope / 2;
      const float* ct = p.rope_cos + (long long)ps * half + (c0 - rb) / 2;
      const float* st = p.rope_sin + (long long)ps * half + (c0 - rb) / 2;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float cs = __ldg(ct + i), sn = __ldg(st + i);
        float x0 = y[2 * i], x1 = y[2 * i + 1];
        y[2 * i] = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
        y[2 * i + 1] = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
      }
    }
  }
  if (p.y_out) {
    float4* yo = reinterpret_cast<float4*>(p.y_out + g * p.d + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) yo[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
  }
  // scale = E4M3_RNE_satfinite(amax / 6); codes = E2M1_RNE_sat(y / scale)
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(y[i]));
  uint32_t sbyte = cvt_e4m3(__fdiv_rn(a, 6.0f));
  float s = e4m3_to_f32(sbyte);
  uint32_t w0 = 0, w1 = 0;
  if (s > 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w0 |= cvt_e2m1x2(__fdiv_rn(y[2 * i], s), __fdiv_rn(y[2 * i + 1], s)) << (8 * i);
      w1 |= cvt_e2m1x2(__fdiv_rn(y[8 + 2 * i], s), __fdiv_rn(y[9 + 2 * i], s)) << (8 * i);
    }
  }
  long long row = entry_row(p.cache, __ldg(p.seq + g), __ldg(p.entry + g), &g_err_compress);
  if (row < 0) return;
  uint2* cd = reinterpret_cast<uint2*>(p.cache.codes + row * (p.d / 2) + q * 8);
  *cd = make_uint2(w0, w1);
  p.cache.scales[row * (p.d / 16) + q] = (uint8_t)sbyte;
}

// ---------------------------------------------------------------------------------
// Indexer K: idx_k[e][j] = bf16( sum_c dequant(e)[c] * W_ik[c][j] ), float32 FMA in
// ascending c.  16 entries per CTA, one thread per output column.
// ---------------------------------------------------------------------------------
constexpr int IK_E = 16;

__global__ void __launch_bounds__(128) k_index_k(csa2_cache cache, const int* __restrict__ seq,
                                                 const int* __restrict__ entry, int G,
                                                 const uint16_t* __restrict__ Wik) {
  extern __shared__ float deq[];                 // [IK_E][d]
  __shared__ long long rows[IK_E];
  const int d = cache.d, dik = cache.d_ik;
  const int g0 = blockIdx.x * IK_E;
  if (threadIdx.x < IK_E) {
    int g = g0 + threadIdx.x;
    rows[threadIdx.x] = (g < G) ? entry_row(cache, __ldg(seq + g), __ldg(entry + g), &g_err_compress) : -1;
  }
  __syncthreads();
  // dequantise: each thread handles one code byte (2 channels) at a time
  for (int i = threadIdx.x; i < IK_E * d / 2; i += blockDim.x) {
    int e = i / (d / 2), cb = i % (d / 2);
    long long r = rows[e];
    float v0 = 0.f, v1 = 0.f;
    if (r >= 0) {
      uint32_t byte = cache.codes[r * (d / 2) + cb];
      float s = e4m3_to_f32(cache.scales[r * (d / 16) + (2 * cb) / 16]);
      uint32_t h2 = e2m1x2_to_f16x2(byte);
      __half2 hv = *reinterpret_cast<__half2*>(&h2);
      v0 = __low2float(hv) * s;
      v1 = __high2float(hv) * s;
    }
    deq[e * d + 2 * cb] = v0;
    deq[e * d + 2 * cb + 1] = v1;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < dik; j += blockDim.x) {
    float acc[IK_E];
#pragma unroll
    for (int e = 0; e < IK_E; ++e) acc[e] = 0.f;
    for (int c = 0; c < d; ++c) {
      float w = bf16_bits_to_f32(__ldg(Wik + (long long)c * dik + j));
#pragma unroll
      for (int e = 0; e < IK_E; ++e) acc[e] = fmaf(deq[e * d + c], w, acc[e]);
    }
#pragma unroll
    for (int e = 0; e < IK_E; ++e) {
      long long r = rows[e];
      if (r >= 0) {
        __nv_bfloat16 hb = __float2bfloat16_rn(acc[e]);
        cache.idx_k[r * dik + j] = *reinterpret_cast<uint16_t*>(&hb);
      }
    }
  }
}

// ---------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------
static int pick_splits(int T, int d_model, int N) {
  // enough CTAs to cover the GPU when T is small (decode append): split K so that
  // (tiles x splits) >= ~2 waves of 152 SMs, keeping each split >= 128 deep.
  long long tiles = (long long)((T + PBM - 1) / PBM) * (N / PBN);
  int s = 1;
  while (tiles * s < 304 && d_model / (s * 2) >= 128) s *= 2;
  return s;
}

size_t compress_workspace_bytes(const csa2_compress_args& a) {
  if (!a.W_kv) return 0;
  int N = a.cache.d * (a.m > 1 ? 2 : 1);
  int s = pick_splits(a.T, a.d_model, N);
  return (size_t)s * a.T * N * sizeof(float);
}

cudaError_t launch_compress(const csa2_compress_args& a, void* ws, cudaStream_t st) {
  const int d = a.cache.d;
  const int G = a.T / a.m;
  QuantParams qp{};
  if (a.W_kv) {
    int N = d * (a.m > 1 ? 2 : 1);
    int s = pick_splits(a.T, a.d_model, N);
    int kps = ((a.d_model / s + PBK - 1) / PBK) * PBK;
    dim3 grid(N / PBN, (a.T + PBM - 1) / PBM, s);
    float* out = static_cast<float*>(ws);
    if (a.h_dtype == CSA2_F32)
      k_project<float><<<grid, 256, 0, st>>>(static_cast<const float*>(a.H), a.W_kv, a.W_z, out,
                                             a.T, a.d_model, d, N, kps);
    else
      k_project<uint16_t><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(a.H), a.W_kv, a.W_z,
                                                out, a.T, a.d_model, d, N, kps);
    qp.Cp = out;
    qp.Zp = out + d;
    qp.split_stride = (long long)a.T * N;
    qp.nsplit = s;
    qp.ldc = N;
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
  if (threads > 0) k_quant<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(qp);
  if (a.W_ik && G > 0) {
    size_t sm = (size_t)IK_E * d * sizeof(float);
    k_index_k<<<(G + IK_E - 1) / IK_E, 128, sm, st>>>(a.cache, a.seq, a.entry, G, a.W_ik);
  }
  return cudaGetLastError();
}

uint32_t read_clear_error_compress() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_compress, sizeof(v));
  cudaMemcpyToSymbol(g_err_compress, &z, sizeof(z));
  return v;
}

}  // namespace csa2
