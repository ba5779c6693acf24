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
#include "tmap.h"

namespace csa2 {

CSA2_DEFINE_ERROR_WORD(g_err_proj);

namespace ptc {
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;                 // 16 KB
constexpr int B_BYTES = BN * BK * 2;                 // 32 KB: four 64-column blocks of 8 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM = STAGES * STAGE_BYTES + 128;     // + mbarriers and the TMEM slot (< 128 B)
constexpr int THREADS = 192;
constexpr uint32_t MAX_POLL = 1u << 24;
}  // namespace ptc


// The pooling / RoPE / FP4 epilogue fused into the GEMM (m = 1 or 2): at m = 2 a tile holds
// channels [128 x, 128 x + 128) of C (TMEM columns 0..127) and of Z (128..255), and the two
// tokens of a group are adjacent TMEM lanes of one warp, paired by a shuffle; at m = 1 a
// tile holds channels [256 x, 256 x + 256) of C.  The arithmetic is k_quant's.
struct ProjEpi {
  csa2_cache cache;
  const int* seq;
  const int* entry;
  const int* pos;
  const float* rope_cos;
  const float* rope_sin;
  int d_rope, rope_max_pos, m, G;
  float* y_out;
};

template <bool FUSE>
__global__ void __launch_bounds__(ptc::THREADS, 1)
    k_proj_tc(const __grid_constant__ CUtensorMap mh, const __grid_constant__ CUtensorMap mkv,
              const __grid_constant__ CUtensorMap mz, float* __restrict__ out, int T, int d_model, int d, int N,
              int ntn, int ntiles, ProjEpi ep) {
  using namespace ptc;
  pdl_wait();                                        // a persistent grid: dependents start at completion
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023) != 0) {                // the same in every CTA
    if (tid == 0) raise_error(&g_err_proj, CSA2_DEVERR_SMEM_ALIGN);
    return;
  }
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;                   // [2] accumulator buffer b complete
  uint64_t* acce = accf + 2;                         // [2] accumulator buffer b drained
  uint32_t* tslot = reinterpret_cast<uint32_t*>(acce + 2);
  const bool pair = FUSE && ep.m == 2;
  if (warp == 1) tc::tmem_alloc(tslot, 2 * BN);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 4);                    // one arrival per epilogue warp
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = *tslot;
  const int nk = d_model / BK;
  // tile t: output rows [128 (t / ntn), +128), column tile t % ntn (consecutive tiles share
  // their rows of H, which L2 then serves to the other column tiles)
  if (warp == 0) {
    if (lane == 0) {
      long long it = 0;                              // K blocks issued by this CTA
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int m0 = (t / ntn) * BM, nt = t % ntn;
        const int n0 = nt * BN;
        const CUtensorMap* mw = (n0 < d) ? &mkv : &mz;
        const int nw0 = (n0 < d) ? n0 : n0 - d;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          if (it >= STAGES && !tc::mbar_wait(&empty[s], (uint32_t)(((it / STAGES) - 1) & 1), MAX_POLL)) {
            raise_error(&g_err_proj, CSA2_DEVERR_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * STAGE_BYTES;
          tc::mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          tc::tma_load_2d(st, &mh, kb * BK, m0, &full[s]);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j) {
            const CUtensorMap* mj = pair ? (j < 2 ? &mkv : &mz) : mw;
            const int col = pair ? 128 * nt + 64 * (j & 1) : nw0 + 64 * j;
            tc::tma_load_2d(st + A_BYTES + j * 8192, mj, col, kb * BK, &full[s]);
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_f16(BM, BN, 1, 0, 1);   // bf16; A K-major, B MN-major
      long long it = 0;
      int tl = 0;                                    // tiles of this CTA
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++tl) {
        const int b = tl & 1;
        if (tl >= 2 && !tc::mbar_wait(&acce[b], (uint32_t)(((tl >> 1) - 1) & 1), MAX_POLL)) {
          raise_error(&g_err_proj, CSA2_DEVERR_TIMEOUT);
          break;
        }
        tc::fence_after_sync();
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          if (!tc::mbar_wait(&full[s], (uint32_t)((it / STAGES) & 1), MAX_POLL)) {
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
            tc::mma_f16_ss(tb + (uint32_t)(BN * b), ad, bd, idesc, (kb | k16) != 0 ? 1u : 0u);
          }
          tc::mma_commit(&empty[s]);                 // the stage is free once these have read it
        }
        tc::mma_commit(&accf[b]);                    // buffer b holds tile t
      }
    }
  } else {
    const int q = warp & 3;                          // warps 2..5 -> lane quarters 2, 3, 0, 1
    int tl = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tl) {
      const int b = tl & 1;
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&accf[b], (uint32_t)((tl >> 1) & 1), MAX_POLL));
      if (!ok) {
        if (lane == 0) raise_error(&g_err_proj, CSA2_DEVERR_TIMEOUT);
        break;
      }
      tc::fence_after_sync();
      const uint32_t tq = tb + ((uint32_t)(32 * q) << 16) + (uint32_t)(BN * b);
      const int m0 = (t / ntn) * BM, nt = t % ntn;
      const int row = m0 + 32 * q + lane;
      if (!FUSE) {
        const int n0 = nt * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tc::tmem_ld32(tq + (uint32_t)c, r);
          tc::tmem_ld_wait();
          if (row < T) {
            float4* o = reinterpret_cast<float4*>(out + (long long)row * N + n0 + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              o[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
          }
        }
      } else {
        const int CW = pair ? 128 : 256;             // channels of the tile
        const int cbase = nt * CW;
        const int g = row / ep.m;                    // entry (group)
        const bool writer = row < T && (!pair || (lane & 1) == 0);
        long long erow = -1;
        int ps = -1;
        if (writer && g < ep.G) {
          erow = entry_row(ep.cache, __ldg(ep.seq + g), __ldg(ep.entry + g), &g_err_proj);
          if (ep.d_rope > 0 && cbase + CW > d - ep.d_rope) {
            ps = __ldg(ep.pos + g);
            if (ps < 0 || ps >= ep.rope_max_pos) {
              raise_error(&g_err_proj, CSA2_DEVERR_POS);
              ps = -1;
            }
          }
        }
        const int rb = d - ep.d_rope, half = ep.d_rope / 2;
#pragma unroll 1
        for (int c = 0; c < CW; c += 32) {
          uint32_t cv[32], zv[32];
          tc::tmem_ld32(tq + (uint32_t)c, cv);
          if (pair) tc::tmem_ld32(tq + 128u + (uint32_t)c, zv);
          tc::tmem_ld_wait();
          float y[32];
          if (pair) {
            const bool first = (lane & 1) == 0;      // the group's first token
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float c_me = __uint_as_float(cv[i]), z_me = __uint_as_float(zv[i]);
              const float c_ot = __shfl_xor_sync(0xffffffffu, c_me, 1), z_ot = __shfl_xor_sync(0xffffffffu, z_me, 1);
              const float c0 = first ? c_me : c_ot, c1 = first ? c_ot : c_me;
              const float z0 = first ? z_me : z_ot, z1 = first ? z_ot : z_me;
              const float zmax = fmaxf(fmaxf(-INFINITY, z0), z1);
              const float e0 = expf(z0 - zmax), e1 = expf(z1 - zmax);
              float den = 0.f, num = 0.f;
              den += e0;
              num = fmaf(e0, c0, num);
              den += e1;
              num = fmaf(e1, c1, num);
              y[i] = num / den;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(cv[i]);
          }
          if (!writer) continue;
          const int ch0 = cbase + c;
          if (ps >= 0) {
#pragma unroll
            for (int i = 0; i < 32; i += 2)
              if (ch0 + i >= rb) {
                const long long ti = (long long)ps * half + (ch0 + i - rb) / 2;
                rope_pair(y[i], y[i + 1], __ldg(ep.rope_cos + ti), __ldg(ep.rope_sin + ti));
              }
          }
          if (ep.y_out && g < ep.G) {
            float4* yo = reinterpret_cast<float4*>(ep.y_out + (long long)g * d + ch0);
#pragma unroll
            for (int i = 0; i < 8; ++i) yo[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
          }
          if (erow >= 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t w0, w1, sb;
              fp4_group16(y + 16 * h, w0, w1, sb);
              const int grp = (ch0 + 16 * h) / 16;
              *reinterpret_cast<uint2*>(ep.cache.codes + erow * (d / 2) + grp * 8) = make_uint2(w0, w1);
              ep.cache.scales[erow * (d / 16) + grp] = (uint8_t)sb;
            }
          }
        }
      }
      tc::fence_before_sync();                       // this warp's TMEM reads of buffer b are done
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acce[b]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tb, 2 * BN);
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
  if (warp < 4 && ok_flag && cache.idx_k_dtype == CSA2_FP8E4M3) {
    // the compressed form: each thread owns one entry's row (TMEM lane); a first pass finds
    // the largest |bf16 value|, a second quantises (s = amax / 448, float32 divisions)
    const long long row = rows[32 * warp + lane];
    const uint32_t lanes = (uint32_t)(32 * warp) << 16;
    float a = 0.f;
#pragma unroll 1
    for (int c = 0; c < NK; c += 32) {
      uint32_t v[32];
      tc::tmem_ld32(tb + lanes + (uint32_t)c, v);
      tc::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(__bfloat162float(__float2bfloat16_rn(__uint_as_float(v[i])))));
    }
    const float sc = __fdiv_rn(a, 448.0f);
#pragma unroll 1
    for (int c = 0; c < NK; c += 32) {
      uint32_t v[32];
      tc::tmem_ld32(tb + lanes + (uint32_t)c, v);
      tc::tmem_ld_wait();
      if (row >= 0) {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pk[i] = 0u;
          if (sc > 0.f)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              pk[i] |= cvt_e4m3(__fdiv_rn(__bfloat162float(__float2bfloat16_rn(__uint_as_float(v[4 * i + j]))), sc))
                       << (8 * j);
        }
        uint4* dst = reinterpret_cast<uint4*>(cache.idx_k8 + row * NK + c);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    if (row >= 0) cache.idx_k8_scale[row] = sc;
  } else if (warp < 4 && ok_flag) {                  // warp w: TMEM lanes (rows) 32 w ..
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
// The fused epilogue handles m = 1 (256-channel tiles) and m = 2 (128 channels of C and Z).
bool project_tc_fused(const csa2_compress_args& a) {
  return project_tc_supported(a) && (a.m == 1 || a.m == 2) && a.cache.d % 256 == 0 && a.d_rope % 2 == 0;
}

bool project_tc_supported(const csa2_compress_args& a) {
  const int N = a.cache.d * (a.m > 1 ? 2 : 1);
  const bool aligned = ((uintptr_t)a.H & 15) == 0 && ((uintptr_t)a.W_kv & 15) == 0 &&
                       (a.m == 1 || ((uintptr_t)a.W_z & 15) == 0);
  return a.h_dtype == CSA2_BF16 && a.T > 64 && a.d_model % ptc::BK == 0 && a.cache.d % ptc::BN == 0 &&
         N % ptc::BN == 0 && aligned && tensor_map_encoder() != nullptr;
}

cudaError_t launch_project_tc(const csa2_compress_args& a, float* out, bool fuse, cudaStream_t st) {
  const int d = a.cache.d, N = d * (a.m > 1 ? 2 : 1);
  CUtensorMap mh, mkv, mz;
  if (!bf16_map(&mh, a.H, a.T, a.d_model, ptc::BM) || !bf16_map(&mkv, a.W_kv, a.d_model, d, ptc::BK) ||
      !bf16_map(&mz, a.m > 1 ? a.W_z : a.W_kv, a.d_model, d, ptc::BK))
    return cudaErrorInvalidValue;
  ProjEpi ep{};
  ep.cache = a.cache;
  ep.seq = a.seq;
  ep.entry = a.entry;
  ep.pos = a.pos;
  ep.rope_cos = a.rope_cos;
  ep.rope_sin = a.rope_sin;
  ep.d_rope = a.d_rope;
  ep.rope_max_pos = a.rope_max_pos;
  ep.m = a.m;
  ep.G = a.T / a.m;
  ep.y_out = a.y_out;
  const int ntn = fuse ? (a.m == 2 ? d / 128 : d / 256) : N / ptc::BN;
  const int ntiles = ntn * ((a.T + ptc::BM - 1) / ptc::BM);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const dim3 grid((unsigned)(ntiles < sms ? ntiles : (sms > 0 ? sms : 1)));   // persistent: one CTA per SM
  if (fuse) {
    static bool attr_set = false;
    if (!attr_set) {
      cudaError_t e = cudaFuncSetAttribute(k_proj_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, ptc::SMEM);
      if (e != cudaSuccess) return e;
      attr_set = true;
    }
    return launch_k_late(k_proj_tc<true>, grid, ptc::THREADS, ptc::SMEM, st, mh, mkv, mz, out, a.T, a.d_model, d,
                         N, ntn, ntiles, ep);
  }
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_proj_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, ptc::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // persistent (one CTA per SM): started only once the previous kernel has completed
  return launch_k_late(k_proj_tc<false>, grid, ptc::THREADS, ptc::SMEM, st, mh, mkv, mz, out, a.T, a.d_model, d, N,
                       ntn, ntiles, ep);
}

uint32_t read_clear_error_proj() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_err_proj, sizeof(v));
  if (v) cudaMemcpyToSymbol(g_err_proj, &z, sizeof(z));
  return v;
}

}  // namespace csa2
