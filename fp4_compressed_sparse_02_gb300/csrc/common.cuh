// Shared device helpers of the CSA2 library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "csa2.h"

namespace csa2 {

constexpr int kPage = CSA2_PAGE_SIZE;   // entries per page
constexpr int kPageShift = 6;

// Each translation unit owns one device error word; the API layer ORs them.
// A kernel that meets an out-of-range value reported by the device (a page id, an
// n_vis, a pool length) sets a bit here and skips the access.
#define CSA2_DEFINE_ERROR_WORD(name) static __device__ unsigned int name = 0u

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation (launch_k): its CTAs may be scheduled while the
// previous kernel of the stream is still running.  So each kernel calls pdl_wait()
// before its first global-memory access -- it returns once the previous grid has
// completed and its writes are visible, which keeps stream order for everything the
// kernel reads or writes -- and pdl_trigger() to let the next kernel be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Host: launch `kernel` on stream `st` with programmatic stream serialisation
// (launch_k), or without it (launch_k_late: the kernel starts only once the previous
// kernel has completed, and its pdl_wait() is a no-op).  The cluster Top-k is launched
// late: its 8-CTA clusters placed early on the few SMs a running attention leaves idle
// pack worse than on an empty GPU.  So are the persistent kernels (the Full scan, the
// tensor-core scoring and projection), whose grids are sized to fill an empty GPU.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_late(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void raise_error(unsigned int* word, unsigned int bit) {
  atomicOr(word, bit);
}

// Resolve entry e of sequence s to a row index in the page planes (page*64 + slot),
// or -1 (with an error bit) when the page table points outside the planes.
__device__ __forceinline__ long long entry_row(const csa2_cache& c, int s, long long e,
                                               unsigned int* err) {
  long long p = e >> kPageShift;
  if (s < 0 || s >= c.num_seqs) { raise_error(err, CSA2_DEVERR_SEQ); return -1; }
  if (e < 0 || p >= c.max_pages) { raise_error(err, CSA2_DEVERR_PAGE_SLOT); return -1; }
  int page = __ldg(c.page_table + (long long)s * c.max_pages + p);
  if (page < 0 || page >= c.num_pages) { raise_error(err, CSA2_DEVERR_PAGE_ID); return -1; }
  return ((long long)page << kPageShift) | (e & (kPage - 1));
}

// entry_row in two halves, so that other loads can be issued between the page-table load and
// the use of its value: the first checks the slot and issues the load (slot_ok false after a
// reported error), the second checks the page id and forms the row.
__device__ __forceinline__ int entry_page_load(const csa2_cache& c, int s, long long e, unsigned int* err,
                                               bool& slot_ok) {
  const long long p = e >> kPageShift;
  slot_ok = false;
  if (s < 0 || s >= c.num_seqs) { raise_error(err, CSA2_DEVERR_SEQ); return -1; }
  if (e < 0 || p >= c.max_pages) { raise_error(err, CSA2_DEVERR_PAGE_SLOT); return -1; }
  slot_ok = true;
  return __ldg(c.page_table + (long long)s * c.max_pages + p);
}
__device__ __forceinline__ long long entry_row_of_page(const csa2_cache& c, int page, long long e, unsigned int* err) {
  if (page < 0 || page >= c.num_pages) { raise_error(err, CSA2_DEVERR_PAGE_ID); return -1; }
  return ((long long)page << kPageShift) | (e & (kPage - 1));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// --- PTX wrappers -------------------------------------------------------------

// Two float32 -> packed E2M1 pair (lo nibble = a), round-to-nearest-even, satfinite.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float a, float b) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n mov.b16 %0, {t, 0};\n}"
      : "=h"(r) : "f"(a), "f"(b));
  return (uint32_t)(r & 0xFF);
}

// float32 -> E4M3 byte, round-to-nearest-even, satfinite.
__device__ __forceinline__ uint32_t cvt_e4m3(float a) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(a));
  return (uint32_t)(r & 0xFF);
}

// One byte of two E2M1 codes -> fp16x2 (lo nibble -> low half).  Exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(r) : "r"(byte));
  return r;
}

// Two E4M3 bytes (lo byte -> low half) -> fp16x2.  Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2 = e4m3x2_to_f16x2((uint16_t)(byte & 0xFF));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}


// mma.sync m16n8k16, fp32 accumulate.  BF16 or F16 operands.
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The low / high two E4M3 bytes of a word as an f16 pair.
__device__ __forceinline__ uint32_t e4m3x2_lo_f16x2(uint32_t w) { return e4m3x2_to_f16x2((uint16_t)(w & 0xffffu)); }
__device__ __forceinline__ uint32_t e4m3x2_hi_f16x2(uint32_t w) { return e4m3x2_to_f16x2((uint16_t)(w >> 16)); }

__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(saddr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3, uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(saddr));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte streaming load that does not allocate in L1 (single-use HBM data).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Bring `bytes` (a multiple of 16) from the 16-byte aligned global address p into L2 with one
// bulk request (nothing is returned to the thread): later loads of those bytes hit L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// The same for scattered rows shorter than 256 bytes: no L2 prefetch beyond the requested
// 128-byte line (the 256-byte hint would double the DRAM bytes of a 128-byte row).
__device__ __forceinline__ uint4 ldg_gather_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::128B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// 32-byte streaming load (p 32-byte aligned) into two 16-byte halves: half the load
// requests of two 16-byte loads for the same bytes.
__device__ __forceinline__ void ldg_stream_v8(const void* p, uint4& lo, uint4& hi) {
  asm("ld.global.nc.L1::no_allocate.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
      : "l"(p));
}

// FP4 of one 16-channel group: scale byte = E4M3_RNE_satfinite(amax / 6), codes =
// E2M1_RNE_sat(y_i / s) (float32 divisions), two codes per byte with the even channel in
// the low nibble; a zero scale gives zero codes.
__device__ __forceinline__ void fp4_group16(const float* y, uint32_t& w0, uint32_t& w1, uint32_t& sbyte) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(y[i]));
  sbyte = cvt_e4m3(__fdiv_rn(a, 6.0f));
  const float s = e4m3_to_f32(sbyte);
  w0 = 0;
  w1 = 0;
  if (s > 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w0 |= cvt_e2m1x2(__fdiv_rn(y[2 * i], s), __fdiv_rn(y[2 * i + 1], s)) << (8 * i);
      w1 |= cvt_e2m1x2(__fdiv_rn(y[8 + 2 * i], s), __fdiv_rn(y[9 + 2 * i], s)) << (8 * i);
    }
  }
}

// One row quantised to E4M3 with one float32 scale, spread over a warp (lane l holds
// N consecutive values): s = amax / 448, byte = E4M3_RNE_satfinite(x / s) (float32
// divisions), s == 0 -> zero bytes.  Stores the lane's N bytes at dst (N = 4: one 32-bit
// store; N = 2: 16-bit) and lane 0 the scale.  Every lane of the warp must call it.
template <int N>
__device__ __forceinline__ float fp8_row_store(const float* v, uint8_t* dst, float* scale) {
  float a = 0.f;
#pragma unroll
  for (int j = 0; j < N; ++j) a = fmaxf(a, fabsf(v[j]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float s = __fdiv_rn(a, 448.0f);
  uint32_t w = 0;
  if (s > 0.f)
#pragma unroll
    for (int j = 0; j < N; ++j) w |= cvt_e4m3(__fdiv_rn(v[j], s)) << (8 * j);
  if constexpr (N == 4) {
    *reinterpret_cast<uint32_t*>(dst) = w;
  } else {
    static_assert(N == 2, "2 or 4 values a lane");
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w;
  }
  if ((threadIdx.x & 31) == 0) *scale = s;
  return s;
}

// RoPE of one channel pair, every product and sum rounded on its own.
__device__ __forceinline__ void rope_pair(float& x0, float& x1, float cs, float sn) {
  const float y0 = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
  const float y1 = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, cs));
  x0 = y0;
  x1 = y1;
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0 maps like +0.
__device__ __forceinline__ uint32_t float_key(float f) {
  if (f == 0.0f) f = 0.0f;   // -0 and +0 get one key
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace csa2
