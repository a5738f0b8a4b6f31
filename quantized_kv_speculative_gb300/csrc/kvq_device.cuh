// Device-side building blocks shared by the kernels of this library:
// mbarrier + 1-D bulk (TMA) copies, bounded waits, thread-block cluster
// helpers, the m16n8k16 tensor-core MMA, f16 packing, and the warp reductions
// of the exact top-k score.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_internal.h"

namespace kvq {

// ------------------------------------------------------------------------------
// Shared-memory addresses, mbarriers, bulk copies
// ------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// True in exactly one lane of the calling warp, which must be converged
// (elect.sync over the full mask).
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(e));
  return e != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// `limit` SM clocks.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// 1-D bulk copy global -> shared through the TMA unit, completing on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Pull the 128-byte line at p into L2 and keep it ahead of streamed data.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------------------
// Thread-block clusters: the hardware cluster barrier (every thread of every
// CTA of the cluster arrives; release / acquire order shared and global memory
// at cluster scope) and loads from another CTA's shared memory.
// ------------------------------------------------------------------------------
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of this CTA's shared location `p` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_dsmem(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t ld_dsmem_u64(uint32_t a) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_dsmem4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// ------------------------------------------------------------------------------
// Tensor-core MMA: D[16x8] += A[16x16] (row) * B[16x8] (col), f16 in, f32 acc.
//   a[0] = (row g,   k 2q..2q+1)   a[1] = (row g+8, k 2q..2q+1)
//   a[2] = (row g,   k 2q+8..+9)   a[3] = (row g+8, k 2q+8..+9)
//   b[0] = (k 2q..2q+1, col g)     b[1] = (k 2q+8..+9, col g)
//   c[0..1] = (row g, col 2q..2q+1), c[2..3] = (row g+8, col 2q..2q+1)
// with g = lane / 4, q = lane % 4; the lower half of a register is the lower
// index.
// ------------------------------------------------------------------------------

// Not volatile: the MMA is a pure function of its operands, so the compiler
// may interleave independent accumulation chains.
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same MMA with a separate accumulator input: D = A * B + C.
__device__ __forceinline__ void mma16816_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                           const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// bf16 inputs, f32 accumulate: C += A * B.
__device__ __forceinline__ void mma16816_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit elements held one pair per lane (lane
// 4r + c holds row r, columns 2c and 2c + 1): lane 4r + c receives rows 2c and
// 2c + 1 of column r.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_half2(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^e as an fp32 for -126 <= e <= 127.
__device__ __forceinline__ float pow2f_exact(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// Largest value over the warp of a non-negative finite fp32 (its bit pattern
// orders like its value): one warp reduction.
__device__ __forceinline__ float warp_max_nonneg(float x) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(x)));
}

// The top-k score's zero-point term of one key group, by one warp: lane l
// holds the products p_d = fp32(qs_d z_d) of CPL channels.  With f the
// exponent of max|p| (max|p| < 2^f, floored at -80), beta = fp32(Z) 2^(f-40)
// with Z = sum_d rint(p_d 2^(40-f)), an exact 64-bit integer sum, so the
// lanes may add in any order.  Each term (|t| < 2^40) is split as
// hi 2^20 + lo with 0 <= lo < 2^20; the warp sums hi and lo in 32-bit
// integer reductions (both stay below 2^27 for at most 128 channels), then
// recombines.  Every lane returns beta.
template <int CPL>
__device__ __forceinline__ float zero_term_warp(const float (&p)[CPL]) {
  static_assert(CPL * 32 <= 128, "the 32-bit partial sums assume at most 128 channels");
  float mx = 0.f;
#pragma unroll
  for (int c = 0; c < CPL; ++c) mx = fmaxf(mx, fabsf(p[c]));
  mx = warp_max_nonneg(mx);
  int f = 0;
  if (mx > 0.f) frexpf(mx, &f);
  f = max(f, -80);
  const float up = pow2f_exact(40 - f);
  int hs = 0, ls = 0;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const long long t = __float2ll_rn(__fmul_rn(p[c], up));
    hs += static_cast<int>(t >> 20);
    ls += static_cast<int>(t & 0xFFFFFLL);
  }
  hs = __reduce_add_sync(0xffffffffu, hs);
  ls = __reduce_add_sync(0xffffffffu, ls);
  const long long z = (static_cast<long long>(hs) << 20) + ls;
  return __fmul_rn(__ll2float_rn(z), pow2f_exact(f - 40));
}

}  // namespace kvq

namespace kvq {
// Opt a kernel into more than 48 KB of dynamic shared memory, once per device
// (also keeps the call out of CUDA-graph captures after the first launch).
inline cudaError_t set_smem_once(const void* func, int bytes) {
  constexpr int kMaxDev = 64;
  static int done_bytes[kMaxDev][8] = {};
  static const void* done_func[kMaxDev][8] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  for (int i = 0; i < 8; ++i) {
    if (done_func[dev][i] == func && done_bytes[dev][i] >= bytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < 8; ++i) {
    if (done_func[dev][i] == nullptr || done_func[dev][i] == func) {
      done_func[dev][i] = func;
      done_bytes[dev][i] = bytes;
      break;
    }
  }
  return cudaSuccess;
}
}  // namespace kvq
