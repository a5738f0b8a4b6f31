// Quantize-and-append kernels.
//
// KIVI-style asymmetric min/max quantization (SpeCache page, "Approach" and the
// "Measured effects" table: 2-bit and 1-bit KIVI with g = 32/64; QuantSpec page,
// "Experimental setup": builds on KIVI).  Keys get one (scale, zero) per channel
// over a group of G tokens; values one per token over a block of G channels.
// The hierarchical INT8 code is stored as two nibble planes: the upper nibble
// is the INT4 draft code, and upper + lower rebuild the INT8 target code
// (QuantSpec page, "Approach").  Groups are flushed from the double
// full-precision buffer of 2G tokens (same section).
//
// Every step is an fp32 operation with round-to-nearest-even, written with
// explicit intrinsics so that nothing is contracted into an FMA:
//   mn = min + 0, mx = max + 0, scale = (mx - mn) / (2^b - 1),
//   inv = scale == 0 ? 0 : 1 / scale, code = clamp(rint((x - mn) * inv), 0, 2^b - 1).
#include "kvq_device.cuh"

namespace kvq {
namespace {

constexpr int kFlushThreads = 256;

__device__ __forceinline__ uint32_t quant_code(float x, float mn, float inv, float levels) {
  float t = rintf(__fmul_rn(__fsub_rn(x, mn), inv));
  t = fminf(fmaxf(t, 0.0f), levels);
  return static_cast<uint32_t>(t);
}

__device__ __forceinline__ void scale_inv(float mn, float mx, float levels, float& scale, float& inv) {
  scale = __fdiv_rn(__fsub_rn(mx, mn), levels);
  inv = (scale == 0.0f) ? 0.0f : __fdiv_rn(1.0f, scale);
}

// One CTA quantizes one group of G tokens of one (b, kv head).
// Stream position p of this call: p < r comes from the residual buffer (slot
// (res_start + p) mod 2G), otherwise from the new tokens (index p - r).
template <int FMT>
__global__ void __launch_bounds__(kFlushThreads) flush_kernel(FlushParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D, G = p.G, NJ = D / G;
  const int gi = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long u = static_cast<long long>(b) * p.Hkv + kvh;
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);            // [G][D]
  uint16_t* Vs = Ks + G * D;                                    // [G][D]
  float* kmn = reinterpret_cast<float*>(Vs + G * D);            // [D]
  float* kinv = kmn + D;                                        // [D]
  float* vmn = kinv + D;                                        // [G][NJ]
  float* vinv = vmn + G * NJ;                                   // [G][NJ]

  // ---- gather the group's G source tokens (16-byte vectors) ----
  const int vec_per_tok = D / 8;
  for (int e = threadIdx.x; e < G * vec_per_tok; e += blockDim.x) {
    const int i = e / vec_per_tok, c = e % vec_per_tok;
    const int pos = gi * G + i;
    const uint4* srck;
    const uint4* srcv;
    if (pos < p.r) {
      const int slot = (p.res_start + pos) % (2 * G);
      const long long off = (u * 2 * G + slot) * D;
      srck = reinterpret_cast<const uint4*>(p.res_k + off);
      srcv = reinterpret_cast<const uint4*>(p.res_v + off);
    } else {
      const long long off = (u * p.n + (pos - p.r)) * D;
      srck = reinterpret_cast<const uint4*>(p.k_new + off);
      srcv = reinterpret_cast<const uint4*>(p.v_new + off);
    }
    reinterpret_cast<uint4*>(Ks + i * D)[c] = srck[c];
    reinterpret_cast<uint4*>(Vs + i * D)[c] = srcv[c];
  }
  __syncthreads();

  constexpr int BITS = FMT;  // 8, 2 or 1
  const float levels = static_cast<float>((1 << BITS) - 1);
  const long long grp = p.Lq / G + gi;       // global group index
  const long long tok0 = p.Lq + static_cast<long long>(gi) * G;

  // ---- key statistics: per channel over the G tokens ----
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float mn = bf16_to_f32(Ks[d]), mx = mn;
    for (int i = 1; i < G; ++i) {
      const float x = bf16_to_f32(Ks[i * D + d]);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    float scale, inv;
    scale_inv(mn, mx, levels, scale, inv);
    kmn[d] = mn;
    kinv[d] = inv;
    float* dst = p.ksz + (u * (p.C / G) + grp) * 2 * D;
    dst[d] = scale;
    dst[D + d] = mn;
  }
  // ---- value statistics: per token over each block of G channels ----
  {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
    for (int e = warp; e < G * NJ; e += nw) {
      const int i = e / NJ, jv = e % NJ;
      float mn = __int_as_float(0x7f800000), mx = -mn;
      for (int c = lane; c < G; c += 32) {
        const float x = bf16_to_f32(Vs[i * D + jv * G + c]);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      if (lane == 0) {
        mn = __fadd_rn(mn, 0.0f);
        mx = __fadd_rn(mx, 0.0f);
        float scale, inv;
        scale_inv(mn, mx, levels, scale, inv);
        vmn[i * NJ + jv] = mn;
        vinv[i * NJ + jv] = inv;
        float* dst = p.vsz + (u * p.C + tok0 + i) * 2 * NJ;
        dst[jv] = scale;
        dst[NJ + jv] = mn;
      }
    }
  }
  __syncthreads();

  // ---- key codes: token-major rows, channels packed (8/pb per byte) ----
  if constexpr (FMT == KVQ_FMT_HIER8) {
    // Each thread writes one 32-bit word of both nibble planes: 8 channels.
    const int words = D / 8;
    for (int e = threadIdx.x; e < G * words; e += blockDim.x) {
      const int i = e / words, w = e % words;
      uint32_t hi = 0, lo = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int d = 8 * w + k;
        const uint32_t c = quant_code(bf16_to_f32(Ks[i * D + d]), kmn[d], kinv[d], levels);
        hi |= (c >> 4) << (4 * k);
        lo |= (c & 15u) << (4 * k);
      }
      const long long row = (u * p.C + tok0 + i) * (D / 2);
      reinterpret_cast<uint32_t*>(p.kplane[0] + row)[w] = hi;
      reinterpret_cast<uint32_t*>(p.kplane[1] + row)[w] = lo;
    }
  } else {
    constexpr int PER = 8 / BITS;             // codes per byte
    constexpr int CPW = 4 * PER;              // codes per 32-bit word
    const int words = D / CPW;                // 2-bit: D/16, 1-bit: D/32
    const int rowbytes = D * BITS / 8;
    for (int e = threadIdx.x; e < G * words; e += blockDim.x) {
      const int i = e / words, w = e % words;
      uint32_t v = 0;
#pragma unroll
      for (int k = 0; k < CPW; ++k) {
        const int d = CPW * w + k;
        v |= quant_code(bf16_to_f32(Ks[i * D + d]), kmn[d], kinv[d], levels) << (BITS * k);
      }
      reinterpret_cast<uint32_t*>(p.kplane[0] + (u * p.C + tok0 + i) * rowbytes)[w] = v;
    }
  }

  // ---- value codes: 32-token slabs, rows = channels, tokens packed ----
  {
    const int nslab = G / 32;
    const long long slab0 = (u * p.C + tok0) / 32;
    if constexpr (FMT == KVQ_FMT_HIER8) {
      // row = 16 bytes per plane = 4 words; word w holds tokens 8w..8w+7
      for (int e = threadIdx.x; e < nslab * 4 * D; e += blockDim.x) {
        const int d = e % D, w = (e / D) % 4, s = e / (4 * D);
        const int jv = d / G;
        uint32_t hi = 0, lo = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = 32 * s + 8 * w + k;
          const uint32_t c =
              quant_code(bf16_to_f32(Vs[i * D + d]), vmn[i * NJ + jv], vinv[i * NJ + jv], levels);
          hi |= (c >> 4) << (4 * k);
          lo |= (c & 15u) << (4 * k);
        }
        const long long off = ((slab0 + s) * D + d) * 16;
        reinterpret_cast<uint32_t*>(p.vplane[0] + off)[w] = hi;
        reinterpret_cast<uint32_t*>(p.vplane[1] + off)[w] = lo;
      }
    } else {
      constexpr int PER = 8 / BITS;
      constexpr int CPW = 4 * PER;            // tokens per word
      constexpr int WPR = 32 / CPW;           // words per slab row (2-bit: 2, 1-bit: 1)
      constexpr int ROWB = 32 * BITS / 8;
      for (int e = threadIdx.x; e < nslab * WPR * D; e += blockDim.x) {
        const int d = e % D, w = (e / D) % WPR, s = e / (WPR * D);
        const int jv = d / G;
        uint32_t v = 0;
#pragma unroll
        for (int k = 0; k < CPW; ++k) {
          const int i = 32 * s + CPW * w + k;
          v |= quant_code(bf16_to_f32(Vs[i * D + d]), vmn[i * NJ + jv], vinv[i * NJ + jv], levels)
               << (BITS * k);
        }
        reinterpret_cast<uint32_t*>(p.vplane[0] + ((slab0 + s) * D + d) * ROWB)[w] = v;
      }
    }
  }
}

// Copy the new tokens that stay in the residual buffer into their slots.
__global__ void residual_write_kernel(ResidualWriteParams p) {
  const int j = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long u = static_cast<long long>(b) * p.Hkv + kvh;
  const int pos = p.first_new + j;                    // stream position
  const int slot = (p.res_start + pos) % (2 * p.G);
  const long long src = (u * p.n + (pos - p.r)) * p.D;
  const long long dst = (u * 2 * p.G + slot) * p.D;
  const int nvec = p.D / 8;
  for (int c = threadIdx.x; c < 2 * nvec; c += blockDim.x) {
    if (c < nvec) {
      reinterpret_cast<uint4*>(p.res_k + dst)[c] = reinterpret_cast<const uint4*>(p.k_new + src)[c];
    } else {
      reinterpret_cast<uint4*>(p.res_v + dst)[c - nvec] =
          reinterpret_cast<const uint4*>(p.v_new + src)[c - nvec];
    }
  }
}

template <int FMT>
cudaError_t launch_flush_t(const FlushParams& p, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(2) * p.G * p.D * sizeof(uint16_t) +
                      (2 * p.D + 2 * p.G * (p.D / p.G)) * sizeof(float);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&flush_kernel<FMT>), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.nflush, p.Hkv, p.B);
  flush_kernel<FMT><<<grid, kFlushThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_flush(const FlushParams& p, cudaStream_t s) {
  switch (p.fmt) {
    case KVQ_FMT_HIER8: return launch_flush_t<KVQ_FMT_HIER8>(p, s);
    case KVQ_FMT_INT2: return launch_flush_t<KVQ_FMT_INT2>(p, s);
    case KVQ_FMT_INT1: return launch_flush_t<KVQ_FMT_INT1>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_residual_write(const ResidualWriteParams& p, cudaStream_t s) {
  dim3 grid(p.count, p.Hkv, p.B);
  residual_write_kernel<<<grid, 64, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
