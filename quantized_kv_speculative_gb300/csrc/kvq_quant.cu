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

constexpr int kFlushThreads = 512;

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
// Every phase spreads over all threads: key statistics by (channel pair, token
// stripe), value statistics by (token, channel block, part of the block).
template <int FMT>
__global__ void __launch_bounds__(kFlushThreads) flush_kernel(FlushParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int D = p.D, G = p.G, NJ = D / G;
  const int tid = threadIdx.x;
  const int gi = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long u = static_cast<long long>(b) * p.Hkv + kvh;
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);            // [G][D]
  uint16_t* Vs = Ks + G * D;                                    // [G][D]
  float* kmn = reinterpret_cast<float*>(Vs + G * D);            // [D]
  float* kinv = kmn + D;                                        // [D]
  float* vmn = kinv + D;                                        // [G][NJ]
  float* vinv = vmn + G * NJ;                                   // [G][NJ]
  float* part = vinv + G * NJ;                                  // [2][kFlushThreads * 2] stripe min/max

  // ---- gather the group's G source tokens (16-byte vectors, 4 in flight per thread) ----
  const int vec_per_tok = D / 8;
  const int nvec = G * vec_per_tok;
  for (int e0 = tid; e0 < nvec; e0 += 4 * kFlushThreads) {
    uint4 kv[4], vv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + j * kFlushThreads;
      if (e < nvec) {
        const int i = e / vec_per_tok, c = e % vec_per_tok;
        const int pos = gi * G + i;
        long long off;
        const uint16_t *sk, *sv;
        if (pos < p.r) {
          const int slot = (p.res_start + pos) % (2 * G);
          off = (u * 2 * G + slot) * D;
          sk = p.res_k;
          sv = p.res_v;
        } else {
          off = (u * p.n + (pos - p.r)) * D;
          sk = p.k_new;
          sv = p.v_new;
        }
        kv[j] = reinterpret_cast<const uint4*>(sk + off)[c];
        vv[j] = reinterpret_cast<const uint4*>(sv + off)[c];
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + j * kFlushThreads;
      if (e < nvec) {
        reinterpret_cast<uint4*>(Ks)[e] = kv[j];
        reinterpret_cast<uint4*>(Vs)[e] = vv[j];
      }
    }
  }
  __syncthreads();
  // A single flushed group reads this head's old slots only in the gather
  // above, so the new tokens that stay in the buffer can be written now.
  if (p.res_count > 0) {
    const int nv = p.res_count * vec_per_tok;
    for (int e = tid; e < 2 * nv; e += kFlushThreads) {
      const int kv = e >= nv, e2 = kv ? e - nv : e;
      const int j = e2 / vec_per_tok, c = e2 % vec_per_tok;
      const int pos = p.first_new + j;
      const int slot = (p.res_start + pos) % (2 * G);
      const long long src = (u * p.n + (pos - p.r)) * D;
      const long long dst = (u * 2 * G + slot) * D;
      const uint16_t* from = kv ? p.v_new : p.k_new;
      uint16_t* to = kv ? p.res_v_w : p.res_k_w;
      reinterpret_cast<uint4*>(to + dst)[c] = reinterpret_cast<const uint4*>(from + src)[c];
    }
  }

  constexpr int BITS = FMT;  // 8, 2 or 1
  const float levels = static_cast<float>((1 << BITS) - 1);
  const long long grp = p.Lq / G + gi;       // global group index
  const long long tok0 = p.Lq + static_cast<long long>(gi) * G;
  const float pinf = __int_as_float(0x7f800000);

  // ---- key statistics: per channel over the G tokens ----
  // thread = (channel pair cp, token stripe st); stripes combine through shared memory
  {
    const int npair = D / 2, nst = kFlushThreads / npair;   // 4 stripes (D=128) or 8 (D=64)
    const int cp = tid % npair, st = tid / npair;
    float mn0 = pinf, mx0 = -pinf, mn1 = pinf, mx1 = -pinf;
    for (int i = st; i < G; i += nst) {
      const uint32_t w = reinterpret_cast<const uint32_t*>(Ks + i * D)[cp];
      const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
      mn0 = fminf(mn0, x0); mx0 = fmaxf(mx0, x0);
      mn1 = fminf(mn1, x1); mx1 = fmaxf(mx1, x1);
    }
    part[st * D + 2 * cp] = mn0;
    part[st * D + 2 * cp + 1] = mn1;
    part[kFlushThreads * 2 + st * D + 2 * cp] = mx0;
    part[kFlushThreads * 2 + st * D + 2 * cp + 1] = mx1;
  }
  // ---- value statistics: per token over each block of G channels ----
  // item = (token i, block jv), D items; `per` adjacent lanes per item, each
  // over a multiple of 8 channels
  {
    const int per = min(kFlushThreads / D, G / 8);
    const int item = tid / per, sub = tid % per;
    const int i = item / NJ, jv = item % NJ;
    const int cw = G / per;
    const bool active = item < D;
    const uint16_t* src = Vs + (active ? i * D + jv * G + sub * cw : 0);
    float mn = pinf, mx = -pinf;
    for (int c = 0; active && c < cw; c += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(src + c);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x0 = __uint_as_float(ws[k] << 16), x1 = __uint_as_float(ws[k] & 0xFFFF0000u);
        mn = fminf(mn, fminf(x0, x1));
        mx = fmaxf(mx, fmaxf(x0, x1));
      }
    }
    for (int o = 1; o < per; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (active && sub == 0) {
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
  __syncthreads();
  if (tid < D) {
    const int nst = kFlushThreads / (D / 2);
    float mn = part[tid], mx = part[kFlushThreads * 2 + tid];
    for (int s2 = 1; s2 < nst; ++s2) {
      mn = fminf(mn, part[s2 * D + tid]);
      mx = fmaxf(mx, part[kFlushThreads * 2 + s2 * D + tid]);
    }
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    float scale, inv;
    scale_inv(mn, mx, levels, scale, inv);
    kmn[tid] = mn;
    kinv[tid] = inv;
    float* dst = p.ksz + (u * (p.C / G) + grp) * 2 * D;
    dst[tid] = scale;
    dst[D + tid] = mn;
  }
  __syncthreads();

  // ---- key codes: token-major rows, channels packed (8/pb per byte) ----
  if constexpr (FMT == KVQ_FMT_HIER8) {
    // Each thread writes one 32-bit word of both nibble planes: 8 channels.
    const int words = D / 8;
    for (int e = tid; e < G * words; e += kFlushThreads) {
      const int i = e / words, w = e % words;
      const uint4 x = reinterpret_cast<const uint4*>(Ks + i * D)[w];
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
      uint32_t hi = 0, lo = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int d = 8 * w + k;
        const uint32_t xb = (k & 1) ? (xs[k / 2] & 0xFFFF0000u) : (xs[k / 2] << 16);
        const uint32_t c = quant_code(__uint_as_float(xb), kmn[d], kinv[d], levels);
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
    for (int e = tid; e < G * words; e += kFlushThreads) {
      const int i = e / words, w = e % words;
      uint32_t v = 0;
#pragma unroll
      for (int k8 = 0; k8 < CPW; k8 += 8) {
        const uint4 x = reinterpret_cast<const uint4*>(Ks + i * D + CPW * w + k8)[0];
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int d = CPW * w + k8 + k;
          const uint32_t xb = (k & 1) ? (xs[k / 2] & 0xFFFF0000u) : (xs[k / 2] << 16);
          v |= quant_code(__uint_as_float(xb), kmn[d], kinv[d], levels) << (BITS * (k8 + k));
        }
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
      for (int e = tid; e < nslab * 4 * D; e += kFlushThreads) {
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
      for (int e = tid; e < nslab * WPR * D; e += kFlushThreads) {
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
                      (2 * p.D + 2 * p.G * (p.D / p.G) + 4 * kFlushThreads) * sizeof(float);
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
