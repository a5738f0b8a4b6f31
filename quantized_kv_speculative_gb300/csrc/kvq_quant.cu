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
constexpr int kKeyPart = 32;             // channels of one key part
constexpr int kStripes = kFlushThreads / (kKeyPart / 2);   // token stripes of the key statistics

__device__ __forceinline__ uint32_t quant_code(float x, float mn, float inv, float levels) {
  float t = rintf(__fmul_rn(__fsub_rn(x, mn), inv));
  t = fminf(fmaxf(t, 0.0f), levels);
  return static_cast<uint32_t>(t);
}

__device__ __forceinline__ void scale_inv(float mn, float mx, float levels, float& scale, float& inv) {
  scale = __fdiv_rn(__fsub_rn(mx, mn), levels);
  inv = (scale == 0.0f) ? 0.0f : __fdiv_rn(1.0f, scale);
}

// This CTA's sequence's part of the append: the launch's scalars, or its row
// of the per-sequence table for a ragged cache.
__device__ __forceinline__ SeqAppend seq_append(const FlushParams& p, int b) {
  if (p.ragged) return p.seq[b];
  SeqAppend a;
  a.lq = static_cast<int32_t>(p.Lq);
  a.r = static_cast<int16_t>(p.r);
  a.start = static_cast<int16_t>(p.res_start);
  a.n = p.n;
  a.nflush = p.nflush;
  a.first_new = p.first_new;
  a.res_count = p.res_count;
  return a;
}

// bf16 row of stream position pos: pos < r comes from the residual buffer (slot
// (res_start + pos) mod 2G), otherwise from the new tokens (index pos - r; the
// new tokens' rows are p.n apart per head).
__device__ __forceinline__ const uint16_t* stream_row(const FlushParams& p, const SeqAppend& sa, long long u, int pos,
                                                      bool value) {
  if (pos < sa.r) {
    const int slot = (sa.start + pos) % (2 * p.G);
    return (value ? p.res_v : p.res_k) + (u * 2 * p.G + slot) * p.D;
  }
  return (value ? p.v_new : p.k_new) + (u * p.n + (pos - sa.r)) * p.D;
}

// After this CTA has read its old residual slots: arrive at the head's counter;
// the last CTA of the head writes the new residual tokens and resets it.
__device__ void residual_ticket(const FlushParams& p, const SeqAppend& sa, long long u, int ncta, int* sh_flag) {
  if (sa.res_count <= 0) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.ctr + u, 1u);
    const int last = prev == static_cast<unsigned>(ncta - 1);
    if (last) atomicExch(p.ctr + u, 0u);
    *sh_flag = last;
  }
  __syncthreads();
  if (!*sh_flag) return;
  __threadfence();
  const int vec = p.D / 8;
  const int nv = sa.res_count * vec;
  for (int e = threadIdx.x; e < 2 * nv; e += kFlushThreads) {
    const int kv = e >= nv, e2 = kv ? e - nv : e;
    const int j = e2 / vec, c = e2 % vec;
    const int pos = sa.first_new + j;
    const int slot = (sa.start + pos) % (2 * p.G);
    const long long src = (u * p.n + (pos - sa.r)) * p.D;
    const long long dst = (u * 2 * p.G + slot) * p.D;
    const uint16_t* from = kv ? p.v_new : p.k_new;
    uint16_t* to = kv ? p.res_v_w : p.res_k_w;
    reinterpret_cast<uint4*>(to + dst)[c] = reinterpret_cast<const uint4*>(from + src)[c];
  }
}

// One CTA quantizes one part of one group of G tokens of one (b, kv head):
// blockIdx.x = group * (npk + npv) + part.
//  * key part: channels [32 kp, 32 kp + 32) over the G tokens; statistics by
//    (channel pair, token stripe), combined through shared memory;
//  * value part: one block of G channels over its tokens; statistics by
//    (token, lanes of the block).
template <int FMT>
__global__ void __launch_bounds__(kFlushThreads) flush_kernel(FlushParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int sh_flag;
  const int D = p.D, G = p.G, NJ = D / G;
  const FlushSplit sp = flush_split(D, G);
  const int npart = sp.npk + sp.npv;
  const int gi = blockIdx.x / npart, part = blockIdx.x % npart;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const long long u = static_cast<long long>(b) * p.Hkv + kvh;
  const int tid = threadIdx.x;
  const SeqAppend sa = seq_append(p, b);
  if (gi >= sa.nflush) return;               // a ragged sequence that flushes fewer groups
  constexpr int BITS = FMT;  // 8, 2 or 1
  const float levels = static_cast<float>((1 << BITS) - 1);
  const long long grp = sa.lq / G + gi;      // global group index
  const long long tok0 = static_cast<long long>(sa.lq) + static_cast<long long>(gi) * G;
  const float pinf = __int_as_float(0x7f800000);

  if (part < sp.npk) {
    // ---------------- key part ----------------
    const int c0 = part * kKeyPart;
    uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);              // [G][32]
    float* pmn = reinterpret_cast<float*>(Ks + G * kKeyPart);      // [kStripes][32]
    float* pmx = pmn + kStripes * kKeyPart;                        // [kStripes][32]
    float* kmn = pmx + kStripes * kKeyPart;                        // [32]
    float* kinv = kmn + kKeyPart;                                  // [32]
    // gather: 4 vectors per token, all in flight (G * 4 <= 2 * kFlushThreads)
    {
      uint4 v[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = tid + h * kFlushThreads;
        if (e < G * 4) v[h] = reinterpret_cast<const uint4*>(stream_row(p, sa, u, gi * G + e / 4, false) + c0)[e % 4];
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = tid + h * kFlushThreads;
        if (e < G * 4) reinterpret_cast<uint4*>(Ks)[e] = v[h];
      }
    }
    residual_ticket(p, sa, u, sa.nflush * npart, &sh_flag);
    __syncthreads();
    {
      const int cp = tid % (kKeyPart / 2), st = tid / (kKeyPart / 2);
      float mn0 = pinf, mx0 = -pinf, mn1 = pinf, mx1 = -pinf;
      for (int i = st; i < G; i += kStripes) {
        const uint32_t w = reinterpret_cast<const uint32_t*>(Ks + i * kKeyPart)[cp];
        const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
        mn0 = fminf(mn0, x0); mx0 = fmaxf(mx0, x0);
        mn1 = fminf(mn1, x1); mx1 = fmaxf(mx1, x1);
      }
      pmn[st * kKeyPart + 2 * cp] = mn0;
      pmn[st * kKeyPart + 2 * cp + 1] = mn1;
      pmx[st * kKeyPart + 2 * cp] = mx0;
      pmx[st * kKeyPart + 2 * cp + 1] = mx1;
    }
    __syncthreads();
    if (tid < kKeyPart) {
      float mn = pmn[tid], mx = pmx[tid];
      for (int s2 = 1; s2 < kStripes; ++s2) {
        mn = fminf(mn, pmn[s2 * kKeyPart + tid]);
        mx = fmaxf(mx, pmx[s2 * kKeyPart + tid]);
      }
      mn = __fadd_rn(mn, 0.0f);
      mx = __fadd_rn(mx, 0.0f);
      float scale, inv;
      scale_inv(mn, mx, levels, scale, inv);
      kmn[tid] = mn;
      kinv[tid] = inv;
      float* dst = p.ksz + (u * (p.C / G) + grp) * 2 * D;
      dst[c0 + tid] = scale;
      dst[D + c0 + tid] = mn;
    }
    __syncthreads();
    // ---- key codes: token-major rows, channels packed ----
    if constexpr (FMT == KVQ_FMT_HIER8) {
      // one 32-bit word of both nibble planes = 8 channels; 4 words per token
      for (int e = tid; e < G * 4; e += kFlushThreads) {
        const int i = e / 4, w = e % 4;
        const uint4 x = reinterpret_cast<const uint4*>(Ks + i * kKeyPart)[w];
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
        reinterpret_cast<uint32_t*>(p.kplane[0] + row)[c0 / 8 + w] = hi;
        reinterpret_cast<uint32_t*>(p.kplane[1] + row)[c0 / 8 + w] = lo;
      }
    } else {
      constexpr int PER = 8 / BITS;             // codes per byte
      constexpr int CPW = 4 * PER;              // codes per 32-bit word (16 or 32)
      constexpr int WPT = kKeyPart / CPW;       // words of this part per token
      const int rowbytes = D * BITS / 8;
      for (int e = tid; e < G * WPT; e += kFlushThreads) {
        const int i = e / WPT, w = e % WPT;
        uint32_t v = 0;
#pragma unroll
        for (int k8 = 0; k8 < CPW; k8 += 8) {
          const uint4 x = reinterpret_cast<const uint4*>(Ks + i * kKeyPart + CPW * w + k8)[0];
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int d = CPW * w + k8 + k;
            const uint32_t xb = (k & 1) ? (xs[k / 2] & 0xFFFF0000u) : (xs[k / 2] << 16);
            v |= quant_code(__uint_as_float(xb), kmn[d], kinv[d], levels) << (BITS * (k8 + k));
          }
        }
        reinterpret_cast<uint32_t*>(p.kplane[0] + (u * p.C + tok0 + i) * rowbytes)[c0 / CPW + w] = v;
      }
    }
    return;
  }

  // ---------------- value part ----------------
  const int vp = part - sp.npk;
  const int TV = sp.tv, CV = sp.cv;
  const int t0v = (NJ >= 2) ? 0 : 32 * vp;          // first token of the part (group-relative)
  const int c0v = (NJ >= 2) ? G * vp : 0;           // first channel (= its block's)
  const int jv = c0v / G;
  uint16_t* Vs = reinterpret_cast<uint16_t*>(smem);  // [TV][CV]
  float* vmn = reinterpret_cast<float*>(Vs + TV * CV);
  float* vinv = vmn + TV;
  {
    // gather: TV * CV / 8 <= 2 * kFlushThreads vectors, all in flight
    const int vpt = CV / 8;
    uint4 v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = tid + h * kFlushThreads;
      if (e < TV * vpt) v[h] = reinterpret_cast<const uint4*>(stream_row(p, sa, u, gi * G + t0v + e / vpt, true) + c0v)[e % vpt];
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = tid + h * kFlushThreads;
      if (e < TV * vpt) reinterpret_cast<uint4*>(Vs)[e] = v[h];
    }
  }
  residual_ticket(p, sa, u, sa.nflush * npart, &sh_flag);
  __syncthreads();
  // ---- statistics: per token over the block; `per` adjacent lanes per token ----
  {
    const int per = min(kFlushThreads / TV, CV / 8);
    const int i = tid / per, sub = tid % per;
    const int cw = CV / per;
    const bool active = i < TV;
    const uint16_t* src = Vs + (active ? i * CV + sub * cw : 0);
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
      vmn[i] = mn;
      vinv[i] = inv;
      float* dst = p.vsz + (u * p.C + tok0 + t0v + i) * 2 * NJ;
      dst[jv] = scale;
      dst[NJ + jv] = mn;
    }
  }
  __syncthreads();
  // ---- value codes: 32-token slabs, rows = channels, tokens packed ----
  {
    const int nslab = TV / 32;
    const long long slab0 = (u * p.C + tok0 + t0v) / 32;
    if constexpr (FMT == KVQ_FMT_HIER8) {
      // row = 16 bytes per plane = 4 words; word w holds tokens 8w..8w+7
      for (int e = tid; e < nslab * 4 * CV; e += kFlushThreads) {
        const int d = e % CV, w = (e / CV) % 4, s = e / (4 * CV);
        uint32_t hi = 0, lo = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = 32 * s + 8 * w + k;
          const uint32_t c = quant_code(bf16_to_f32(Vs[i * CV + d]), vmn[i], vinv[i], levels);
          hi |= (c >> 4) << (4 * k);
          lo |= (c & 15u) << (4 * k);
        }
        const long long off = ((slab0 + s) * D + c0v + d) * 16;
        reinterpret_cast<uint32_t*>(p.vplane[0] + off)[w] = hi;
        reinterpret_cast<uint32_t*>(p.vplane[1] + off)[w] = lo;
      }
    } else {
      constexpr int PER = 8 / BITS;
      constexpr int CPW = 4 * PER;            // tokens per word
      constexpr int WPR = 32 / CPW;           // words per slab row (2-bit: 2, 1-bit: 1)
      constexpr int ROWB = 32 * BITS / 8;
      for (int e = tid; e < nslab * WPR * CV; e += kFlushThreads) {
        const int d = e % CV, w = (e / CV) % WPR, s = e / (WPR * CV);
        uint32_t v = 0;
#pragma unroll
        for (int k = 0; k < CPW; ++k) {
          const int i = 32 * s + CPW * w + k;
          v |= quant_code(bf16_to_f32(Vs[i * CV + d]), vmn[i], vinv[i], levels) << (BITS * k);
        }
        reinterpret_cast<uint32_t*>(p.vplane[0] + ((slab0 + s) * D + c0v + d) * ROWB)[w] = v;
      }
    }
  }
}

// Copy the new tokens that stay in the residual buffer into their slots.
__global__ void residual_write_kernel(ResidualWriteParams p) {
  const int j = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const long long u = static_cast<long long>(b) * p.Hkv + kvh;
  const int r = p.ragged ? p.seq[b].r : p.r;
  const int start = p.ragged ? p.seq[b].start : p.res_start;
  const int first_new = p.ragged ? p.seq[b].first_new : p.first_new;
  const int count = p.ragged ? p.seq[b].res_count : p.count;
  if (j >= count) return;                             // a ragged sequence that keeps fewer tokens
  const int pos = first_new + j;                      // stream position
  const int slot = (start + pos) % (2 * p.G);
  const long long src = (u * p.n + (pos - r)) * p.D;
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
  const FlushSplit sp = flush_split(p.D, p.G);
  const size_t key_smem = static_cast<size_t>(p.G) * kKeyPart * 2 + (2 * kStripes + 2) * kKeyPart * 4;
  const size_t val_smem = static_cast<size_t>(sp.tv) * sp.cv * 2 + 2 * sp.tv * 4;
  const size_t smem = key_smem > val_smem ? key_smem : val_smem;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&flush_kernel<FMT>), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.nflush * (sp.npk + sp.npv), p.Hkv, p.B);
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
