#pragma once
// The attention kernel template (fused dequantization + split-K
// flash-decoding attention with a fused combine) and its per-variant launch
// helpers.  Each read mode's variants are instantiated in a translation unit of
// their own (kvq_attend_<mode>.cu) so that they compile in parallel; the
// dispatch over modes is in kvq_attend.cu.
//
// Fused dequantization + split-K flash-decoding attention over the quantized
// KV cache, with a fused combine.
//
// The pages: the INT4 draft reads only the upper 4-bit cache and the INT8
// target reads upper + lower nibbles (QuantSpec page, "Approach" and the kernel
// rows of the "Measured effects" table).  FlashDecoding-style split-K ("Builds
// on: FlashAttention FlashDecoding", QuantSpec page, "Experimental setup").  The
// low-bit copy is attended with the output token and a speculative token, and
// the top-k tokens use their 16-bit KV (SpeCache page, "Approach").
//
// One launch of B*Hkv*(S_q + S_t) CTAs: per (b, kvh) S_q quantized splits and
// S_t tail CTAs, either as one thread-block cluster per (b, kvh) or (when the
// clusters would not fit in the waves the split plan assumed, or S_q + S_t > 16)
// as a plain grid with the tail CTAs after the quantized splits.
//  * Quantized split: four warps each own a contiguous run of 32..64-token
//    tiles; each warp's lane 0 streams its tiles of the mode's planes and
//    scales into the warp's ring of shared-memory slots with 1-D bulk (TMA)
//    copies on mbarriers.  The warps turn codes into f16 in registers and run
//    QK^T and PV on tensor cores (m16n8k16): keys are the A operand (16 tokens
//    x 16 channels) against the folded query weights, values the A operand of
//    O^T = V^T P^T.  The folded weights and the folded probabilities are each
//    split into high + low f16 parts.  Softmax is online in fp32 (base-2
//    logits).
//  * The bf16 tail (residual buffer, pending speculative tokens (causal) and
//    16-bit selected tokens) runs as bf16 m16n8k16 MMAs, either in tail CTAs
//    or shared out over the quantized splits.
//  * Every CTA makes an (m, l, o) partial.  In a cluster the partials stay in
//    shared memory: after a cluster barrier each CTA merges its share of the
//    output items from all of them.  Otherwise they go to the workspace and the
//    CTA that arrives last at a per-(b, kvh) atomic ticket merges them into the
//    bf16 output and LSE, then resets the ticket; no CTA waits on another.
//
// Folding (no per-element dequant FMA).  Codes enter the tensor cores as f16
// subnormals: a key code c of channel d reads as E_d = c f_d 2^-24, with f_d a
// power of two set by the code's bit position in its word.  With
// q~ = q * sm_scale * log2(e), step s (MULT x scale) and zero z per group and
// channel:
//   logit2 = sum_d q~_d (c s + z) = 2^24 sum_d (q~_d s_d / f_d) E_d + sum_d q~_d z_d,
// so the B operand holds w_d = q~_d s_d / f_d (scaled by 2^e) and the
// zero-point sum starts the accumulator.  Value codes read the same way, as
// c m 2^-24 (m the pair's factor), against P'_t = p_t s_t / m_t:
//   o = sum_t p_t (c s + z) = 2^24 sum_t P'_t (c m 2^-24) + sum_t p_t z_t.
// No offset has to be removed, so the accumulators carry only the code terms.
#include "kvq_modes.cuh"

namespace kvq {
namespace {

constexpr int NW = 4;                  // warps per CTA; each streams and consumes its own tiles
constexpr int NTHREADS = NW * 32;
constexpr int kSmemPerSm = 228 * 1024;
// q~ in shared memory: row stride D + 4 floats, each quarter (D/4 channels,
// one lane chunk) padded by one float, so that the lanes deriving weights
// (different rows and chunks, the same channel offset) hit different banks.
template <int D> __host__ __device__ constexpr int qt_row() { return D + 4; }
template <int D> __host__ __device__ constexpr int qt_chunk() { return D / 4 + 1; }

template <int MODE, int D, int NJ, int NT, bool SC>
struct Smem;

// Target CTAs per SM: with one weight n-tile (rows <= 4) as many as fit, up to
// four; with two n-tiles three when their shared memory fits, else two (which
// also frees registers).
template <int MODE, int D, int NJ, int NT, bool SC>
constexpr int target_ctas() {
  constexpr int need = Smem<MODE, D, NJ, NT, SC>::MIN_TOTAL + 1024;
  if constexpr (NT == 1) {
    return 4 * need <= 228 * 1024 ? 4 : (3 * need <= 228 * 1024 ? 3 : 2);
  } else {
    return 3 * need <= 228 * 1024 ? 3 : 2;
  }
}

template <int MODE, int D, int NJ, int NT, bool SC>
struct Smem {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  static constexpr int TT = M::TT;
  static constexpr int KPLANE = TT * RW::KROW;
  static constexpr int VPLANE = (TT / 32) * D * RW::VROW;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = M::NP * KPLANE;
  static constexpr int KSZ_OFF = V_OFF + M::NP * VPLANE;
  static constexpr int G = D / NJ;
  static constexpr int KSZ_BYTES = (TT > G ? TT / G : 1) * 2 * D * 4;   // key groups a tile touches
  static constexpr int VSZ_OFF = KSZ_OFF + KSZ_BYTES;
  static constexpr int VSZ_BYTES = TT * 2 * NJ * 4;
  static constexpr int SLOT = VSZ_OFF + VSZ_BYTES;
  static constexpr int WB_BYTES = NT == 1 ? NW * 16 * D : 0;     // staged weight fragments (one n-tile)
  static constexpr int SQ_BYTES = SC ? D * 4 : 0;                // scoring: the score row's summed query
  static constexpr int SW_BYTES = SC ? NW * 3 * D * 2 : 0;       // scoring: per warp, 3 integer weight parts (f16)
  static constexpr int BM_WORDS = (NT == 2 ? kMaxChunkWide : kMaxChunk) / 32;   // selection bitmap words
  static constexpr int FIXED =
      kMaxRows * qt_row<D>() * 4 + BM_WORDS * 4 + 16 * 8 + WB_BYTES + SQ_BYTES + SW_BYTES + NW * 48 + 272;
  static constexpr int MIN_TOTAL = NW * 2 * SLOT + FIXED;
  // stage slots per warp: as many as fit (2..4) at the target CTAs per SM
  static constexpr int SPW_FIT = (kSmemPerSm / target_ctas<MODE, D, NJ, NT, SC>() - 1024 - FIXED) / (NW * SLOT);
  static constexpr int SPW_BASE = SPW_FIT < 2 ? 2 : (SPW_FIT > 4 ? 4 : SPW_FIT);
  // the slot area is reused for the merge scratch: 2 NW entries (the warps'
  // quantized runs, then the warps' shares of the bf16 tail)
  static constexpr int NENT = 2 * NW;
  static constexpr int SCRATCH_NEED = NENT * 8 * 4 * 7 + NENT * 8 * D * 4;
  static constexpr int SPW_SCR = (SCRATCH_NEED + NW * SLOT - 1) / (NW * SLOT);
  static constexpr int SPW = SPW_BASE > SPW_SCR ? SPW_BASE : SPW_SCR;
  static constexpr int NSLOT = NW * SPW;
  static constexpr int QT_OFF = NSLOT * SLOT;                 // scaled queries q~ [8][qt_row] f32
  static constexpr int BM_OFF = QT_OFF + kMaxRows * qt_row<D>() * 4;   // selection bitmap
  static constexpr int BAR_OFF = BM_OFF + BM_WORDS * 4;
  static constexpr int WB_OFF = (BAR_OFF + NSLOT * 8 + 15) / 16 * 16;   // per warp: staged weight fragments
  static constexpr int SQ_OFF = WB_OFF + WB_BYTES;                  // scoring: summed query [D] f32
  static constexpr int SW_OFF = SQ_OFF + SQ_BYTES;                  // scoring: per warp [3][D] f16, pair order
  static constexpr int QM_OFF = SW_OFF + SW_BYTES;                  // per warp: max |q~| (f32)
  static constexpr int RING_END = QM_OFF + NW * 4;
  static constexpr int COMBINE_END = (2 * kMaxCombine * 8 + 16) * 4;
  // the ticket flag sits after whichever layout (ring, combine) is largest
  static constexpr int MISC_OFF = (RING_END > COMBINE_END ? RING_END + 15 : COMBINE_END + 15) / 16 * 16;
  static constexpr int TOTAL = MISC_OFF + 64;
  // merge scratch (after the pipeline drains), inside the slot area
  static constexpr int WM_OFF = 0;                            // [NENT][8] running max
  static constexpr int WL_OFF = WM_OFF + NENT * 8 * 4;        // [NENT][8] running sum
  static constexpr int WC_OFF = WL_OFF + NENT * 8 * 4;        // [NENT][8][4] value zero-point terms
  static constexpr int FAC_OFF = WC_OFF + NENT * 8 * 4 * 4;   // [NENT][8] entry factors 2^(m_w - M)
  static constexpr int WO_OFF = FAC_OFF + NENT * 8 * 4;       // [NENT][8][D] output sums
  static constexpr int SCRATCH = WO_OFF + NENT * 8 * D * 4;
  static_assert(SCRATCH <= NSLOT * SLOT, "the merge scratch must fit in the slot area");
  static_assert((2 * kMaxCombine * 8 + 16) * 4 <= MISC_OFF, "the combine scratch must not reach the ticket flag");
  static_assert(SLOT % 16 == 0, "slots must stay 16-byte aligned");
  static_assert(kMaxRows * qt_row<D>() >= kPartialFloats(D), "a CTA's partial must fit in the q~ area");
};

// 2^x with the hardware approximation (ex2.approx.ftz: relative error near
// 2^-22; -inf gives +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// True when the second half of a lane chunk's key pairs uses the first half's
// channels shifted by one constant (the eight-row weight setup splits the pairs
// between two lanes that way).
template <int MODE, int D>
__host__ __device__ constexpr bool halves_shift() {
  constexpr int HP = D / 16;
  for (int k = 0; k < HP; ++k)
    for (int e = 0; e < 2; ++e)
      if (kx_chan<MODE, D>(HP + k, e) != kx_chan<MODE, D>(k, e) + kx_chan<MODE, D>(HP, 0)) return false;
  return kx_chan<MODE, D>(0, 0) == 0;
}

// True when the second half of a lane chunk's key pairs carries the first
// half's code factors (the eight-row weight setup scales both halves alike).
template <int MODE, int D>
__host__ __device__ constexpr bool halves_same_factors() {
  constexpr int HP = D / 16;
  for (int k = 0; k < HP; ++k)
    if (ks_log2fac<MODE, D>(HP + k) != ks_log2fac<MODE, D>(k)) return false;
  return true;
}

// Floats of a lane's first-half key pairs, counted from the half's base and
// rounded up to whole float4s: the eight-row weight setup loads that window
// of the key scale and zero rows with 128-bit loads.
template <int MODE, int D>
__host__ __device__ constexpr int half_window() {
  int m = 0;
  for (int k = 0; k < D / 16; ++k)
    for (int e = 0; e < 2; ++e) m = kx_chan<MODE, D>(k, e) + 1 > m ? kx_chan<MODE, D>(k, e) + 1 : m;
  return (m + 3) / 4 * 4;
}

// A token's value scales then zero points (2 NJ floats, 8 NJ-byte aligned) as
// 64- or 128-bit shared loads.
template <int NJ>
__device__ __forceinline__ void load_vrow(const float* v, float (&out)[2 * NJ]) {
  if constexpr (NJ == 1) {
    const float2 x = *reinterpret_cast<const float2*>(v);
    out[0] = x.x; out[1] = x.y;
  } else {
#pragma unroll
    for (int i = 0; i < NJ / 2; ++i) {
      const float4 x = reinterpret_cast<const float4*>(v)[i];
      out[4 * i] = x.x; out[4 * i + 1] = x.y; out[4 * i + 2] = x.z; out[4 * i + 3] = x.w;
    }
  }
}

// The queries of unit (b, kvh) as 16-byte slices of 8 channels: slice e is
// row e / (D/8) (zero for rows >= R); one slice per thread (8 rows x D/8
// slices <= 128 threads).  load_q issues the load, so that it is in flight
// while the copies of the first tiles are issued; store_qt writes the scaled
// queries q~ = q * sm_scale * log2(e) into qt [8][qt_row] (no store when qt is
// null) and returns the slice's max |q~|.
template <int D>
__device__ __forceinline__ uint4 load_q(const AttendParams& p, int b, int kvh, int e) {
  constexpr int V8 = D / 8;
  const int rho = e / V8, c = e % V8;
  if (e >= kMaxRows * V8 || rho >= p.R) return make_uint4(0u, 0u, 0u, 0u);
  const int i = rho / p.HG, hh = rho % p.HG;
  const long long qrow = ((static_cast<long long>(b) * p.gamma + i) * p.Hq + kvh * p.HG + hh) * D;
  return *reinterpret_cast<const uint4*>(p.q + qrow + 8 * c);
}

template <int D>
__device__ __forceinline__ float store_qt(const AttendParams& p, int e, const uint4& w, float* qt) {
  constexpr int V8 = D / 8;
  if (e >= kMaxRows * V8) return 0.f;
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  float v[8], qm = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = __uint_as_float(ww[k] << 16) * p.qscale;
    v[2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u) * p.qscale;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) qm = fmaxf(qm, fabsf(v[k]));
  if (qt) {
    const int ch = 8 * (e % V8);   // 8 channels within one quarter
    float* dst = qt + (e / V8) * qt_row<D>() + (ch / (D / 4)) * qt_chunk<D>() + ch % (D / 4);
#pragma unroll
    for (int k = 0; k < 8; ++k) dst[k] = v[k];
  }
  return qm;
}

// ------------------------------------------------------------------------------
// Combine: merge the S_total partials of unit u into out/lse.  The split
// maxima and weights are staged in shared memory (S_total <= 256); each thread
// owns up to two float4 items of the output.  With PREFETCH (the eight-row
// variants, which have the registers to spare) and at most 10 splits the
// items' partial outputs are loaded first, together with the maxima, so the
// combine takes one round trip to L2; otherwise they stream after the weights
// with several splits in flight.
// ------------------------------------------------------------------------------
// Writes one output item of unit (b, kvh): row rho, channels 4 d4 .. 4 d4 + 3,
// and for d4 = 0 the row's LSE from its base-2 max M and sum L.
template <int D>
__device__ __forceinline__ void put_item(const AttendParams& p, int b, int kvh, int rho, int d4, const float4& acc,
                                         float M, float L) {
  const int i = rho / p.HG, hh = rho % p.HG;
  const int h = kvh * p.HG + hh;
  const long long orow = (static_cast<long long>(b) * p.gamma + i) * p.Hq + h;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p.out + orow * D + 4 * d4) = pk;
  if (p.lse && d4 == 0) p.lse[orow] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : neg_inf();
}

template <int D, bool PREFETCH>
__device__ void combine_unit(const AttendParams& p, long long u, int S_total, float* sm) {
  constexpr int D4 = D / 4;
  constexpr int kPF = PREFETCH ? 10 : 1;   // partial outputs prefetched per item (up to kPF splits)
  const int PF = kPartialFloats(D);
  const float* base = p.partials + u * static_cast<long long>(S_total) * PF;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  float* ms = sm;                       // [S_total][8] split maxima
  float* wt = sm + kMaxCombine * 8;     // [S_total][8] l, then weights
  float* ml = wt + kMaxCombine * 8;     // M[8], L[8]
  const int tid = threadIdx.x;
  const int nitems = p.R * D4;          // <= 2 per thread (R <= 8, D <= 128, 128 threads)
  // With few splits, each thread's partial outputs are loaded before the
  // weights are known, so that all loads are in flight together.
  const bool pf = PREFETCH && S_total <= kPF;
  float4 pre[2][kPF];
  // Otherwise tpi adjacent lanes share an item (few rows leave threads spare)
  // and split its partials between them; the first round's first kPFS partial
  // outputs per lane are loaded here too, before the weights are known.
  constexpr int kPFS = 8;
  const int spare = static_cast<int>(blockDim.x) / max(1, nitems);
  const int tpi = spare >= 8 ? 8 : (spare >= 4 ? 4 : (spare >= 2 ? 2 : 1));
  const int per_round = static_cast<int>(blockDim.x) / tpi;
  float4 pre0[kPFS];
  if (!pf && tid / tpi < nitems) {
    const int item = tid / tpi, part = tid % tpi;
    const float4* src = reinterpret_cast<const float4*>(base + 2 * kMaxRows + (item / D4) * D) + item % D4;
#pragma unroll
    for (int i = 0; i < kPFS; ++i) {
      const int s = part + i * tpi;
      if (s < S_total) pre0[i] = __ldcg(src + static_cast<long long>(s) * (PF / 4));
    }
  }
  if (pf) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int item = tid + k * static_cast<int>(blockDim.x);
      if (item < nitems) {
        const float4* src = reinterpret_cast<const float4*>(base + 2 * kMaxRows + (item / D4) * D) + item % D4;
#pragma unroll
        for (int s = 0; s < kPF; ++s)
          if (s < S_total) pre[k][s] = __ldcg(src + static_cast<long long>(s) * (PF / 4));
      }
    }
  }
  for (int e = tid; e < S_total * 8; e += blockDim.x) {
    const int s = e >> 3, r = e & 7;
    ms[e] = __ldcg(base + s * PF + r);
    wt[e] = __ldcg(base + s * PF + kMaxRows + r);
  }
  __syncthreads();
  // the split weights of each row: warp w takes rows w, w + NW, its lanes the splits
  {
    const int lane = tid % 32;
    for (int rho = tid / 32; rho < p.R; rho += NW) {
      float M = neg_inf();
      for (int s = lane; s < S_total; s += 32) M = fmaxf(M, ms[s * 8 + rho]);
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
      float L = 0.f;
      if (M != neg_inf()) {
        for (int s = lane; s < S_total; s += 32) {
          const float m = ms[s * 8 + rho];
          const float f = (m == neg_inf()) ? 0.f : fast_exp2(m - M);
          L = fmaf(f, wt[s * 8 + rho], L);
          wt[s * 8 + rho] = f;
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
      }
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
      for (int s = lane; s < S_total; s += 32) wt[s * 8 + rho] = (M == neg_inf()) ? 0.f : wt[s * 8 + rho] * inv;
      if (lane == 0) {
        ml[rho] = M;
        ml[8 + rho] = L;
      }
    }
  }
  __syncthreads();
  auto put = [&](int rho, int d4, const float4& acc) { put_item<D>(p, b, kvh, rho, d4, acc, ml[rho], ml[8 + rho]); };
  if (pf) {   // items tid and tid + blockDim, from the prefetched partials
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int item = tid + k * static_cast<int>(blockDim.x);
      if (item >= nitems) continue;
      const int rho = item / D4, d4 = item % D4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < kPF; ++s) {
        if (s < S_total) {
          const float w = wt[s * 8 + rho];
          acc.x = fmaf(w, pre[k][s].x, acc.x);
          acc.y = fmaf(w, pre[k][s].y, acc.y);
          acc.z = fmaf(w, pre[k][s].z, acc.z);
          acc.w = fmaf(w, pre[k][s].w, acc.w);
        }
      }
      put(rho, d4, acc);
    }
    return;
  }
  // Streaming: the first round takes its prefetched partials, then every
  // round streams the rest.
  for (int k = 0; k * per_round < nitems; ++k) {
    const int item = k * per_round + tid / tpi, part = tid % tpi;
    const bool valid = item < nitems;
    const int rho = valid ? item / D4 : 0, d4 = valid ? item % D4 : 0;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
      const float4* src = reinterpret_cast<const float4*>(base + 2 * kMaxRows + rho * D) + d4;
      int s0 = part;
      if (k == 0) {
#pragma unroll
        for (int i = 0; i < kPFS; ++i) {
          const int s = part + i * tpi;
          if (s < S_total) {
            const float w = wt[s * 8 + rho];
            acc.x = fmaf(w, pre0[i].x, acc.x);
            acc.y = fmaf(w, pre0[i].y, acc.y);
            acc.z = fmaf(w, pre0[i].z, acc.z);
            acc.w = fmaf(w, pre0[i].w, acc.w);
          }
        }
        s0 = part + kPFS * tpi;
      }
#pragma unroll 8
      for (int s = s0; s < S_total; s += tpi) {
        const float w = wt[s * 8 + rho];
        const float4 v = __ldcg(src + static_cast<long long>(s) * (PF / 4));
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
    for (int o2 = 1; o2 < tpi; o2 <<= 1) {   // the lanes of one item are adjacent
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o2);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o2);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o2);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o2);
    }
    if (valid && part == 0) put(rho, d4, acc);
  }
}

// Cluster combine: the S_total CTAs of unit u form one cluster and each holds
// its partial in shared memory at `part` (the same offset in every CTA).
// After the cluster barrier, CTA `rank` merges its share of the output items
// (float4 of one row), reading the maxima, sums and outputs of every CTA
// through distributed shared memory: tpi adjacent lanes share an item, each
// taking at most four of the partials, and reduce by shuffles.  The second
// barrier keeps every CTA's shared memory alive until all reads are done.
template <int D>
__device__ void cluster_combine(const AttendParams& p, long long u, int S_total, const float* part) {
  constexpr int D4 = D / 4;
  constexpr int KP = kMaxClusterCtas / 4;   // partials per lane
  static_assert(kMaxClusterCtas % 4 == 0, "four lanes share the partials of an item");
  cluster_sync();
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  const int rank = static_cast<int>(cluster_rank());
  const int n = p.R * D4, per = (n + S_total - 1) / S_total;
  const int lo = rank * per, hi = min(n, lo + per);
  const int tpi = S_total <= KP ? 1 : (S_total <= 2 * KP ? 2 : 4);
  const int tid = threadIdx.x, sub = tid % tpi;
  for (int base = lo; base < hi; base += NTHREADS / tpi) {   // the same trip count in every warp
    const int item = base + tid / tpi;
    const bool valid = item < hi;
    const int rho = valid ? item / D4 : 0, d4 = valid ? item % D4 : 0;
    float m[KP], l[KP];
    float4 o[KP];
    float M = neg_inf();
#pragma unroll
    for (int k = 0; k < KP; ++k) {
      const int s = sub + k * tpi;
      if (valid && s < S_total) {
        m[k] = ld_dsmem(dsmem_addr(part + rho, s));
        l[k] = ld_dsmem(dsmem_addr(part + kMaxRows + rho, s));
        o[k] = ld_dsmem4(dsmem_addr(part + 2 * kMaxRows + rho * D + 4 * d4, s));
      } else {
        m[k] = neg_inf();
        l[k] = 0.f;
        o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      M = fmaxf(M, m[k]);
    }
    for (int o2 = 1; o2 < tpi; o2 <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < KP; ++k) {
      const float f = (m[k] == neg_inf()) ? 0.f : fast_exp2(m[k] - M);
      L = fmaf(f, l[k], L);
      acc.x = fmaf(f, o[k].x, acc.x);
      acc.y = fmaf(f, o[k].y, acc.y);
      acc.z = fmaf(f, o[k].z, acc.z);
      acc.w = fmaf(f, o[k].w, acc.w);
    }
    for (int o2 = 1; o2 < tpi; o2 <<= 1) {
      L += __shfl_xor_sync(0xffffffffu, L, o2);
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o2);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o2);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o2);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o2);
    }
    if (valid && sub == 0) {
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      put_item<D>(p, b, kvh, rho, d4, acc, M, L);
    }
  }
  cluster_sync();
}

// Arrive at the per-unit ticket; the last arriving CTA merges and resets it.
template <int D, bool PREFETCH>
__device__ void ticket_and_combine(const AttendParams& p, long long u, int* sh_flag, float* combine_scratch) {
  __threadfence();
  __syncthreads();
  const int S_total = p.S_q + p.S_t;
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(p.counters + u, 1u);
    const int last = (prev == static_cast<unsigned>(S_total - 1));
    if (last) atomicExch(p.counters + u, 0u);
    *sh_flag = last;
  }
  __syncthreads();
  if (*sh_flag) {
    __threadfence();
    combine_unit<D, PREFETCH>(p, u, S_total, combine_scratch);
  }
}

// ------------------------------------------------------------------------------
// The bf16 tail: the residual buffer, then the pending speculative tokens
// (causal among themselves), then the selected 16-bit tokens.
// ------------------------------------------------------------------------------
// K / V rows of tail token t of unit u; returns its visibility: -1 always
// visible, >= 0 the pending index, -2 absent (a selected slot without a token).
template <int D>
__device__ __forceinline__ int tail_row(const AttendParams& p, long long u, int t, const uint16_t*& kp,
                                        const uint16_t*& vp) {
  const int b = static_cast<int>(u / p.c.Hkv);
  const int r = seq_r(p.c, b);
  if (t < r) {
    const int slot = (seq_start(p.c, b) + t) % (2 * p.c.G);
    const long long off = (u * 2 * p.c.G + slot) * D;
    kp = p.c.res_k + off;
    vp = p.c.res_v + off;
    return -1;
  }
  t -= r;
  if (t < p.P) {
    const long long off = (u * p.P + t) * D;
    kp = p.pend_k + off;
    vp = p.pend_v + off;
    return t;
  }
  t -= p.P;
  const int idx = p.sel_idx[u * p.top_k + t];
  if (idx >= 0 && idx < seq_lq(p.c, b)) {
    const long long off = (u * p.top_k + t) * D;
    kp = p.sel_k + off;
    vp = p.sel_v + off;
    return -1;
  }
  kp = vp = nullptr;
  return -2;
}

// Tail tokens [t_lo, t_hi) of unit u on tensor cores (bf16 in, f32 out), 16
// tokens per warp step, steps dealt round-robin to the warps.  Each warp ends
// with its own (m, l, o) in merge entry entry0 + warp.
//  * S = K Q^T: keys are the A operand straight from global memory (lane
//    (g, q) holds tokens g and g + 8, its quarter D/4 of the channels); the
//    queries are the B operand over the same channel permutation.
//  * O^T = V^T P^T: 8x8 blocks of value rows are transposed in registers
//    (movmatrix), so m-tile 2i + jp row g is channel
//    32 i + 8 (g >> 1) + 4 jp + (g & 1) (row g + 8: that + 2).  P^T comes
//    from the logit fragments by the same transpose, split into high + low
//    bf16 parts.
template <int D>
__device__ void tail_entries(const AttendParams& p, long long u, int t_lo, int t_hi, float* wm, float* wl,
                             float* wc, float* wo, int entry0) {
  constexpr int KS = D / 16;   // k-steps of S, m-tiles of O^T
  constexpr int QC = D / 4;    // channels of a lane's key / query quarter
  constexpr int VC = D / 32;   // 16-byte value chunks per lane and row
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, q = lane & 3;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  const int R = p.R;
  uint32_t qf[QC / 2];   // query row g, channels q QC .. q QC + QC - 1, bf16 pairs
  if (g < R) {
    const int i = g / p.HG, hh = g % p.HG;
    const long long qrow = ((static_cast<long long>(b) * p.gamma + i) * p.Hq + kvh * p.HG + hh) * D;
    const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow + q * QC);
#pragma unroll
    for (int c = 0; c < QC / 8; ++c) {
      const uint4 w = src[c];
      qf[4 * c] = w.x;
      qf[4 * c + 1] = w.y;
      qf[4 * c + 2] = w.z;
      qf[4 * c + 3] = w.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < QC / 2; ++c) qf[c] = 0u;
  }
  float m_run[2] = {neg_inf(), neg_inf()}, l_run[2] = {0.f, 0.f};
  float o[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  const int nsteps = (t_hi - t_lo + 15) / 16;
  for (int st = warp; st < nsteps; st += NW) {
    const int t0 = t_lo + 16 * st;
    uint4 kr[2][QC / 8], vr[2][VC];
    int flag[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + g + 8 * h;
      const uint16_t *kp = nullptr, *vp = nullptr;
      flag[h] = (t < t_hi) ? tail_row<D>(p, u, t, kp, vp) : -2;
#pragma unroll
      for (int c = 0; c < QC / 8; ++c)
        kr[h][c] = kp ? reinterpret_cast<const uint4*>(kp + q * QC)[c] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int i = 0; i < VC; ++i)
        vr[h][i] = vp ? *reinterpret_cast<const uint4*>(vp + 32 * i + 8 * q) : make_uint4(0u, 0u, 0u, 0u);
    }
    // ---- S: tokens g, g + 8 x rows 2q, 2q + 1 ----
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const uint32_t* k0 = reinterpret_cast<const uint32_t*>(&kr[0][0]);
      const uint32_t* k1 = reinterpret_cast<const uint32_t*>(&kr[1][0]);
      const uint32_t a[4] = {k0[2 * kk], k1[2 * kk], k0[2 * kk + 1], k1[2 * kk + 1]};
      mma16816_bf16(sc, a, qf[2 * kk], qf[2 * kk + 1]);
    }
    float x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int h = e >> 1, rho = 2 * q + (e & 1);
      bool vis = (flag[h] != -2) && (rho < R);
      if (vis && flag[h] >= 0) vis = flag[h] <= p.P - p.gamma + rho / p.HG;
      x[e] = vis ? sc[e] * p.qscale : neg_inf();
    }
    // ---- online softmax of rows 2q, 2q + 1 (the 8 lanes of this q) ----
    float alpha[2], pr[4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = fmaxf(x[r], x[r + 2]);
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      const float m_new = fmaxf(m_run[r], mx);
      const float msafe = (m_new == neg_inf()) ? 0.f : m_new;
      alpha[r] = (m_run[r] == neg_inf()) ? 0.f : fast_exp2(m_run[r] - msafe);
      pr[r] = fast_exp2(x[r] - msafe);
      pr[r + 2] = fast_exp2(x[r + 2] - msafe);
      l_run[r] = l_run[r] * alpha[r] + (pr[r] + pr[r + 2]);
      m_run[r] = m_new;
    }
    // ---- P^T fragments: (tokens 2q, 2q + 1; row g), high and low parts ----
    uint32_t ph[2], pl[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(pr[2 * h]), h1 = __float2bfloat16_rn(pr[2 * h + 1]);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(pr[2 * h] - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(pr[2 * h + 1] - __bfloat162float(h1));
      ph[h] = transpose8x8(static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                           (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16));
      pl[h] = transpose8x8(static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                           (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16));
    }
    // ---- O^T += V^T P^T, a fresh accumulator per step ----
#pragma unroll
    for (int i = 0; i < VC; ++i) {
      const uint32_t* v0 = reinterpret_cast<const uint32_t*>(&vr[0][i]);
      const uint32_t* v1 = reinterpret_cast<const uint32_t*>(&vr[1][i]);
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        const int mt = 2 * i + jp;
        const uint32_t a[4] = {transpose8x8(v0[2 * jp]), transpose8x8(v0[2 * jp + 1]), transpose8x8(v1[2 * jp]),
                               transpose8x8(v1[2 * jp + 1])};
        float os[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816_bf16(os, a, ph[0], ph[1]);
        mma16816_bf16(os, a, pl[0], pl[1]);
        o[mt][0] = fmaf(o[mt][0], alpha[0], os[0]);
        o[mt][1] = fmaf(o[mt][1], alpha[1], os[1]);
        o[mt][2] = fmaf(o[mt][2], alpha[0], os[2]);
        o[mt][3] = fmaf(o[mt][3], alpha[1], os[3]);
      }
    }
  }
  // ---- this warp's entry ----
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], o2);
  const int e = entry0 + warp;
  if (g == 0) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      wm[e * 8 + 2 * q + r] = m_run[r];
      wl[e * 8 + 2 * q + r] = l_run[r];
#pragma unroll
      for (int jv = 0; jv < 4; ++jv) wc[(e * 8 + 2 * q + r) * 4 + jv] = 0.f;
    }
  }
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    const int ch = 32 * (mt >> 1) + 8 * (g >> 1) + 4 * (mt & 1) + (g & 1);
    wo[(e * 8 + 2 * q) * D + ch] = o[mt][0];
    wo[(e * 8 + 2 * q + 1) * D + ch] = o[mt][1];
    wo[(e * 8 + 2 * q) * D + ch + 2] = o[mt][2];
    wo[(e * 8 + 2 * q + 1) * D + ch + 2] = o[mt][3];
  }
}

// Where partial `part` of unit u goes: this CTA's shared memory (`local`) when
// the unit's CTAs form a cluster, else the workspace.
template <int D>
__device__ __forceinline__ float* partial_dst(const AttendParams& p, long long u, int part, float* local) {
  return p.cluster ? local : p.partials + (u * (p.S_q + p.S_t) + part) * kPartialFloats(D);
}

// The unit's partials into the output: through the cluster's shared memory, or
// through the workspace and the atomic ticket.
template <int D, bool PREFETCH>
__device__ __forceinline__ void finish_unit(const AttendParams& p, long long u, int* sh_flag, float* combine_scratch,
                                            const float* local) {
  if (p.cluster)
    cluster_combine<D>(p, u, p.S_q + p.S_t, local);
  else
    ticket_and_combine<D, PREFETCH>(p, u, sh_flag, combine_scratch);
}

// Merge entries [0, nent) of the shared scratch into the partial at dst.
static_assert(2 * NW <= 8, "a CTA's merge entries fit in eight lanes");
template <int D>
__device__ void merge_to_partial(const AttendParams& p, float* dst, int nent, int G, const float* wm,
                                 const float* wl, const float* wc, const float* wo, float* fac) {
  const int tid = threadIdx.x, R = p.R;
  {
    // the entries' factors of each row: warp w takes rows w, w + NW, lane i
    // entry i (nent <= 2 NW <= 8)
    const int lane = tid % 32;
    for (int rho = tid / 32; rho < R; rho += NW) {
      const float mw = lane < nent ? wm[lane * 8 + rho] : neg_inf();
      float Mx = mw;
#pragma unroll
      for (int o2 = 4; o2 > 0; o2 >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o2));
      const float f = (mw == neg_inf()) ? 0.f : fast_exp2(mw - Mx);
      float lt = lane < nent ? f * wl[lane * 8 + rho] : 0.f;
#pragma unroll
      for (int o2 = 4; o2 > 0; o2 >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o2);
      if (lane < nent) fac[lane * 8 + rho] = f;
      if (lane == 0) {
        dst[rho] = Mx;
        dst[kMaxRows + rho] = lt;
      }
    }
  }
  __syncthreads();
  for (int e = 4 * tid; e < R * D; e += 4 * NTHREADS) {
    const int rho = e / D, d = e % D;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int w = 0; w < nent; ++w) {
      const float f = fac[w * 8 + rho];
      const float c = wc[(w * 8 + rho) * 4 + d / G];
      const float4 ov = *reinterpret_cast<const float4*>(wo + (w * 8 + rho) * D + d);
      acc.x = fmaf(f, ov.x + c, acc.x);
      acc.y = fmaf(f, ov.y + c, acc.y);
      acc.z = fmaf(f, ov.z + c, acc.z);
      acc.w = fmaf(f, ov.w + c, acc.w);
    }
    *reinterpret_cast<float4*>(dst + 2 * kMaxRows + rho * D + d) = acc;
  }
}

// ------------------------------------------------------------------------------
// Quantized split
// ------------------------------------------------------------------------------
// exponent of |x| as an integer (x finite, nonzero): floor(log2 |x|)
__device__ __forceinline__ int exp2_floor(float x) {
  return static_cast<int>((__float_as_uint(x) >> 23) & 0xFFu) - 127;
}
__device__ __forceinline__ float pow2i(int e) {   // 2^e, -126 <= e <= 127
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// A CTA's role: unit u and quantized split r, or tail slice r.  With clusters,
// CTA r of unit u's cluster is split r (r < S_q) or tail slice r - S_q;
// otherwise the B*Hkv*S_q quantized splits come first and the B*Hkv*S_t tail
// CTAs after them: when the grid is larger than one wave, the short tail CTAs
// take the slots of the first quantized CTAs to finish.  The block index is
// read through a volatile move so that each call derives the role anew.
struct CtaRole {
  long long u;
  int r;
  bool tail;
};

__device__ __forceinline__ CtaRole cta_role(const AttendParams& p, long long nunits) {
  unsigned bx;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(bx));
  const unsigned nquant = static_cast<unsigned>(nunits * p.S_q);
  CtaRole c;
  c.tail = !p.cluster && bx >= nquant;
  const unsigned S = p.cluster ? static_cast<unsigned>(p.S_q + p.S_t) : static_cast<unsigned>(c.tail ? p.S_t : p.S_q);
  const unsigned rel = c.tail ? bx - nquant : bx;
  const unsigned uu = rel / S;
  c.u = static_cast<long long>(uu);
  c.r = static_cast<int>(rel - uu * S);
  if (p.cluster && c.r >= p.S_q) {
    c.tail = true;
    c.r -= p.S_q;
  }
  return c;
}

// Four CTAs per SM when one weight n-tile serves all rows (rows <= 4); two for
// the eight-row variant, which keeps two n-tiles of weights and two sets of P
// fragments.
template <int MODE, int D, int NJ, int NT, bool SC>
__global__ void __launch_bounds__(NTHREADS, (target_ctas<MODE, D, NJ, NT, SC>())) attend_kernel(AttendParams p) {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  using L = Smem<MODE, D, NJ, NT, SC>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = lane >> 2, q = lane & 3;
  const long long nunits = static_cast<long long>(p.c.B) * p.c.Hkv;
  int* sh_flag = reinterpret_cast<int*>(smem + L::MISC_OFF);
  int* sh_abort = sh_flag + 1;
  // Programmatic dependent launch: nothing in global memory is touched before
  // the grids this launch depends on have completed and their writes are
  // visible; every CTA then lets the next dependent launch begin its own
  // start-up (it waits here in turn), which hides the launch gap between
  // back-to-back calls.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  constexpr int G = D / NJ;
  // In either case the partial is staged in the q~ area, which is free once
  // the loop is done and which tail CTAs never use.
  float* part_local = reinterpret_cast<float*>(smem + L::QT_OFF);
  const CtaRole role = cta_role(p, nunits);
  if (role.tail) {  // ---------------- tail CTAs ----
    const long long u = role.u;
    const int ts = role.r;
    const int ntl = seq_r(p.c, static_cast<int>(u / p.c.Hkv)) + p.P + p.top_k, per = (ntl + p.S_t - 1) / p.S_t;
    const int t_lo = min(ntl, ts * per), t_hi = min(ntl, t_lo + per);
    float* wm = reinterpret_cast<float*>(smem + L::WM_OFF);
    float* wl = reinterpret_cast<float*>(smem + L::WL_OFF);
    float* wc = reinterpret_cast<float*>(smem + L::WC_OFF);
    float* wo = reinterpret_cast<float*>(smem + L::WO_OFF);
    tail_entries<D>(p, u, t_lo, t_hi, wm, wl, wc, wo, 0);
    __syncthreads();
    merge_to_partial<D>(p, partial_dst<D>(p, u, p.S_q + ts, part_local), NW, G, wm, wl, wc, wo,
                        reinterpret_cast<float*>(smem + L::FAC_OFF));
    __syncthreads();
    finish_unit<D, NT == 2>(p, u, sh_flag, reinterpret_cast<float*>(smem), part_local);
    return;
  }

  const long long u = role.u;
  const int split = role.r;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  // a ragged cache splits each sequence's own length over the S_q splits (the
  // length is broadcast from lane 0 so that the copy operands below are
  // warp-uniform values for the compiler)
  const long long lq_b = __shfl_sync(0xffffffffu, seq_lq(p.c, b), 0);
  const int wu = __shfl_sync(0xffffffffu, warp, 0);
  const long long chunk =
      p.c.ragged ? (((lq_b + p.S_q - 1) / p.S_q + kChunkAlign - 1) / kChunkAlign) * kChunkAlign : p.chunk;
  const long long t_begin = static_cast<long long>(split) * chunk;
  const long long t_end = min(lq_b, t_begin + chunk);
  const int ntok_chunk = static_cast<int>(max(0LL, t_end - t_begin));
  const int ntiles = (ntok_chunk + M::TT - 1) / M::TT;
  const int per_warp = (ntiles + NW - 1) / NW;
  constexpr int NPK = D / 8;          // key pairs per lane chunk
  constexpr int KSTEPS = D / 16;
  // INT4 reads the upper nibble: step 16 scale; the centred 1-bit reading halves the scale
  const float MULT = (MODE == KVQ_MODE_INT1) ? p.smul : static_cast<float>(M::MULT);
  const int R = p.R;

  float* qt = reinterpret_cast<float*>(smem + L::QT_OFF);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L::BM_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  constexpr int SPW = L::SPW;
  // this warp's tiles: a contiguous run of the chunk
  const int my_first = wu * per_warp;
  const int my_tiles = max(0, min(per_warp, ntiles - my_first));
  const long long u_tok = u * p.c.C;  // first token row of this unit in the planes

  // Each warp streams its own tiles: one elected lane puts tile j into slot
  // j % SPW of the warp's ring with 1-D bulk copies that complete on the slot's
  // mbarrier.  Every copy operand is computed by the whole (converged) warp from
  // warp-uniform values only: the unit and split of the CTA, kernel parameters,
  // the warp index and the tile counter.  Chunk starts are multiples of
  // kChunkAlign, so of G.
  const int rel0 = my_first * M::TT;                       // first token of the run, chunk-relative
  const long long tok_first = u_tok + t_begin + rel0;      // its token row in the planes
  const uint64_t pol = __shfl_sync(0xffffffffu, policy_evict_first(), 0);
  // A tile loads key scales only when it starts a key group (or is the run's
  // first tile): the group's weights are derived from that tile's copy.
  auto issue = [&](int j) {
    const int slot = wu * SPW + (j % SPW);
    const int rel = rel0 + j * M::TT;                        // chunk-relative first token
    const int nt = min(M::TT, ntok_chunk - rel);
    const bool new_grp = (j == 0) || (M::TT > G) || (rel % G == 0);
    const uint32_t kb = nt * RW::KROW, vb = (nt / 32) * D * RW::VROW;
    const uint32_t kszb = new_grp ? static_cast<uint32_t>((nt + G - 1) / G) * 2 * D * 4 : 0u;
    const uint32_t vszb = nt * 2 * NJ * 4;
    const long long tok = tok_first + static_cast<long long>(j) * M::TT;
    uint8_t* sbase = smem + slot * L::SLOT;
    if (elect_one()) {
      // order this warp's earlier reads of the slot before the async-proxy writes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(full + slot, M::NP * (kb + vb) + kszb + vszb);
#pragma unroll
      for (int pl = 0; pl < M::NP; ++pl) {
        bulk_g2s(sbase + L::K_OFF + pl * L::KPLANE, p.c.kplane[pl] + tok * RW::KROW, kb, full + slot, pol);
        bulk_g2s(sbase + L::V_OFF + pl * L::VPLANE, p.c.vplane[pl] + (tok / 32) * D * RW::VROW, vb, full + slot,
                 pol);
      }
      if (new_grp)
        bulk_g2s(sbase + L::KSZ_OFF, p.c.ksz + (u * (p.c.C / G) + (t_begin + rel) / G) * 2 * D, kszb, full + slot,
                 pol);
      bulk_g2s(sbase + L::VSZ_OFF, p.c.vsz + tok * 2 * NJ, vszb, full + slot, pol);
    }
    __syncwarp();
  };

  // ---- setup: each warp's barriers first, so its first tiles load at once ----
  const uint4 q_slice = load_q<D>(p, b, kvh, tid);
  static_assert(kMaxRows * (D / 8) <= NTHREADS, "one query slice per thread");
  if (lane == 0) {
    for (int s2 = 0; s2 < SPW; ++s2) mbar_init(full + wu * SPW + s2, 1);
    fence_mbar_init();
  }
  __syncwarp();
  for (int j = 0; j < min(SPW, my_tiles); ++j) issue(j);
  int issued = min(SPW, my_tiles), consumed = 0;
  if (p.S_t == 0) {
    // This CTA's share of the bf16 tail comes after its quantized tokens; its
    // residual and pending rows are pulled into L2 now, so that the share's
    // loads at the end of the CTA hit L2.  (Selected rows need their index
    // first and are left alone.)
    constexpr int LPR = D / 64;                              // 128-byte lines per bf16 row
    const int r_b = seq_r(p.c, b);
    const int ntl = r_b + p.P + p.top_k, per = (ntl + p.S_q - 1) / p.S_q;
    const int t_lo = min(ntl, split * per), t_hi = min(ntl, t_lo + per);
    const int t_pf = min(t_hi, r_b + p.P);
    for (int i = tid; i < (t_pf - t_lo) * 2 * LPR; i += NTHREADS) {
      const uint16_t *kp = nullptr, *vp = nullptr;
      tail_row<D>(p, u, t_lo + i / (2 * LPR), kp, vp);
      const int j = i % (2 * LPR);
      prefetch_l2((j < LPR ? kp : vp) + (j % LPR) * 64);
    }
  }
  const int bm_words = (ntok_chunk + 31) / 32;
  if (tid == 0) *sh_abort = 0;
  const bool has_sel = p.top_k > 0;
  if (has_sel)
    for (int e = tid; e < bm_words; e += blockDim.x) bitmap[e] = 0u;
  if constexpr (NT == 1) {
    // the staged weight columns of rows that are not in use stay zero
    uint4* wz = reinterpret_cast<uint4*>(smem + L::WB_OFF);
    for (int e = tid; e < L::WB_BYTES / 16; e += NTHREADS) wz[e] = make_uint4(0u, 0u, 0u, 0u);
  }
  // scaled queries, and per warp the max |q~| (for the weight normalizer)
  {
    float qm = store_qt<D>(p, tid, q_slice, qt);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, o2));
    if (lane == 0) reinterpret_cast<float*>(smem + L::QM_OFF)[warp] = qm;
  }
  if constexpr (SC) {
    // the score row's query heads that share this KV head, summed in fp32 in
    // ascending head order (the top-k score's summed query)
    static_assert(D <= NTHREADS, "one channel per thread");
    if (tid < D) {
      const long long base = ((static_cast<long long>(b) * p.gamma + p.score_row) * p.Hq + kvh * p.HG) * D + tid;
      float acc = 0.f;
      for (int hh = 0; hh < p.HG; ++hh) acc = __fadd_rn(acc, bf16_to_f32(p.q[base + hh * D]));
      reinterpret_cast<float*>(smem + L::SQ_OFF)[tid] = acc;
    }
  }
  if (has_sel) {
    __syncthreads();   // the bitmap is clear before any bit is set (has_sel is uniform)
    for (int j = tid; j < p.top_k; j += blockDim.x) {
      const long long idx = p.sel_idx[u * p.top_k + j];
      if (idx >= t_begin && idx < t_end) {
        const int rel = static_cast<int>(idx - t_begin);
        atomicOr(bitmap + rel / 32, 1u << (rel % 32));
      }
    }
  }
  __syncthreads();

  {
    // ---------------- consumers ----------------
    // Keys are the A operand (rows = 16 tokens of an m-tile, k = channels), the
    // folded query weights the B operand (column 2r + h = row 4nt + r, h = high
    // / low f16 part).  Values are the A operand of O^T = V^T P^T (rows =
    // channels, k = tokens).  In m-tile s the lane's rows g and g+8 are the
    // tokens of value pair 2s + (g & 1) of token octet g >> 1, so the P values a
    // lane computes are a whole B register of P.V for one destination lane.
    const int oct = 8 * (g >> 1), par = g & 1;
    int tokA[2], tokB[2];
    float vinv[2];          // 1 / value factor of the lane's pair, per m-tile
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int i = 2 * s + par;
      tokA[s] = oct + xpair_a<MODE>(i);
      tokB[s] = oct + xpair_b<MODE>(i);
      vinv[s] = 1.0f / static_cast<float>(1 << vs_log2fac<MODE>(i));
    }

    uint32_t W[NT][NPK];                 // weights: this lane's B column part, per key pair
    float sc_unit = 0.f;                 // scoring: 2^(e-21) of the current group
    float sc_beta = 0.f;                 // scoring: the group's zero-point term
    float cinit[NT];                     // accumulator start (correction x 2^e) for row 4nt + q
    float kscale = 1.f;                  // 2^-e of the current group
    float o[D / 16][4];                  // O^T, channel m-tile x (col 2q, 2q+1)
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[NT], l_run[NT], vcorr[NT][NJ];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt] = neg_inf();
      l_run[nt] = 0.f;
#pragma unroll
      for (int jv = 0; jv < NJ; ++jv) vcorr[nt][jv] = 0.f;
      cinit[nt] = 0.f;
#pragma unroll
      for (int pp = 0; pp < NPK; ++pp) W[nt][pp] = 0u;
    }
    float evs = 0.f;                     // value normalizer 2^ev (0: not chosen yet)
    int cur_grp = -1;


    for (int j = 0; j < my_tiles; ++j) {
      const int ti = my_first + j;
      const int slot = wu * SPW + (j % SPW);
      const uint32_t parity = (j / SPW) & 1;
      if (!mbar_wait_bounded(full + slot, parity, p.wait_limit)) {
        record_status(p.status, KVQ_ERR_DEVICE_TIMEOUT);
        *reinterpret_cast<volatile int*>(sh_abort) = 1;
        break;
      }
      if (*reinterpret_cast<volatile int*>(sh_abort)) break;
      const int rel = ti * M::TT;                            // chunk-relative first token
      const int nt_tok = min(M::TT, ntok_chunk - rel);
      const int g_first = rel / G;
      const uint8_t* sbase = smem + slot * L::SLOT;
      const float* ksz = reinterpret_cast<const float*>(sbase + L::KSZ_OFF);
      const float* vsz = reinterpret_cast<const float*>(sbase + L::VSZ_OFF);

      for (int sl = 0; sl < nt_tok / 32; ++sl) {
        const int tok0 = rel + 32 * sl;
        const int grp = tok0 / G;
        if (grp != cur_grp) {
          // ---- folded key weights of this group, derived once per warp ----
          // w_c = q~_c * MULT * s_c / f_c (f_c the channel's code factor),
          // scaled by 2^e so that the largest possible |w| sits near 2^13,
          // split into f16 high + low parts.  With one n-tile the lanes split
          // the channels, stage the B fragments of the rows in use in the
          // warp's weight buffer, then each lane loads its column; with two the
          // lanes derive their own columns.  The accumulator starts at
          // 2^(e-24) sum_c q~_c z_c, and the logit is the accumulator times
          // 2^(24-e).
          cur_grp = grp;
          const float* ks = ksz + (grp - g_first) * 2 * D;
          const float* kz = ks + D;
          // rows in use rounded up to a power of two
          const int rpow = R <= 1 ? 1 : (R <= 2 ? 2 : (R <= 4 ? 4 : 8));
          uint32_t* wb = reinterpret_cast<uint32_t*>(smem + L::WB_OFF) + warp * (4 * D);
          (void)wb;
          const float* qmw = reinterpret_cast<const float*>(smem + L::QM_OFF);
          float qmax = qmw[0];
#pragma unroll
          for (int w2 = 1; w2 < NW; ++w2) qmax = fmaxf(qmax, qmw[w2]);
          const float KW = MULT;
          const float zsh = p.zshift;   // zero points read as z + zsh * s (the INT4 midpoint reading)
          float zsum = 0.f;
          float kscale_new, Z2;
          if constexpr (NT == 2) {
            // eight rows: lanes g = 2r and 2r + 1 hold the high and the low
            // part of row 4nt + r (column g).  Each derives both parts for half
            // of its chunk's channel pairs, and the two swap the part the other
            // one keeps.
            constexpr int HP = D / 16;                        // pairs per half chunk
            constexpr int DELTA = kx_chan<MODE, D>(HP, 0);    // channel offset of the second half
            static_assert(halves_shift<MODE, D>(), "the second half's pairs are the first half's, shifted");
            static_assert(halves_same_factors<MODE, D>(), "both halves carry the same code factors");
            const int cb = q * (D / 4) + par * DELTA;         // this lane's channel base
            static_assert(DELTA % 4 == 0, "the halves' windows start on float4 boundaries");
            constexpr int WIN = half_window<MODE, D>();
            const float* ksc = ks + cb;
            const float* kzc = kz + cb;
            float ksw[WIN];
#pragma unroll
            for (int v4 = 0; v4 < WIN / 4; ++v4) {
              const float4 x = reinterpret_cast<const float4*>(ksc)[v4];
              ksw[4 * v4] = x.x; ksw[4 * v4 + 1] = x.y; ksw[4 * v4 + 2] = x.z; ksw[4 * v4 + 3] = x.w;
            }
            float kv[HP][2];
            float smax = 0.f;
#pragma unroll
            for (int k = 0; k < HP; ++k) {
              kv[k][0] = ksw[kx_chan<MODE, D>(k, 0)];
              kv[k][1] = ksw[kx_chan<MODE, D>(k, 1)];
              smax = fmaxf(smax, fmaxf(kv[k][0], kv[k][1]));
            }
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 4));
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 1));
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 2));
            const float bound = qmax * smax * KW;
            const int e = (bound > 0.f) ? max(-100, min(100, 13 - exp2_floor(bound))) : 0;
            Z2 = pow2i(e - 24);
            kscale_new = pow2i(24 - e);
            const float f = pow2i(e) * KW;
#pragma unroll
            for (int k = 0; k < HP; ++k) {
              kv[k][0] *= f * ks_inv_fac<MODE, D>(k);
              kv[k][1] *= f * ks_inv_fac<MODE, D>(k);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float* qr = qt + (4 * nt + (g >> 1)) * qt_row<D>() + q * qt_chunk<D>() + par * DELTA;
              float zs = 0.f;
              uint32_t keep[HP], send[HP];
              float kzw[WIN];
#pragma unroll
              for (int v4 = 0; v4 < WIN / 4; ++v4) {
                const float4 x = reinterpret_cast<const float4*>(kzc)[v4];
                kzw[4 * v4] = x.x; kzw[4 * v4 + 1] = x.y; kzw[4 * v4 + 2] = x.z; kzw[4 * v4 + 3] = x.w;
              }
#pragma unroll
              for (int k = 0; k < HP; ++k) {
                const int c0 = kx_chan<MODE, D>(k, 0), c1 = kx_chan<MODE, D>(k, 1);
                const float q0 = qr[c0], q1 = qr[c1];
                float z0 = kzw[c0], z1 = kzw[c1];
                if (zsh != 0.f) {
                  z0 = fmaf(zsh, ksw[c0], z0);
                  z1 = fmaf(zsh, ksw[c1], z1);
                }
                zs = fmaf(q0, z0, fmaf(q1, z1, zs));
                const float w0 = q0 * kv[k][0], w1 = q1 * kv[k][1];
                const uint32_t hi = pack_half2(w0, w1);
                const float2 hf = unpack_half2(hi);
                const uint32_t lo = pack_half2(w0 - hf.x, w1 - hf.y);
                keep[k] = par ? lo : hi;
                send[k] = par ? hi : lo;
              }
#pragma unroll
              for (int k = 0; k < HP; ++k) {
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send[k], 4);
                W[nt][k] = par ? recv : keep[k];
                W[nt][HP + k] = par ? keep[k] : recv;
              }
              float cwn = zs * Z2;
              cwn += __shfl_xor_sync(0xffffffffu, cwn, 4);
              cwn += __shfl_xor_sync(0xffffffffu, cwn, 1);
              cwn += __shfl_xor_sync(0xffffffffu, cwn, 2);
              // this lane's C rows belong to row 4nt + q, whose weights lanes g = 2q hold
              cinit[nt] = __shfl_sync(0xffffffffu, cwn, 8 * q);
            }
          } else {
            // Lane l takes channels CPL l .. CPL l + CPL - 1 (CPL = D / 32) of
            // every row in use: their scales and zero points are read once, and
            // each row's high and low weight parts go to those channels' halves
            // of the staged B fragments (column 2 rho + part, chunk qq, half
            // kx_slot of the channel).
            constexpr int CPL = D / 32;
            static_assert(CPL == 4 || CPL == 2, "four or two channels per lane");
            const int c_lo = CPL * lane, qq = c_lo / (D / 4), cl0 = c_lo % (D / 4);
            float ksv[CPL], kzv[CPL];
            if constexpr (CPL == 4) {
              const float4 a = *reinterpret_cast<const float4*>(ks + c_lo);
              const float4 z = *reinterpret_cast<const float4*>(kz + c_lo);
              ksv[0] = a.x; ksv[1] = a.y; ksv[2] = a.z; ksv[3] = a.w;
              kzv[0] = z.x; kzv[1] = z.y; kzv[2] = z.z; kzv[3] = z.w;
            } else {
              const float2 a = *reinterpret_cast<const float2*>(ks + c_lo);
              const float2 z = *reinterpret_cast<const float2*>(kz + c_lo);
              ksv[0] = a.x; ksv[1] = a.y;
              kzv[0] = z.x; kzv[1] = z.y;
            }
            float smax = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) smax = fmaxf(smax, ksv[i]);
            smax = warp_max_nonneg(smax);        // scales are >= 0
            const float bound = qmax * smax * KW;
            const int e = (bound > 0.f) ? max(-100, min(100, 13 - exp2_floor(bound))) : 0;
            Z2 = pow2i(e - 24);
            kscale_new = pow2i(24 - e);
            const float f = pow2i(e) * KW;
            uint16_t* wbh = reinterpret_cast<uint16_t*>(wb);
#pragma unroll
            for (int i = 0; i < CPL; ++i) kzv[i] = fmaf(zsh, ksv[i], kzv[i]);   // zero points as the mode reads them
            for (int rho = 0; rho < rpow; ++rho) {
              const float* qr = qt + rho * qt_row<D>() + qq * qt_chunk<D>() + cl0;
              float zs = 0.f;
#pragma unroll
              for (int i = 0; i < CPL; ++i) {
                const int slot = kx_slot<MODE, D>(cl0 + i);
                const float qv = qr[i];
                const float w = qv * ksv[i] * (f * pow2i(-ks_log2fac<MODE, D>(slot >> 1)));
                const __half hi = __float2half_rn(w);
                const __half lo = __float2half_rn(w - __half2float(hi));
                wbh[(2 * rho) * D + qq * (D / 4) + slot] = __half_as_ushort(hi);
                wbh[(2 * rho + 1) * D + qq * (D / 4) + slot] = __half_as_ushort(lo);
                zs = fmaf(qv, kzv[i], zs);
              }
#pragma unroll
              for (int o2 = 16; o2 > 0; o2 >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o2);
              if (rho == q) zsum = zs;       // the rows of this lane's accumulator (row q)
            }
          }
          kscale = kscale_new;
          if constexpr (NT == 1) {
            __syncwarp();
            // columns of rows past rpow were zeroed at the start and are never written
            const uint4* src = reinterpret_cast<const uint4*>(wb + (g * 4 + q) * (D / 8));
#pragma unroll
            for (int v = 0; v < D / 32; ++v) {
              const uint4 x4 = src[v];
              W[0][4 * v] = x4.x; W[0][4 * v + 1] = x4.y; W[0][4 * v + 2] = x4.z; W[0][4 * v + 3] = x4.w;
            }
            cinit[0] = zsum * Z2;                // zero for rows q >= rpow
            __syncwarp();
          }
          if constexpr (SC) {
            // ---- integer score weights and zero-point term of this group (the top-k score) ----
            // w_d = fp32(qs_d * fp32(MULT s_d)); e with max|w| < 2^e (floored at
            // -100); W_d = rint(w_d 2^(21-e)) = 2^14 h + 2^7 m + l with
            // |h| <= 128 and |m|, |l| <= 64 (h = rint(W 2^-14), m = rint(r 2^-7)
            // with r = W - 2^14 h, l = r - 2^7 m: all exact fp32 steps, the
            // roundings by adding and subtracting 1.5 * 2^23).  The parts times 2^(SLF - f_p)
            // (f_p the pair's code factor) are exact f16 values, so the MMA
            // over the subnormal codes sums c * part * 2^(SLF-24) exactly.
            // Lane l derives key pairs l and l + 32 (quarter (l + 32 i) / (D/8),
            // pair (l + 32 i) mod (D/8)), both channels of each, and writes each
            // part as a half2 in the pairs' order.
            constexpr int NIT = D / 64;                 // pairs per lane
            constexpr int SLF = score_log2fac_max<MODE, D>();
            const float* qsum = reinterpret_cast<const float*>(smem + L::SQ_OFF);
            uint32_t* whs = reinterpret_cast<uint32_t*>(smem + L::SW_OFF) + warp * 3 * (D / 2);
            const int pp = lane % (D / 8);
            const int c0 = kx_chan<MODE, D>(pp, 0), c1 = kx_chan<MODE, D>(pp, 1);
            const int sh = SLF - ks_log2fac<MODE, D>(pp);
            float wv[2 * NIT], zp[2 * NIT];
            float mxw = 0.f;
#pragma unroll
            for (int i = 0; i < NIT; ++i) {
              const int base = ((lane + 32 * i) / (D / 8)) * (D / 4);
              const int d0 = base + c0, d1 = base + c1;
              wv[2 * i] = __fmul_rn(qsum[d0], __fmul_rn(ks[d0], MULT));
              wv[2 * i + 1] = __fmul_rn(qsum[d1], __fmul_rn(ks[d1], MULT));
              zp[2 * i] = __fmul_rn(qsum[d0], fmaf(zsh, ks[d0], kz[d0]));   // zero points as the mode reads them
              zp[2 * i + 1] = __fmul_rn(qsum[d1], fmaf(zsh, ks[d1], kz[d1]));
              mxw = fmaxf(mxw, fmaxf(fabsf(wv[2 * i]), fabsf(wv[2 * i + 1])));
            }
            mxw = warp_max_nonneg(mxw);
            // beta: the products rounded to integers at the largest one's unit, summed exactly
            sc_beta = zero_term_warp<2 * NIT>(zp);
            int es = 0;
            if (mxw > 0.f) frexpf(mxw, &es);
            es = max(es, -100);
            const float up = pow2i(21 - es);
            sc_unit = pow2i(es - 21);
            constexpr float kRnd = 12582912.0f;        // 1.5 * 2^23: x + kRnd - kRnd = rint(x) for |x| < 2^22
            const float fsh = pow2i(sh);
#pragma unroll
            for (int i = 0; i < NIT; ++i) {
              float v[2][3];
#pragma unroll
              for (int e2 = 0; e2 < 2; ++e2) {
                const float W = __fsub_rn(__fadd_rn(__fmul_rn(wv[2 * i + e2], up), kRnd), kRnd);   // |W| <= 2^21
                const float h = __fsub_rn(__fadd_rn(__fmul_rn(W, 1.0f / 16384.f), kRnd), kRnd);
                const float r = __fmaf_rn(h, -16384.f, W);
                const float m = __fsub_rn(__fadd_rn(__fmul_rn(r, 1.0f / 128.f), kRnd), kRnd);
                const float l = __fmaf_rn(m, -128.f, r);
                v[e2][0] = __fmul_rn(h, fsh);
                v[e2][1] = __fmul_rn(m, fsh);
                v[e2][2] = __fmul_rn(l, fsh);
              }
              uint32_t part[3];
#pragma unroll
              for (int k3 = 0; k3 < 3; ++k3) part[k3] = pack_half2(v[0][k3], v[1][k3]);   // exact f16 values
              const int word = lane + 32 * i;          // quarter * (D/8) + pair
#pragma unroll
              for (int k3 = 0; k3 < 3; ++k3) whs[k3 * (D / 2) + word] = part[k3];
            }
            __syncwarp();
          }
        }
        const uint8_t* kslab = sbase + L::K_OFF + (32 * sl) * RW::KROW + q * RW::KCHUNK;
        const uint8_t* vslab = sbase + L::V_OFF + sl * D * RW::VROW;

        // ---- logits: S = K W, two m-tiles of 16 tokens ----
        float x[2][NT][2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          uint32_t PA[NPK], PB[NPK];
          key_pairs_s<MODE, D>(kslab + tokA[s] * RW::KROW, L::KPLANE, PA);
          key_pairs_s<MODE, D>(kslab + tokB[s] * RW::KROW, L::KPLANE, PB);
          float acc[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = cinit[nt]; acc[nt][1] = 0.f; acc[nt][2] = cinit[nt]; acc[nt][3] = 0.f;
          }
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            const uint32_t a[4] = {PA[2 * kk], PB[2 * kk], PA[2 * kk + 1], PB[2 * kk + 1]};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt], a, W[nt][2 * kk], W[nt][2 * kk + 1]);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            x[s][nt][0] = (acc[nt][0] + acc[nt][1]) * kscale;
            x[s][nt][1] = (acc[nt][2] + acc[nt][3]) * kscale;
          }
          if constexpr (SC) {
            // ---- the top-k score of the m-tile's tokens, from the same key fragments ----
            // columns 0, 1 (lanes q = 0) hold the h and m parts, column 2 (lanes
            // q = 1) the l part; S_t = 2^14 S_h + 2^7 S_m + S_l exactly in 64 bits
            // lane (g, q) reads column g of the weight parts (zero past column 2)
            // from the warp's staging area at each k-step: no registers held
            // across the slab
            float cs[4] = {0.f, 0.f, 0.f, 0.f};
            const uint2* wsrc = reinterpret_cast<const uint2*>(
                reinterpret_cast<const uint32_t*>(smem + L::SW_OFF) + warp * 3 * (D / 2) + min(g, 2) * (D / 2) + q * (D / 8));
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
              const uint32_t a[4] = {PA[2 * kk], PB[2 * kk], PA[2 * kk + 1], PB[2 * kk + 1]};
              const uint2 w2 = wsrc[kk];
              mma16816(cs, a, g < 3 ? w2.x : 0u, g < 3 ? w2.y : 0u);
            }
            const float lA = __shfl_down_sync(0xffffffffu, cs[0], 1);
            const float lB = __shfl_down_sync(0xffffffffu, cs[2], 1);
            if (q == 0) {
              // The part sums are exact: S_x = cs_x * 2^(24 - SLF).  2^14 S_h is an
              // exact fp32 value and so is 2^7 S_m + S_l (below 2^24), so one
              // correctly rounded add gives fp32(S_t).
              constexpr float INV = static_cast<float>(1 << (24 - score_log2fac_max<MODE, D>()));
              const float SA = __fadd_rn(__fmul_rn(cs[0], INV * 16384.f), __fmaf_rn(cs[1], INV * 128.f, __fmul_rn(lA, INV)));
              const float SB = __fadd_rn(__fmul_rn(cs[2], INV * 16384.f), __fmaf_rn(cs[3], INV * 128.f, __fmul_rn(lB, INV)));
              float* dst = p.pre + u * p.c.C + t_begin + tok0;
              dst[tokA[s]] = __fadd_rn(__fmul_rn(SA, sc_unit), sc_beta);
              dst[tokB[s]] = __fadd_rn(__fmul_rn(SB, sc_unit), sc_beta);
            }
          }
        }
        if (has_sel) {
          const uint32_t bm = bitmap[tok0 / 32];
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const bool ma = (bm >> tokA[s]) & 1u, mb = (bm >> tokB[s]) & 1u;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (ma) x[s][nt][0] = neg_inf();
              if (mb) x[s][nt][1] = neg_inf();
            }
          }
        }
        // ---- online softmax ----
        float m_new[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float mx = fmaxf(fmaxf(x[0][nt][0], x[0][nt][1]), fmaxf(x[1][nt][0], x[1][nt][1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          m_new[nt] = fmaxf(m_run[nt], mx);
        }
        float alpha[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          alpha[nt] = (m_run[nt] == m_new[nt]) ? 1.f
                      : (m_run[nt] == neg_inf()) ? 0.f : fast_exp2(m_run[nt] - m_new[nt]);
          m_run[nt] = m_new[nt];
          l_run[nt] *= alpha[nt];
#pragma unroll
          for (int jv = 0; jv < NJ; ++jv) vcorr[nt][jv] *= alpha[nt];
        }
        // rows of this lane's O^T columns: their rescale factors
        float a_lo, a_hi;
        if constexpr (NT == 1) {
          a_lo = a_hi = alpha[0];
        } else {
          const int src_lo = 4 * g + ((2 * q) & 3), src_hi = 4 * g + ((2 * q + 1) & 3);
          const float l0 = __shfl_sync(0xffffffffu, alpha[0], src_lo), l1 = __shfl_sync(0xffffffffu, alpha[1], src_lo);
          const float h0 = __shfl_sync(0xffffffffu, alpha[0], src_hi), h1 = __shfl_sync(0xffffffffu, alpha[1], src_hi);
          a_lo = (q >> 1) ? l1 : l0;
          a_hi = (q >> 1) ? h1 : h0;
        }
        // value scales of the lane's tokens; the value normalizer keeps P' below 2^15
        float sA[2][NJ], zA[2][NJ], sB[2][NJ], zB[2][NJ];
        float smx = 0.f;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          float va[2 * NJ], vb[2 * NJ];
          load_vrow<NJ>(vsz + (32 * sl + tokA[s]) * 2 * NJ, va);
          load_vrow<NJ>(vsz + (32 * sl + tokB[s]) * 2 * NJ, vb);
#pragma unroll
          for (int jv = 0; jv < NJ; ++jv) {
            sA[s][jv] = va[jv] * MULT; zA[s][jv] = fmaf(p.zshift, va[jv], va[NJ + jv]);
            sB[s][jv] = vb[jv] * MULT; zB[s][jv] = fmaf(p.zshift, vb[jv], vb[NJ + jv]);
            smx = fmaxf(smx, fmaxf(sA[s][jv], sB[s][jv]));
          }
        }
        if (__any_sync(0xffffffffu, smx * evs >= 32768.f || evs == 0.f)) {
          float wmx = smx;
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) wmx = fmaxf(wmx, __shfl_xor_sync(0xffffffffu, wmx, o2));
          const float nev = (wmx > 0.f) ? pow2i(max(-100, min(100, 13 - exp2_floor(wmx)))) : 1.f;
          const float fac = (evs == 0.f) ? 0.f : nev / evs;
          evs = nev;
          a_lo *= fac;
          a_hi *= fac;
        }
        float pr[2][NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float msafe = (m_run[nt] == neg_inf()) ? 0.f : m_run[nt];
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            pr[s][nt][0] = fast_exp2(x[s][nt][0] - msafe);
            pr[s][nt][1] = fast_exp2(x[s][nt][1] - msafe);
            l_run[nt] += pr[s][nt][0] + pr[s][nt][1];
          }
        }

        // ---- P.V, one channel block (G channels) at a time ----
#pragma unroll
        for (int jv = 0; jv < NJ; ++jv) {
          // P' = p * s * MULT * 2^ev / m (m the value pair's factor) as f16
          // high + low parts, per m-tile
          uint32_t H[2][NT], Lo[2][NT];
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const float fa = sA[s][jv] * (evs * vinv[s]), fb = sB[s][jv] * (evs * vinv[s]);
            const float za = zA[s][jv], zb = zB[s][jv];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float pa = pr[s][nt][0] * fa, pb = pr[s][nt][1] * fb;
              H[s][nt] = pack_half2(pa, pb);
              const float2 hf = unpack_half2(H[s][nt]);
              Lo[s][nt] = pack_half2(pa - hf.x, pb - hf.y);
              vcorr[nt][jv] = fmaf(pr[s][nt][0], za, fmaf(pr[s][nt][1], zb, vcorr[nt][jv]));
            }
          }
          // B fragments of P^T for k-step s: b0 from lane (g = 2q), b1 from lane (g = 2q + 1)
          uint32_t bh[2][2], bl[2][2];
          if constexpr (NT == 1) {
            // column g = 2 * row + part
            const int r = g >> 1;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const int src = 8 * q + 4 * k2 + r;
                const uint32_t vh = __shfl_sync(0xffffffffu, H[s][0], src);
                const uint32_t vl = __shfl_sync(0xffffffffu, Lo[s][0], src);
                bh[s][k2] = par ? vl : vh;
              }
            }
          } else {
            // column g = row; high and low parts go through separate MMAs
            const int r = g & 3;
            const bool hi_nt = g >= 4;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const int src = 8 * q + 4 * k2 + r;
                const uint32_t h0 = __shfl_sync(0xffffffffu, H[s][0], src);
                const uint32_t h1 = __shfl_sync(0xffffffffu, H[s][NT - 1], src);
                const uint32_t l0 = __shfl_sync(0xffffffffu, Lo[s][0], src);
                const uint32_t l1 = __shfl_sync(0xffffffffu, Lo[s][NT - 1], src);
                bh[s][k2] = hi_nt ? h1 : h0;
                bl[s][k2] = hi_nt ? l1 : l0;
              }
            }
          }
          // The slab's products go into a fresh accumulator, folded into the
          // running output with one rounding per element: a long MMA chain
          // would accumulate the tensor core's truncation.
#pragma unroll
          for (int mt = jv * (G / 16); mt < (jv + 1) * (G / 16); ++mt) {
            uint32_t a[2][4];
            const uint8_t* va = vslab + (16 * mt + g) * RW::VROW;
            value_frags_s<MODE>(va, va + 8 * RW::VROW, L::VPLANE, q, a);
            float os[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(os, a[0], bh[0][0], bh[0][1]);
            if constexpr (NT == 2) mma16816(os, a[0], bl[0][0], bl[0][1]);
            mma16816(os, a[1], bh[1][0], bh[1][1]);
            if constexpr (NT == 2) mma16816(os, a[1], bl[1][0], bl[1][1]);
            o[mt][0] = fmaf(o[mt][0], a_lo, os[0]);
            o[mt][1] = fmaf(o[mt][1], a_hi, os[1]);
            o[mt][2] = fmaf(o[mt][2], a_lo, os[2]);
            o[mt][3] = fmaf(o[mt][3], a_hi, os[3]);
          }
        }
      }
      __syncwarp();
      consumed = j + 1;
      if (issued < my_tiles) {
        issue(issued);
        ++issued;
      }
    }
    // after an abort: let this warp's copies still in flight land before exit
    if (lane == 0) {
      for (int jj = consumed; jj < issued; ++jj)
        mbar_wait_bounded(full + wu * SPW + (jj % SPW), (jj / SPW) & 1, p.wait_limit);
    }
    __syncwarp();

    // ---- per-warp results to shared scratch (after everyone left the ring) ----
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {
        l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], o2);
#pragma unroll
        for (int jv = 0; jv < NJ; ++jv) vcorr[nt][jv] += __shfl_xor_sync(0xffffffffu, vcorr[nt][jv], o2);
      }
    }
    // the stage rings must be idle before the slot area is reused
    __syncthreads();
    float* wm = reinterpret_cast<float*>(smem + L::WM_OFF);
    float* wl = reinterpret_cast<float*>(smem + L::WL_OFF);
    float* wc = reinterpret_cast<float*>(smem + L::WC_OFF);
    float* wo = reinterpret_cast<float*>(smem + L::WO_OFF);
    if (g == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int rho = 4 * nt + q;
        wm[warp * 8 + rho] = m_run[nt];
        wl[warp * 8 + rho] = l_run[nt];
#pragma unroll
        for (int jv = 0; jv < NJ; ++jv) wc[(warp * 8 + rho) * 4 + jv] = vcorr[nt][jv];
      }
    }
    const float oscale = (evs > 0.f) ? 16777216.0f / evs : 0.f;   // 2^24 / 2^ev
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      const int ca = 16 * mt + g, cb = ca + 8;
      if constexpr (NT == 1) {
        wo[(warp * 8 + q) * D + ca] = (o[mt][0] + o[mt][1]) * oscale;
        wo[(warp * 8 + q) * D + cb] = (o[mt][2] + o[mt][3]) * oscale;
      } else {
        wo[(warp * 8 + 2 * q) * D + ca] = o[mt][0] * oscale;
        wo[(warp * 8 + 2 * q + 1) * D + ca] = o[mt][1] * oscale;
        wo[(warp * 8 + 2 * q) * D + cb] = o[mt][2] * oscale;
        wo[(warp * 8 + 2 * q + 1) * D + cb] = o[mt][3] * oscale;
      }
    }
  }
  __syncthreads();

  // ---- this CTA's share of the bf16 tail (residual, pending, selected tokens) ----
  // Without tail CTAs the quantized splits share the tail list: entries
  // NW .. 2 NW - 1.  (The role is derived again rather than kept in registers
  // through the loop.)
  {
    const CtaRole role2 = cta_role(p, nunits);
    const long long u = role2.u;
    const int split = role2.r;
    const float* wm = reinterpret_cast<const float*>(smem + L::WM_OFF);
    if (p.S_t == 0) {
      const int ntl = seq_r(p.c, static_cast<int>(u / p.c.Hkv)) + p.P + p.top_k, per = (ntl + p.S_q - 1) / p.S_q;
      const int t_lo = min(ntl, split * per), t_hi = min(ntl, t_lo + per);
      tail_entries<D>(p, u, t_lo, t_hi, reinterpret_cast<float*>(smem + L::WM_OFF),
                      reinterpret_cast<float*>(smem + L::WL_OFF), reinterpret_cast<float*>(smem + L::WC_OFF),
                      reinterpret_cast<float*>(smem + L::WO_OFF), NW);
      __syncthreads();
    }
    // ---- CTA merge of the entries -> partial ----
    merge_to_partial<D>(p, partial_dst<D>(p, u, split, part_local), (p.S_t == 0) ? 2 * NW : NW, G, wm,
                        reinterpret_cast<const float*>(smem + L::WL_OFF), reinterpret_cast<const float*>(smem + L::WC_OFF),
                        reinterpret_cast<const float*>(smem + L::WO_OFF), reinterpret_cast<float*>(smem + L::FAC_OFF));
    __syncthreads();
    finish_unit<D, NT == 2>(p, u, sh_flag, reinterpret_cast<float*>(smem), part_local);
  }
}

template <int MODE, int D, int NJ, int NT, bool SC>
constexpr int smem_bytes() {
  using L = Smem<MODE, D, NJ, NT, SC>;
  return L::TOTAL;
}

// Lets the variant launch clusters of more than 8 CTAs (up to 16); once per device.
template <int MODE, int D, int NJ, int NT, bool SC>
cudaError_t allow_wide_clusters() {
  constexpr int kMaxDev = 64;
  static bool done[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&attend_kernel<MODE, D, NJ, NT, SC>),
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDev) done[dev] = true;
  return e;
}

// Launch configuration with one cluster of `size` CTAs per (b, kvh).
inline void cluster_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute& at, long long grid, int smem, int size,
                           cudaStream_t s) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  at = cudaLaunchAttribute{};
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = static_cast<unsigned>(size);
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
}

template <int MODE, int D, int NJ, int NT, bool SC>
cudaError_t launch_t(const AttendParams& p, cudaStream_t s) {
  constexpr int smem = smem_bytes<MODE, D, NJ, NT, SC>();
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&attend_kernel<MODE, D, NJ, NT, SC>), smem);
  if (e != cudaSuccess) return e;
  const long long nunits = static_cast<long long>(p.c.B) * p.c.Hkv;
  const int S_all = p.S_q + p.S_t;
  const long long grid = nunits * S_all;
  if (!p.cluster) {
    // a plain grid may start while the previous kernel in the stream finishes
    // (the kernel waits for it before any global access)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute at = {};
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attend_kernel<MODE, D, NJ, NT, SC>, p);
  }
  if (S_all < 1 || S_all > kMaxClusterCtas) return cudaErrorInvalidValue;
  if (S_all > 8 && (e = allow_wide_clusters<MODE, D, NJ, NT, SC>()) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute at;
  cluster_config(cfg, at, grid, smem, S_all, s);
  return cudaLaunchKernelEx(&cfg, attend_kernel<MODE, D, NJ, NT, SC>, p);
}

// Clusters of `size` CTAs of one kernel variant that fit on the device at
// once, queried once per device and size (0: unknown or not launchable).
template <int MODE, int D, int NJ, int NT, bool SC>
int resident_clusters_t(int size) {
  if (size < 1 || size > kMaxClusterCtas) return 0;
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev][kMaxClusterCtas + 1] = {};   // 0: not queried, -1: none
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int& c = cached[dev][size];
  if (c != 0) return c > 0 ? c : 0;
  constexpr int smem = smem_bytes<MODE, D, NJ, NT, SC>();
  const void* fn = reinterpret_cast<const void*>(&attend_kernel<MODE, D, NJ, NT, SC>);
  if (set_smem_once(fn, smem) != cudaSuccess) return 0;
  if (size > 8 && allow_wide_clusters<MODE, D, NJ, NT, SC>() != cudaSuccess) {
    cudaGetLastError();
    c = -1;
    return 0;
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute at;
  cluster_config(cfg, at, size, smem, size, nullptr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    c = -1;
    return 0;
  }
  c = n;
  return n;
}

// Resident CTAs per SM of one kernel variant times the SM count, queried once
// per device (the split count is sized to fill whole waves).
template <int MODE, int D, int NJ, int NT, bool SC>
int resident_ctas_t() {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  if (cached[dev] > 0) return cached[dev];
  constexpr int smem = smem_bytes<MODE, D, NJ, NT, SC>();
  if (set_smem_once(reinterpret_cast<const void*>(&attend_kernel<MODE, D, NJ, NT, SC>), smem) != cudaSuccess) return 0;
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attend_kernel<MODE, D, NJ, NT, SC>, NTHREADS, smem) !=
      cudaSuccess)
    return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cached[dev] = per_sm * sms;
  return cached[dev];
}

// Dispatch over (D, G): F<D, NJ>::run() with NJ = D / G.
template <int MODE, int NT, bool SC>
struct Variant {
  static int resident(int D, int NJ) {
    if (D == 128) {
      if (NJ == 1) return resident_ctas_t<MODE, 128, 1, NT, SC>();
      if (NJ == 2) return resident_ctas_t<MODE, 128, 2, NT, SC>();
      if (NJ == 4) return resident_ctas_t<MODE, 128, 4, NT, SC>();
    } else if (D == 64) {
      if (NJ == 1) return resident_ctas_t<MODE, 64, 1, NT, SC>();
      if (NJ == 2) return resident_ctas_t<MODE, 64, 2, NT, SC>();
    }
    return 0;
  }
  static int clusters(int D, int NJ, int size) {
    if (D == 128) {
      if (NJ == 1) return resident_clusters_t<MODE, 128, 1, NT, SC>(size);
      if (NJ == 2) return resident_clusters_t<MODE, 128, 2, NT, SC>(size);
      if (NJ == 4) return resident_clusters_t<MODE, 128, 4, NT, SC>(size);
    } else if (D == 64) {
      if (NJ == 1) return resident_clusters_t<MODE, 64, 1, NT, SC>(size);
      if (NJ == 2) return resident_clusters_t<MODE, 64, 2, NT, SC>(size);
    }
    return 0;
  }
  static cudaError_t launch(const AttendParams& p, cudaStream_t s) {
    const int D = p.c.D, NJ = p.c.D / p.c.G;
    if (D == 128) {
      if (NJ == 1) return launch_t<MODE, 128, 1, NT, SC>(p, s);
      if (NJ == 2) return launch_t<MODE, 128, 2, NT, SC>(p, s);
      if (NJ == 4) return launch_t<MODE, 128, 4, NT, SC>(p, s);
    } else if (D == 64) {
      if (NJ == 1) return launch_t<MODE, 64, 1, NT, SC>(p, s);
      if (NJ == 2) return launch_t<MODE, 64, 2, NT, SC>(p, s);
    }
    return cudaErrorInvalidValue;
  }
};

template <int MODE, bool SC>
int resident_mode(int D, int NJ, int R) {
  return R <= 4 ? Variant<MODE, 1, SC>::resident(D, NJ) : Variant<MODE, 2, SC>::resident(D, NJ);
}

template <int MODE, bool SC>
int clusters_mode(int D, int NJ, int R, int size) {
  return R <= 4 ? Variant<MODE, 1, SC>::clusters(D, NJ, size) : Variant<MODE, 2, SC>::clusters(D, NJ, size);
}

template <int MODE, bool SC>
cudaError_t launch_mode(const AttendParams& p, cudaStream_t s) {
  return p.R <= 4 ? Variant<MODE, 1, SC>::launch(p, s) : Variant<MODE, 2, SC>::launch(p, s);
}

}  // namespace

// Per-mode entry points, explicitly instantiated in kvq_attend_<mode>.cu.
template <int MODE, bool SC>
int attend_resident_m(int D, int NJ, int R) { return resident_mode<MODE, SC>(D, NJ, R); }
template <int MODE, bool SC>
int attend_clusters_m(int D, int NJ, int R, int size) { return clusters_mode<MODE, SC>(D, NJ, R, size); }
template <int MODE, bool SC>
cudaError_t attend_launch_m(const AttendParams& p, cudaStream_t s) { return launch_mode<MODE, SC>(p, s); }
}  // namespace kvq
