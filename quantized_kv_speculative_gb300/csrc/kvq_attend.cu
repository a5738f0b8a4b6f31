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
// One launch, grid = B*Hkv tail CTAs followed by B*Hkv*S_q quantized-split CTAs.
//  * Quantized split: one producer warp streams 32..64-token tiles of the
//    mode's planes and scales into shared memory with 1-D bulk (TMA) copies on
//    an mbarrier ring.  Four consumer warps each own a contiguous run of tiles.
//    They dequantize in registers and run QK^T and PV on tensor cores
//    (m16n8k16, f16 codes exact; the folded key weights and the folded
//    probabilities are each split into high + low f16 parts).
//    Softmax is online in fp32 (base-2 logits).
//  * Tail CTA: the bf16 residual buffer, the pending speculative tokens (causal)
//    and the 16-bit selected tokens, on CUDA cores.
//  * Every CTA writes an (m, l, o) partial.  The CTA that arrives last at a
//    per-(b, kvh) atomic ticket merges all partials into the bf16 output and LSE,
//    then resets the ticket.  No CTA ever waits on another.
//
// Folding (no per-element dequant FMA): with q~ = q * sm_scale * log2(e) and
// key codes c (scale s, zero z per group and channel),
//   logit2 = sum_d q~_d (c s + z) = sum_d w'_d (1 + c/2^b) + sum_d (q~_d z_d - w'_d),
// with w'_d = 2^b q~_d s_d.  The value scale folds into the probabilities:
//   o = sum_t p_t (c s_t + z_t) = sum_t P'_t (1 + c/2^b) + sum_t (p_t z_t - P'_t),
// with P'_t = 2^b p_t s_t.
#include "kvq_modes.cuh"

namespace kvq {
namespace {

constexpr int NW = 4;                  // consumer warps
constexpr int SPW = 2;                 // stage slots per consumer warp
constexpr int NSLOT = NW * SPW;
constexpr int NTHREADS = (NW + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;

// Tail-CTA shared layout (overlays the slot area of the same dynamic buffer).
// K and V rows of one 64-token chunk are staged with a padded row stride so
// that lanes reading different rows hit different banks.
template <int D>
struct TailSmem {
  static constexpr int TC = 32;                               // tokens per chunk
  static constexpr int ROW = D * 2 + 16;                      // padded bf16 row, bytes
  static constexpr int QT_OFF = 0;                            // q~ [8][D] f32
  static constexpr int K_OFF = QT_OFF + kMaxRows * D * 4;     // [TC][ROW]
  static constexpr int V_OFF = K_OFF + TC * ROW;              // [TC][ROW]
  static constexpr int LG_OFF = V_OFF + TC * ROW;             // logits / p [8][TC]
  static constexpr int ST_OFF = LG_OFF + kMaxRows * TC * 4;   // m[8], l[8], alpha[8]
  static constexpr int OK_OFF = ST_OFF + 3 * kMaxRows * 4;    // per-token flags [TC]
  static constexpr int TOTAL = OK_OFF + TC * 4;
};

template <int MODE, int D, int NJ>
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
  static constexpr int QX_OFF = NSLOT * SLOT;                 // folded query, [D/8][32 lanes] float2
  static constexpr int BM_OFF = QX_OFF + (D / 8) * 32 * 8;    // selection bitmap
  static constexpr int BM_WORDS = kMaxChunk / 32;
  static constexpr int BAR_OFF = BM_OFF + BM_WORDS * 4;
  static constexpr int RING_END = BAR_OFF + 2 * NSLOT * 8;
  static constexpr int COMBINE_END = (2 * kMaxCombine * 8 + 16) * 4;
  // the ticket flag sits after whichever layout (ring, tail CTA, combine) is largest
  static constexpr int MISC_OFF0 = RING_END > TailSmem<D>::TOTAL ? RING_END : TailSmem<D>::TOTAL;
  static constexpr int MISC_OFF = (MISC_OFF0 > COMBINE_END ? MISC_OFF0 : COMBINE_END + 15) / 16 * 16;
  static constexpr int TOTAL = MISC_OFF + 64;
  // warp-merge scratch (after the pipeline drains), inside the slot area
  static constexpr int WM_OFF = 0;                            // [NW][8]
  static constexpr int WL_OFF = WM_OFF + NW * 8 * 4;          // [NW][8]
  static constexpr int WC_OFF = WL_OFF + NW * 8 * 4;          // [NW][8][4]
  static constexpr int WO_OFF = WC_OFF + NW * 8 * 4 * 4;      // [NW][8][D]
  static constexpr int SCRATCH = WO_OFF + NW * 8 * D * 4;
  static_assert(SCRATCH <= NSLOT * SLOT, "merge scratch must fit in the slot area");
  static_assert(TailSmem<D>::TOTAL <= MISC_OFF, "the tail layout must not reach the ticket flag");
  static_assert((2 * kMaxCombine * 8 + 16) * 4 <= MISC_OFF, "the combine scratch must not reach the ticket flag");
  static_assert(SLOT % 16 == 0, "slots must stay 16-byte aligned");
};

// 2^x with the hardware approximation (ex2.approx.ftz: relative error near
// 2^-22; -inf gives +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------------------
// Combine: merge the S_total partials of unit u into out/lse.  The split
// maxima and weights are staged in shared memory (S_total <= 256), then each
// thread streams float4 rows of the partial outputs with several splits in
// flight.
// ------------------------------------------------------------------------------
template <int D>
__device__ void combine_unit(const AttendParams& p, long long u, int S_total, float* sm) {
  const int PF = kPartialFloats(D);
  const float* base = p.partials + u * static_cast<long long>(S_total) * PF;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  float* ms = sm;                       // [S_total][8] split maxima
  float* wt = sm + kMaxCombine * 8;     // [S_total][8] l, then weights
  float* ml = wt + kMaxCombine * 8;     // M[8], L[8]
  const int tid = threadIdx.x;
  for (int e = tid; e < S_total * 8; e += blockDim.x) {
    const int s = e >> 3, r = e & 7;
    ms[e] = __ldcg(base + s * PF + r);
    wt[e] = __ldcg(base + s * PF + kMaxRows + r);
  }
  __syncthreads();
  if (tid < p.R) {
    float M = neg_inf();
    for (int s = 0; s < S_total; ++s) M = fmaxf(M, ms[s * 8 + tid]);
    float L = 0.f;
    if (M != neg_inf()) {
      for (int s = 0; s < S_total; ++s) {
        const float m = ms[s * 8 + tid];
        const float f = (m == neg_inf()) ? 0.f : fast_exp2(m - M);
        L += f * wt[s * 8 + tid];
        wt[s * 8 + tid] = f;
      }
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    for (int s = 0; s < S_total; ++s) wt[s * 8 + tid] = (M == neg_inf()) ? 0.f : wt[s * 8 + tid] * inv;
    ml[tid] = M;
    ml[8 + tid] = L;
  }
  __syncthreads();
  constexpr int D4 = D / 4;
  for (int item = tid; item < p.R * D4; item += blockDim.x) {
    const int rho = item / D4, d4 = item % D4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* src = reinterpret_cast<const float4*>(base + 2 * kMaxRows + rho * D) + d4;
#pragma unroll 8
    for (int s = 0; s < S_total; ++s) {
      const float w = wt[s * 8 + rho];
      const float4 v = __ldcg(src + static_cast<long long>(s) * (PF / 4));
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    const int i = rho / p.HG, hh = rho % p.HG;
    const int h = kvh * p.HG + hh;
    const long long orow = (static_cast<long long>(b) * p.gamma + i) * p.Hq + h;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p.out + orow * D + 4 * d4) = pk;
    if (p.lse && d4 == 0) {
      const float M = ml[rho], L = ml[8 + rho];
      p.lse[orow] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : neg_inf();
    }
  }
}

// Arrive at the per-unit ticket; the last arriving CTA merges and resets it.
template <int D>
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
    combine_unit<D>(p, u, S_total, combine_scratch);
  }
}

// ------------------------------------------------------------------------------
// Tail CTAs: residual bf16 tokens + causal pending tokens + selected 16-bit
// tokens, fp32 on CUDA cores.  The tail of one (b, kv head) is split over
// S_t CTAs.  Each stages 64-token chunks of K and V rows in shared memory (all
// loads in flight), then computes logits (thread <-> (row, token)), an online
// softmax, and P.V (thread <-> channel) from shared memory.
// ------------------------------------------------------------------------------
template <int D>
__device__ void tail_partial(const AttendParams& p, long long u, int tsplit, uint8_t* smem) {
  using TS = TailSmem<D>;
  float* qt = reinterpret_cast<float*>(smem + TS::QT_OFF);
  uint8_t* ks = smem + TS::K_OFF;
  uint8_t* vs = smem + TS::V_OFF;
  float* lg = reinterpret_cast<float*>(smem + TS::LG_OFF);
  float* st_m = reinterpret_cast<float*>(smem + TS::ST_OFF);
  float* st_l = st_m + kMaxRows;
  float* st_a = st_l + kMaxRows;
  int* tok_pend = reinterpret_cast<int*>(smem + TS::OK_OFF);   // -2 absent, -1 always visible, else pending index
  const int tid = threadIdx.x;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  const int R = p.R;
  const int G = p.c.G;
#pragma unroll 8
  for (int e = tid; e < kMaxRows * D; e += blockDim.x) {
    const int rho = e / D, d = e % D;
    float v = 0.f;
    if (rho < R) {
      const int i = rho / p.HG, hh = rho % p.HG;
      const long long qoff = ((static_cast<long long>(b) * p.gamma + i) * p.Hq + kvh * p.HG + hh) * D + d;
      v = bf16_to_f32(p.q[qoff]) * p.qscale;
    }
    qt[e] = v;
  }
  if (tid < kMaxRows) {
    st_m[tid] = neg_inf();
    st_l[tid] = 0.f;
  }
  // this CTA's token range of the unit's tail list
  const int NT = p.c.r + p.P + p.top_k;
  const int per = (NT + p.S_t - 1) / p.S_t;
  const int t_lo = min(NT, tsplit * per), t_hi = min(NT, t_lo + per);
  float o[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) o[r] = 0.f;
  __syncthreads();

  constexpr int VEC = D / 8;   // 16-byte vectors per row
  for (int c0 = t_lo; c0 < t_hi; c0 += TS::TC) {
    const int nt = min(TS::TC, t_hi - c0);
    // ---- stage K and V rows (16-byte vectors, all in flight) ----
#pragma unroll 4
    for (int e = tid; e < nt * VEC; e += blockDim.x) {
      const int j = e / VEC, c = e % VEC;
      int t = c0 + j;
      const uint16_t *kp = nullptr, *vp = nullptr;
      int flag = -2;
      if (t < p.c.r) {
        const int slot = (p.c.res_start + t) % (2 * G);
        const long long off = (u * 2 * G + slot) * D;
        kp = p.c.res_k + off;
        vp = p.c.res_v + off;
        flag = -1;
      } else if ((t -= p.c.r) < p.P) {
        const long long off = (u * p.P + t) * D;
        kp = p.pend_k + off;
        vp = p.pend_v + off;
        flag = t;
      } else {
        t -= p.P;
        const int idx = p.sel_idx[u * p.top_k + t];
        if (idx >= 0 && idx < p.c.Lq) {
          const long long off = (u * p.top_k + t) * D;
          kp = p.sel_k + off;
          vp = p.sel_v + off;
          flag = -1;
        }
      }
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (kp) {
        kv = reinterpret_cast<const uint4*>(kp)[c];
        vv = reinterpret_cast<const uint4*>(vp)[c];
      }
      *reinterpret_cast<uint4*>(ks + j * TS::ROW + c * 16) = kv;
      *reinterpret_cast<uint4*>(vs + j * TS::ROW + c * 16) = vv;
      if (c == 0) tok_pend[j] = flag;
    }
    __syncthreads();
    // ---- logits: thread <-> (row, token) ----
    for (int e = tid; e < kMaxRows * TS::TC; e += blockDim.x) {
      const int rho = e / TS::TC, j = e % TS::TC;
      float acc = neg_inf();
      const int flag = (j < nt) ? tok_pend[j] : -2;
      bool vis = (rho < R) && (flag != -2);
      if (vis && flag >= 0) vis = flag <= p.P - p.gamma + rho / p.HG;
      if (vis) {
        acc = 0.f;
        const float* qr = qt + rho * D;
        const uint8_t* kr = ks + j * TS::ROW;
#pragma unroll 4
        for (int c = 0; c < VEC; ++c) {
          const uint4 kw = *reinterpret_cast<const uint4*>(kr + c * 16);
          const float4 qa = *reinterpret_cast<const float4*>(qr + 8 * c);
          const float4 qb = *reinterpret_cast<const float4*>(qr + 8 * c + 4);
          acc = fmaf(qa.x, __uint_as_float(kw.x << 16), acc);
          acc = fmaf(qa.y, __uint_as_float(kw.x & 0xFFFF0000u), acc);
          acc = fmaf(qa.z, __uint_as_float(kw.y << 16), acc);
          acc = fmaf(qa.w, __uint_as_float(kw.y & 0xFFFF0000u), acc);
          acc = fmaf(qb.x, __uint_as_float(kw.z << 16), acc);
          acc = fmaf(qb.y, __uint_as_float(kw.z & 0xFFFF0000u), acc);
          acc = fmaf(qb.z, __uint_as_float(kw.w << 16), acc);
          acc = fmaf(qb.w, __uint_as_float(kw.w & 0xFFFF0000u), acc);
        }
      }
      lg[rho * TS::TC + j] = acc;
    }
    __syncthreads();
    // ---- online softmax statistics (one warp per row) ----
    {
      const int warp = tid / 32, lane = tid % 32;
      static_assert(TS::TC == 32, "one token per lane");
      for (int r = warp; r < R; r += NTHREADS / 32) {
        const float x0 = lg[r * TS::TC + lane];
        float mx = x0;
#pragma unroll
        for (int s2 = 16; s2 > 0; s2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s2));
        const float m_old = st_m[r];
        const float m_new = fmaxf(m_old, mx);
        const float msafe = (m_new == neg_inf()) ? 0.f : m_new;
        const float p0 = (x0 == neg_inf()) ? 0.f : fast_exp2(x0 - msafe);
        lg[r * TS::TC + lane] = p0;
        float sum = p0;
#pragma unroll
        for (int s2 = 16; s2 > 0; s2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s2);
        if (lane == 0) {
          const float alpha = (m_old == neg_inf()) ? 0.f : fast_exp2(m_old - msafe);
          st_a[r] = alpha;
          st_l[r] = st_l[r] * alpha + sum;
          st_m[r] = m_new;
        }
      }
    }
    __syncthreads();
    // ---- P.V: thread d accumulates channel d for all rows ----
    if (tid < D) {
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r)
        if (r < R) o[r] *= st_a[r];
      for (int j = 0; j < nt; ++j) {
        const float v = bf16_to_f32(*reinterpret_cast<const uint16_t*>(vs + j * TS::ROW + tid * 2));
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
          if (r < R) o[r] = fmaf(lg[r * TS::TC + j], v, o[r]);
      }
    }
    __syncthreads();
  }
  // write the partial (index S_q + tsplit of this unit)
  const int PF = kPartialFloats(D);
  float* dst = p.partials + (u * (p.S_q + p.S_t) + p.S_q + tsplit) * PF;
  if (tid < kMaxRows) {
    dst[tid] = (tid < R) ? st_m[tid] : neg_inf();
    dst[kMaxRows + tid] = (tid < R) ? st_l[tid] : 0.f;
  }
  if (tid < D) {
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r)
      if (r < R) dst[2 * kMaxRows + r * D + tid] = o[r];
  }
}

// ------------------------------------------------------------------------------
// Quantized split
// ------------------------------------------------------------------------------
// Three CTAs per SM for one channel block per token (G = D, the hierarchical
// cache's usual shape); the other variants keep more state per lane.
template <int MODE, int D, int NJ>
__global__ void __launch_bounds__(NTHREADS, (NJ == 1 ? 3 : 1)) attend_kernel(AttendParams p) {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  using L = Smem<MODE, D, NJ>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = lane >> 2, q = lane & 3;
  const long long nunits = static_cast<long long>(p.c.B) * p.c.Hkv;
  int* sh_flag = reinterpret_cast<int*>(smem + L::MISC_OFF);
  int* sh_abort = sh_flag + 1;

  const long long ntail = nunits * p.S_t;
  if (blockIdx.x < ntail) {  // ---------------- tail CTAs ----------------
    const long long u = blockIdx.x / p.S_t;
    tail_partial<D>(p, u, static_cast<int>(blockIdx.x % p.S_t), smem);
    __syncthreads();
    ticket_and_combine<D>(p, u, sh_flag, reinterpret_cast<float*>(smem));
    return;
  }

  const long long qi = blockIdx.x - ntail;
  const long long u = qi / p.S_q;
  const int split = static_cast<int>(qi % p.S_q);
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  const long long t_begin = static_cast<long long>(split) * p.chunk;
  const long long t_end = min(p.c.Lq, t_begin + p.chunk);
  const int ntok_chunk = static_cast<int>(max(0LL, t_end - t_begin));
  const int ntiles = (ntok_chunk + M::TT - 1) / M::TT;
  const int per_warp = (ntiles + NW - 1) / NW;
  constexpr int G = D / NJ;
  const int R = p.R;

  float2* qx = reinterpret_cast<float2*>(smem + L::QX_OFF);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L::BM_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + NSLOT;

  // ---- setup: barriers first, so the producer can start loading at once ----
  const int bm_words = (ntok_chunk + 31) / 32;
  if (tid == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    *sh_abort = 0;
    fence_mbar_init();
  }
  for (int e = tid; e < bm_words; e += blockDim.x) bitmap[e] = 0u;
  __syncthreads();
  const long long u_tok = u * p.c.C;  // first token row of this unit in the planes
  const float qmul = static_cast<float>((1 << M::CB) * M::MULT);
  if (warp < NW) {
    // consumers: folded queries and the selection bitmap, while the first tiles load
    constexpr int NC = NW * 32;
    // q^ = 2^CB * MULT * sm_scale * log2(e) * q, stored per (pair, lane) as the
    // two channels that lane needs for that pair: conflict-free 8-byte reads
#pragma unroll 4
    for (int e = tid; e < (D / 8) * 32; e += NC) {
      const int pp = e / 32, ln = e % 32;
      const int rho = ln >> 2, qq = ln & 3;
      float2 v = make_float2(0.f, 0.f);
      if (rho < R) {
        const int i = rho / p.HG, hh = rho % p.HG;
        const long long qrow = ((static_cast<long long>(b) * p.gamma + i) * p.Hq + kvh * p.HG + hh) * D;
        const int2 ch = pair_chan<MODE, D>(pp);
        const int c0 = qq * (D / 4) + ch.x, c1 = qq * (D / 4) + ch.y;
        v.x = bf16_to_f32(p.q[qrow + c0]) * p.qscale * qmul;
        v.y = bf16_to_f32(p.q[qrow + c1]) * p.qscale * qmul;
      }
      qx[e] = v;
    }
    for (int j = tid; j < p.top_k; j += NC) {
      const long long idx = p.sel_idx[u * p.top_k + j];
      if (idx >= t_begin && idx < t_end) {
        const int rel = static_cast<int>(idx - t_begin);
        atomicOr(bitmap + rel / 32, 1u << (rel % 32));
      }
    }
    asm volatile("bar.sync 2, %0;" ::"n"(NW * 32));
  }

  if (warp == NW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int j = 0; j < per_warp && !*reinterpret_cast<volatile int*>(sh_abort); ++j) {
        for (int w = 0; w < NW; ++w) {
          const int ti = w * per_warp + j;
          if (ti >= ntiles || j >= per_warp) continue;
          const int slot = w * SPW + (j % SPW);
          const uint32_t par = ((j / SPW) & 1) ^ 1;
          if (!mbar_wait_bounded(empty + slot, par, p.wait_limit)) {
            record_status(p.status, KVQ_ERR_DEVICE_TIMEOUT);
            *reinterpret_cast<volatile int*>(sh_abort) = 1;
            break;
          }
          const long long t0 = t_begin + static_cast<long long>(ti) * M::TT;
          const int nt = static_cast<int>(min(static_cast<long long>(M::TT), t_end - t0));
          const long long g_first = t0 / G, g_last = (t0 + nt - 1) / G;
          const uint32_t kb = nt * RW::KROW, vb = (nt / 32) * D * RW::VROW;
          const uint32_t kszb = static_cast<uint32_t>(g_last - g_first + 1) * 2 * D * 4;
          const uint32_t vszb = nt * 2 * NJ * 4;
          uint8_t* sbase = smem + slot * L::SLOT;
          mbar_arrive_expect_tx(full + slot, M::NP * (kb + vb) + kszb + vszb);
#pragma unroll
          for (int pl = 0; pl < M::NP; ++pl) {
            bulk_g2s(sbase + L::K_OFF + pl * L::KPLANE, p.c.kplane[pl] + (u_tok + t0) * RW::KROW, kb,
                     full + slot, pol);
            bulk_g2s(sbase + L::V_OFF + pl * L::VPLANE,
                     p.c.vplane[pl] + ((u_tok + t0) / 32) * D * RW::VROW, vb, full + slot, pol);
          }
          bulk_g2s(sbase + L::KSZ_OFF, p.c.ksz + (u * (p.c.C / G) + g_first) * 2 * D, kszb,
                   full + slot, pol);
          bulk_g2s(sbase + L::VSZ_OFF, p.c.vsz + (u_tok + t0) * 2 * NJ, vszb, full + slot, pol);
        }
      }
    }
  } else {
    // ---------------- consumers ----------------
    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run = neg_inf(), l_run = 0.f;
    uint32_t wa[D / 16][4];
    float corr = 0.f;
    long long cur_grp = -1;
    const int qbase = q * (D / 4);
    const bool row_ok = g < R;

    for (int j = 0; j < per_warp; ++j) {
      const int ti = warp * per_warp + j;
      if (ti >= ntiles) break;
      const int slot = warp * SPW + (j % SPW);
      const uint32_t par = (j / SPW) & 1;
      if (!mbar_wait_bounded(full + slot, par, p.wait_limit)) {
        record_status(p.status, KVQ_ERR_DEVICE_TIMEOUT);
        *reinterpret_cast<volatile int*>(sh_abort) = 1;
        break;
      }
      if (*reinterpret_cast<volatile int*>(sh_abort)) break;
      const long long t0 = t_begin + static_cast<long long>(ti) * M::TT;
      const int nt = static_cast<int>(min(static_cast<long long>(M::TT), t_end - t0));
      const long long g_first = t0 / G;
      const uint8_t* sbase = smem + slot * L::SLOT;
      const float* ksz = reinterpret_cast<const float*>(sbase + L::KSZ_OFF);
      const float* vsz = reinterpret_cast<const float*>(sbase + L::VSZ_OFF);

      for (int sl = 0; sl < nt / 32; ++sl) {
        const long long tok0 = t0 + 32 * sl;
        const long long grp = tok0 / G;
        if (grp != cur_grp) {
          // ---- folded key weights for this group (high + low f16 parts) ----
          cur_grp = grp;
          const float* ks = ksz + (grp - g_first) * 2 * D;
          const float* kz = ks + D;
          // correction sum_d (q~_d z_d - w'_d), with q~ = q^ / (2^CB MULT) exactly
          float zsum = 0.f, wsum = 0.f;
#pragma unroll
          for (int pp = 0; pp < D / 8; ++pp) {
            const int2 ch = pair_chan<MODE, D>(pp);
            const int c0 = qbase + ch.x, c1 = qbase + ch.y;
            const float2 qv = qx[pp * 32 + lane];
            const float w0 = qv.x * ks[c0];
            const float w1 = qv.y * ks[c1];
            const uint32_t hi = pack_half2(w0, w1);
            const float2 hf = unpack_half2(hi);
            const uint32_t lo = pack_half2(w0 - hf.x, w1 - hf.y);
            wa[pp / 2][(pp % 2) * 2 + 0] = hi;
            wa[pp / 2][(pp % 2) * 2 + 1] = lo;
            zsum = fmaf(qv.x, kz[c0], fmaf(qv.y, kz[c1], zsum));
            wsum += w0 + w1;
          }
          float cpart = fmaf(zsum, 1.0f / qmul, -wsum);
          cpart += __shfl_xor_sync(0xffffffffu, cpart, 1);
          cpart += __shfl_xor_sync(0xffffffffu, cpart, 2);
          corr = cpart;
        }
        // ---- S^T = W x K^T over 4 n-tiles of 8 tokens ----
        float c[4][4];
        const uint8_t* kslab = sbase + L::K_OFF + (32 * sl) * RW::KROW + q * RW::KCHUNK;
        {
          // the four n-tiles are independent accumulation chains: k-step outer
          uint32_t P[4][D / 8];
#pragma unroll
          for (int jt = 0; jt < 4; ++jt) {
            c[jt][0] = corr; c[jt][1] = corr; c[jt][2] = 0.f; c[jt][3] = 0.f;
            key_pairs<MODE, D>(kslab + (4 * g + jt) * RW::KROW, L::KPLANE, P[jt]);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
            for (int jt = 0; jt < 4; ++jt) mma16816(c[jt], wa[kk], P[jt][2 * kk], P[jt][2 * kk + 1]);
        }
        // ---- mask + online softmax (row g; tokens 8q+jt and 8q+jt+4) ----
        const uint32_t bm = bitmap[static_cast<int>(tok0 - t_begin) / 32] >> (8 * q);
        float x[4][2];
        float mx = neg_inf();
#pragma unroll
        for (int jt = 0; jt < 4; ++jt) {
          const bool m0 = !row_ok || ((bm >> jt) & 1u);
          const bool m1 = !row_ok || ((bm >> (jt + 4)) & 1u);
          x[jt][0] = m0 ? neg_inf() : c[jt][0] + c[jt][2];
          x[jt][1] = m1 ? neg_inf() : c[jt][1] + c[jt][3];
          mx = fmaxf(mx, fmaxf(x[jt][0], x[jt][1]));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float msafe = (m_new == neg_inf()) ? 0.f : m_new;
        const float alpha = (m_run == neg_inf()) ? 0.f : fast_exp2(m_run - msafe);
        float pr[4][2];
        float psum = 0.f;
#pragma unroll
        for (int jt = 0; jt < 4; ++jt) {
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            pr[jt][e2] = (x[jt][e2] == neg_inf()) ? 0.f : fast_exp2(x[jt][e2] - msafe);
            psum += pr[jt][e2];
          }
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        // rows 2q, 2q+1 of O^T live in this lane: their rescale factors
        const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * q);
        const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * q + 4);

        // ---- P.V, one channel block (G channels) at a time ----
        // The slab's products go into fresh accumulators.  Its correction
        // sum_t (p_t z_t - P'_t), which removes the zero points and the
        // encoding's constant 1, is added before the merge into the running
        // output.  So the running sum only ever holds output-sized values.
        const uint8_t* vslab = sbase + L::V_OFF + sl * D * RW::VROW;
        const float vmul = qmul;  // 2^CB * MULT
#pragma unroll
        for (int jv = 0; jv < NJ; ++jv) {
          // P'_t = 2^CB * MULT * p_t * s_t, split into f16 high + low parts
          float pq[4][2];
          float zc = 0.f;
#pragma unroll
          for (int jt = 0; jt < 4; ++jt) {
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int tk = 32 * sl + 8 * q + jt + 4 * e2;   // token within the tile
              const float s = vsz[tk * 2 * NJ + jv];
              const float z = vsz[tk * 2 * NJ + NJ + jv];
              pq[jt][e2] = pr[jt][e2] * s * vmul;
              zc += pr[jt][e2] * z;
            }
          }
          uint32_t bq[2][2][2];   // [k-step][high/low][register]
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
              const float x0 = pq[2 * ks + r2][0], x1 = pq[2 * ks + r2][1];
              const uint32_t hi = pack_half2(x0, x1);
              const float2 fh = unpack_half2(hi);
              const uint32_t lo = pack_half2(x0 - fh.x, x1 - fh.y);
              const float2 fl = unpack_half2(lo);
              bq[ks][0][r2] = hi;
              bq[ks][1][r2] = lo;
              zc -= (fh.x + fh.y) + (fl.x + fl.y);
            }
          }
          // row g's correction for this slab, then the values for rows 2q, 2q+1
          zc += __shfl_xor_sync(0xffffffffu, zc, 1);
          zc += __shfl_xor_sync(0xffffffffu, zc, 2);
          const float z_lo = __shfl_sync(0xffffffffu, zc, 8 * q);
          const float z_hi = __shfl_sync(0xffffffffu, zc, 8 * q + 4);
#pragma unroll
          for (int mt = jv * (G / 16); mt < (jv + 1) * (G / 16); ++mt) {
            uint32_t a[2][4];
            const uint8_t* va = vslab + (16 * mt + g) * RW::VROW;
            value_frags<MODE>(va, va + 8 * RW::VROW, L::VPLANE, q, a);
            float os[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(os, a[0], bq[0][0][0], bq[0][0][1]);
            mma16816(os, a[0], bq[0][1][0], bq[0][1][1]);
            mma16816(os, a[1], bq[1][0][0], bq[1][0][1]);
            mma16816(os, a[1], bq[1][1][0], bq[1][1][1]);
            o[mt][0] = fmaf(o[mt][0], a_lo, os[0] + z_lo);
            o[mt][1] = fmaf(o[mt][1], a_hi, os[1] + z_hi);
            o[mt][2] = fmaf(o[mt][2], a_lo, os[2] + z_lo);
            o[mt][3] = fmaf(o[mt][3], a_hi, os[3] + z_hi);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + slot);
    }

    // ---- per-warp results to shared scratch (after everyone left the ring) ----
    float lsum = l_run;
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    // the stage ring must be idle before the slot area is reused
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32));
    float* wm = reinterpret_cast<float*>(smem + L::WM_OFF);
    float* wl = reinterpret_cast<float*>(smem + L::WL_OFF);
    float* wo = reinterpret_cast<float*>(smem + L::WO_OFF);
    if (q == 0) {
      wm[warp * 8 + g] = m_run;
      wl[warp * 8 + g] = lsum;
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      const int ca = 16 * mt + g, cb = ca + 8;
      wo[(warp * 8 + 2 * q) * D + ca] = o[mt][0];
      wo[(warp * 8 + 2 * q + 1) * D + ca] = o[mt][1];
      wo[(warp * 8 + 2 * q) * D + cb] = o[mt][2];
      wo[(warp * 8 + 2 * q + 1) * D + cb] = o[mt][3];
    }
  }
  __syncthreads();

  // ---- drain: the producer's copies must all have landed before exit ----
  // (only matters after an abort; in normal runs every phase completed)
  if (*reinterpret_cast<volatile int*>(sh_abort) && warp == NW && lane == 0) {
    for (int w = 0; w < NW; ++w) {
      const int issued = min(per_warp, max(0, ntiles - w * per_warp));
      for (int s2 = 0; s2 < SPW && s2 < issued; ++s2) {
        // last use of slot (w, s2): j = largest j < issued with j % SPW == s2
        const int jl = ((issued - 1 - s2) / SPW) * SPW + s2;
        mbar_wait_bounded(full + w * SPW + s2, (jl / SPW) & 1, p.wait_limit);
      }
    }
  }
  __syncthreads();

  // ---- CTA merge of the four warps -> partial ----
  {
    const float* wm = reinterpret_cast<const float*>(smem + L::WM_OFF);
    const float* wl = reinterpret_cast<const float*>(smem + L::WL_OFF);
    const float* wo = reinterpret_cast<const float*>(smem + L::WO_OFF);
    const int PF = kPartialFloats(D);
    float* dst = p.partials + (u * (p.S_q + p.S_t) + split) * PF;
    for (int e = tid; e < R * D; e += blockDim.x) {
      const int rho = e / D, d = e % D;
      float Mx = neg_inf();
#pragma unroll
      for (int w = 0; w < NW; ++w) Mx = fmaxf(Mx, wm[w * 8 + rho]);
      float lt = 0.f, ot = 0.f;
      if (Mx != neg_inf()) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float mw = wm[w * 8 + rho];
          if (mw == neg_inf()) continue;
          const float f = fast_exp2(mw - Mx);
          lt += f * wl[w * 8 + rho];
          ot += f * wo[(w * 8 + rho) * D + d];
        }
      }
      dst[2 * kMaxRows + rho * D + d] = ot;
      if (d == 0) {
        dst[rho] = Mx;
        dst[kMaxRows + rho] = lt;
      }
    }
  }
  __syncthreads();
  ticket_and_combine<D>(p, u, sh_flag, reinterpret_cast<float*>(smem));
}

template <int MODE, int D, int NJ>
cudaError_t launch_t(const AttendParams& p, cudaStream_t s) {
  using L = Smem<MODE, D, NJ>;
  constexpr int smem = (L::TOTAL > TailSmem<D>::TOTAL) ? L::TOTAL : TailSmem<D>::TOTAL;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&attend_kernel<MODE, D, NJ>), smem);
  if (e != cudaSuccess) return e;
  const long long nunits = static_cast<long long>(p.c.B) * p.c.Hkv;
  const long long grid = nunits * (p.S_q + p.S_t);
  attend_kernel<MODE, D, NJ><<<static_cast<unsigned>(grid), NTHREADS, smem, s>>>(p);
  return cudaGetLastError();
}

// Resident CTAs per SM of one kernel variant times the SM count, queried once
// per device (the split count is sized to fill whole waves).
template <int MODE, int D, int NJ>
int resident_ctas_t() {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  if (cached[dev] > 0) return cached[dev];
  using L = Smem<MODE, D, NJ>;
  constexpr int smem = (L::TOTAL > TailSmem<D>::TOTAL) ? L::TOTAL : TailSmem<D>::TOTAL;
  if (set_smem_once(reinterpret_cast<const void*>(&attend_kernel<MODE, D, NJ>), smem) != cudaSuccess) return 0;
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attend_kernel<MODE, D, NJ>, NTHREADS, smem) != cudaSuccess)
    return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cached[dev] = per_sm * sms;
  return cached[dev];
}

template <int MODE>
int resident_mode(int D, int NJ) {
  if (D == 128) {
    if (NJ == 1) return resident_ctas_t<MODE, 128, 1>();
    if (NJ == 2) return resident_ctas_t<MODE, 128, 2>();
    if (NJ == 4) return resident_ctas_t<MODE, 128, 4>();
  } else if (D == 64) {
    if (NJ == 1) return resident_ctas_t<MODE, 64, 1>();
    if (NJ == 2) return resident_ctas_t<MODE, 64, 2>();
  }
  return 0;
}

template <int MODE>
cudaError_t launch_mode(const AttendParams& p, cudaStream_t s) {
  const int D = p.c.D, NJ = p.c.D / p.c.G;
  if (D == 128) {
    if (NJ == 1) return launch_t<MODE, 128, 1>(p, s);
    if (NJ == 2) return launch_t<MODE, 128, 2>(p, s);
    if (NJ == 4) return launch_t<MODE, 128, 4>(p, s);
  } else if (D == 64) {
    if (NJ == 1) return launch_t<MODE, 64, 1>(p, s);
    if (NJ == 2) return launch_t<MODE, 64, 2>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int attend_resident_ctas(int mode, int D, int G) {
  const int NJ = D / G;
  switch (mode) {
    case KVQ_MODE_INT8: return resident_mode<KVQ_MODE_INT8>(D, NJ);
    case KVQ_MODE_INT4: return resident_mode<KVQ_MODE_INT4>(D, NJ);
    case KVQ_MODE_INT2: return resident_mode<KVQ_MODE_INT2>(D, NJ);
    case KVQ_MODE_INT1: return resident_mode<KVQ_MODE_INT1>(D, NJ);
    default: return 0;
  }
}

cudaError_t launch_attend(const AttendParams& p, int mode, cudaStream_t s) {
  switch (mode) {
    case KVQ_MODE_INT8: return launch_mode<KVQ_MODE_INT8>(p, s);
    case KVQ_MODE_INT4: return launch_mode<KVQ_MODE_INT4>(p, s);
    case KVQ_MODE_INT2: return launch_mode<KVQ_MODE_INT2>(p, s);
    case KVQ_MODE_INT1: return launch_mode<KVQ_MODE_INT1>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

// Bounded-wait self test: one CTA waits on an mbarrier that nothing arrives at.
__global__ void wait_selftest_kernel(int* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0, limit)) record_status(status, KVQ_ERR_DEVICE_TIMEOUT);
    // leave the barrier consistent: complete the pending phase before exit
    mbar_arrive(&bar);
  }
}

cudaError_t launch_wait_selftest(int* status, long long limit, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit);
  return cudaGetLastError();
}

}  // namespace kvq
