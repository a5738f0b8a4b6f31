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

template <int MODE, int D>
struct Smem {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  static constexpr int TT = M::TT;
  static constexpr int KPLANE = TT * RW::KROW;
  static constexpr int VPLANE = (TT / 32) * D * RW::VROW;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = M::NP * KPLANE;
  static constexpr int KSZ_OFF = V_OFF + M::NP * VPLANE;
  static constexpr int KSZ_BYTES = (TT / 32) * 2 * D * 4;
  static constexpr int VSZ_OFF = KSZ_OFF + KSZ_BYTES;
  static constexpr int VSZ_BYTES = TT * 2 * (D / 32) * 4;
  static constexpr int SLOT = VSZ_OFF + VSZ_BYTES;
  static constexpr int QT_OFF = NSLOT * SLOT;                 // q~  [8][D] f32
  static constexpr int QH_OFF = QT_OFF + kMaxRows * D * 4;    // q^  [8][D] f32
  static constexpr int BM_OFF = QH_OFF + kMaxRows * D * 4;    // selection bitmap
  static constexpr int BM_WORDS = kMaxChunk / 32;
  static constexpr int BAR_OFF = BM_OFF + BM_WORDS * 4;
  static constexpr int MISC_OFF = BAR_OFF + 2 * NSLOT * 8;
  static constexpr int TOTAL = MISC_OFF + 64;
  // warp-merge scratch (after the pipeline drains), inside the slot area
  static constexpr int WM_OFF = 0;                            // [NW][8]
  static constexpr int WL_OFF = WM_OFF + NW * 8 * 4;          // [NW][8]
  static constexpr int WC_OFF = WL_OFF + NW * 8 * 4;          // [NW][8][4]
  static constexpr int WO_OFF = WC_OFF + NW * 8 * 4 * 4;      // [NW][8][D]
  static constexpr int SCRATCH = WO_OFF + NW * 8 * D * 4;
  static_assert(SCRATCH <= NSLOT * SLOT, "merge scratch must fit in the slot area");
  static_assert(SLOT % 16 == 0, "slots must stay 16-byte aligned");
};

// Tail-CTA shared layout (overlays the slot area of the same dynamic buffer).
template <int D>
struct TailSmem {
  static constexpr int TC = NTHREADS;                         // tokens per chunk
  static constexpr int QT_OFF = 0;                            // [8][D]
  static constexpr int LG_OFF = QT_OFF + kMaxRows * D * 4;    // [8][TC]
  static constexpr int ST_OFF = LG_OFF + kMaxRows * TC * 4;   // m[8], l[8], alpha[8]
  static constexpr int TOTAL = ST_OFF + 3 * kMaxRows * 4;
};

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// ------------------------------------------------------------------------------
// Combine: merge the S_total partials of unit u into out/lse.
// ------------------------------------------------------------------------------
template <int D>
__device__ void combine_unit(const AttendParams& p, long long u, int S_total) {
  const int PF = kPartialFloats(D);
  const float* base = p.partials + u * static_cast<long long>(S_total) * PF;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  for (int e = threadIdx.x; e < p.R * D; e += blockDim.x) {
    const int rho = e / D, d = e % D;
    float M = neg_inf();
    for (int s = 0; s < S_total; ++s) M = fmaxf(M, __ldcg(base + s * PF + rho));
    float L = 0.f, O = 0.f;
    if (M != neg_inf()) {
      for (int s = 0; s < S_total; ++s) {
        const float ms = __ldcg(base + s * PF + rho);
        if (ms == neg_inf()) continue;
        const float f = fast_exp2(ms - M);
        L += f * __ldcg(base + s * PF + kMaxRows + rho);
        O += f * __ldcg(base + s * PF + 2 * kMaxRows + rho * D + d);
      }
    }
    const int i = rho / p.HG, hh = rho % p.HG;
    const int h = kvh * p.HG + hh;
    const long long orow = (static_cast<long long>(b) * p.gamma + i) * p.Hq + h;
    const float val = (L > 0.f) ? O / L : 0.f;
    p.out[orow * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
    if (p.lse && d == 0) {
      p.lse[orow] = (L > 0.f) ? (M + log2f(L)) * 0.6931471805599453f : neg_inf();
    }
  }
}

// Arrive at the per-unit ticket; the last arriving CTA merges and resets it.
template <int D>
__device__ void ticket_and_combine(const AttendParams& p, long long u, int* sh_flag) {
  __threadfence();
  __syncthreads();
  const int S_total = p.S_q + 1;
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(p.counters + u, 1u);
    const int last = (prev == static_cast<unsigned>(S_total - 1));
    if (last) atomicExch(p.counters + u, 0u);
    *sh_flag = last;
  }
  __syncthreads();
  if (*sh_flag) {
    __threadfence();
    combine_unit<D>(p, u, S_total);
  }
}

// ------------------------------------------------------------------------------
// Tail CTA: residual bf16 tokens + causal pending tokens + selected 16-bit
// tokens, fp32 on CUDA cores, online softmax over chunks of TC tokens.
// ------------------------------------------------------------------------------
template <int D>
__device__ void tail_partial(const AttendParams& p, long long u, uint8_t* smem) {
  using TS = TailSmem<D>;
  float* qt = reinterpret_cast<float*>(smem + TS::QT_OFF);
  float* lg = reinterpret_cast<float*>(smem + TS::LG_OFF);
  float* st_m = reinterpret_cast<float*>(smem + TS::ST_OFF);
  float* st_l = st_m + kMaxRows;
  float* st_a = st_l + kMaxRows;
  const int tid = threadIdx.x;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  const int R = p.R;
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
  __syncthreads();

  const int G = p.c.G;
  const int NT = p.c.r + p.P + p.top_k;
  float o[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) o[r] = 0.f;

  // K/V row pointer of tail token `t`, and whether it exists at all.
  auto tail_row = [&](int t, const uint16_t*& kp, const uint16_t*& vp, int& pend) -> bool {
    pend = -1;
    if (t < p.c.r) {
      const int slot = (p.c.res_start + t) % (2 * G);
      const long long off = (u * 2 * G + slot) * D;
      kp = p.c.res_k + off;
      vp = p.c.res_v + off;
      return true;
    }
    t -= p.c.r;
    if (t < p.P) {
      const long long off = (u * p.P + t) * D;
      kp = p.pend_k + off;
      vp = p.pend_v + off;
      pend = t;
      return true;
    }
    t -= p.P;
    const int idx = p.sel_idx[u * p.top_k + t];
    if (idx < 0 || idx >= p.c.Lq) return false;
    const long long off = (u * p.top_k + t) * D;
    kp = p.sel_k + off;
    vp = p.sel_v + off;
    return true;
  };

  for (int c0 = 0; c0 < NT; c0 += TS::TC) {
    // logits
    {
      const int t = c0 + tid;
      float acc[kMaxRows];
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) acc[r] = 0.f;
      const uint16_t *kp = nullptr, *vp = nullptr;
      int pend = -1;
      const bool ok = (t < NT) && tail_row(t, kp, vp, pend);
      if (ok) {
        for (int d0 = 0; d0 < D; d0 += 8) {
          const uint4 raw = *reinterpret_cast<const uint4*>(kp + d0);
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
          float kf[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            kf[2 * k] = __uint_as_float(w4[k] << 16);
            kf[2 * k + 1] = __uint_as_float(w4[k] & 0xFFFF0000u);
          }
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) {
            if (r < R) {
#pragma unroll
              for (int k = 0; k < 8; ++k) acc[r] = fmaf(qt[r * D + d0 + k], kf[k], acc[r]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        bool vis = ok && r < R;
        if (vis && pend >= 0) vis = pend <= p.P - p.gamma + r / p.HG;
        lg[r * TS::TC + tid] = vis ? acc[r] : neg_inf();
      }
    }
    __syncthreads();
    // row statistics (one warp per row)
    {
      const int warp = tid / 32, lane = tid % 32;
      for (int r = warp; r < R; r += NTHREADS / 32) {
        float mx = neg_inf();
        for (int t = lane; t < TS::TC; t += 32) mx = fmaxf(mx, lg[r * TS::TC + t]);
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
        const float m_old = st_m[r];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        const float msafe = (m_new == neg_inf()) ? 0.f : m_new;
        for (int t = lane; t < TS::TC; t += 32) {
          const float x = lg[r * TS::TC + t];
          const float pr = (x == neg_inf()) ? 0.f : fast_exp2(x - msafe);
          lg[r * TS::TC + t] = pr;
          sum += pr;
        }
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
        if (lane == 0) {
          const float alpha = (m_old == neg_inf()) ? 0.f : fast_exp2(m_old - msafe);
          st_a[r] = alpha;
          st_l[r] = st_l[r] * alpha + sum;
          st_m[r] = m_new;
        }
      }
    }
    __syncthreads();
    // P.V: thread d accumulates channel d for all rows
    if (tid < D) {
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r)
        if (r < R) o[r] *= st_a[r];
      const int nt = min(TS::TC, NT - c0);
      for (int j = 0; j < nt; ++j) {
        const uint16_t *kp = nullptr, *vp = nullptr;
        int pend;
        if (!tail_row(c0 + j, kp, vp, pend)) continue;
        const float v = bf16_to_f32(vp[tid]);
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
          if (r < R) o[r] = fmaf(lg[r * TS::TC + j], v, o[r]);
      }
    }
    __syncthreads();
  }
  // write the partial (slot S_q of this unit)
  const int PF = kPartialFloats(D);
  float* dst = p.partials + (u * (p.S_q + 1) + p.S_q) * PF;
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
template <int MODE, int D, int NJ>
__global__ void __launch_bounds__(NTHREADS) attend_kernel(AttendParams p) {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  using L = Smem<MODE, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = lane >> 2, q = lane & 3;
  const long long nunits = static_cast<long long>(p.c.B) * p.c.Hkv;
  int* sh_flag = reinterpret_cast<int*>(smem + L::MISC_OFF);
  int* sh_abort = sh_flag + 1;

  if (blockIdx.x < nunits) {  // ---------------- tail CTA ----------------
    const long long u = blockIdx.x;
    tail_partial<D>(p, u, smem);
    ticket_and_combine<D>(p, u, sh_flag);
    return;
  }

  const long long qi = blockIdx.x - nunits;
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

  float* qt = reinterpret_cast<float*>(smem + L::QT_OFF);
  float* qh = reinterpret_cast<float*>(smem + L::QH_OFF);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L::BM_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + NSLOT;

  // ---- setup ----
  if (tid == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    *sh_abort = 0;
    fence_mbar_init();
  }
  const float qmul = static_cast<float>((1 << M::CB) * M::MULT);
  for (int e = tid; e < kMaxRows * D; e += blockDim.x) {
    const int rho = e / D, d = e % D;
    float v = 0.f;
    if (rho < R) {
      const int i = rho / p.HG, hh = rho % p.HG;
      const long long qoff = ((static_cast<long long>(b) * p.gamma + i) * p.Hq + kvh * p.HG + hh) * D + d;
      v = bf16_to_f32(p.q[qoff]) * p.qscale;
    }
    qt[e] = v;
    qh[e] = v * qmul;
  }
  const int bm_words = (ntok_chunk + 31) / 32;
  for (int e = tid; e < bm_words; e += blockDim.x) bitmap[e] = 0u;
  __syncthreads();
  for (int j = tid; j < p.top_k; j += blockDim.x) {
    const long long idx = p.sel_idx[u * p.top_k + j];
    if (idx >= t_begin && idx < t_end) {
      const int rel = static_cast<int>(idx - t_begin);
      atomicOr(bitmap + rel / 32, 1u << (rel % 32));
    }
  }
  __syncthreads();

  const long long u_tok = u * p.c.C;  // first token row of this unit in the planes

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
          float cpart = 0.f;
#pragma unroll
          for (int pp = 0; pp < D / 8; ++pp) {
            const int2 ch = pair_chan<MODE, D>(pp);
            const int c0 = qbase + ch.x, c1 = qbase + ch.y;
            const float w0 = qh[g * D + c0] * ks[c0];
            const float w1 = qh[g * D + c1] * ks[c1];
            const uint32_t hi = pack_half2(w0, w1);
            const float2 hf = unpack_half2(hi);
            const uint32_t lo = pack_half2(w0 - hf.x, w1 - hf.y);
            wa[pp / 2][(pp % 2) * 2 + 0] = hi;
            wa[pp / 2][(pp % 2) * 2 + 1] = lo;
            cpart += qt[g * D + c0] * kz[c0] + qt[g * D + c1] * kz[c1] - w0 - w1;
          }
          cpart += __shfl_xor_sync(0xffffffffu, cpart, 1);
          cpart += __shfl_xor_sync(0xffffffffu, cpart, 2);
          corr = cpart;
        }
        // ---- S^T = W x K^T over 4 n-tiles of 8 tokens ----
        float c[4][4];
        const uint8_t* kslab = sbase + L::K_OFF + (32 * sl) * RW::KROW + q * RW::KCHUNK;
#pragma unroll
        for (int jt = 0; jt < 4; ++jt) {
          c[jt][0] = corr; c[jt][1] = corr; c[jt][2] = 0.f; c[jt][3] = 0.f;
          uint32_t P[D / 8];
          key_pairs<MODE, D>(kslab + (4 * g + jt) * RW::KROW, L::KPLANE, P);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) mma16816(c[jt], wa[kk], P[2 * kk], P[2 * kk + 1]);
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
    float* dst = p.partials + (u * (p.S_q + 1) + split) * PF;
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
  ticket_and_combine<D>(p, u, sh_flag);
}

template <int MODE, int D, int NJ>
cudaError_t launch_t(const AttendParams& p, cudaStream_t s) {
  using L = Smem<MODE, D>;
  constexpr int smem = (L::TOTAL > TailSmem<D>::TOTAL) ? L::TOTAL : TailSmem<D>::TOTAL;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&attend_kernel<MODE, D, NJ>), smem);
  if (e != cudaSuccess) return e;
  const long long nunits = static_cast<long long>(p.c.B) * p.c.Hkv;
  const long long grid = nunits * (p.S_q + 1);
  attend_kernel<MODE, D, NJ><<<static_cast<unsigned>(grid), NTHREADS, smem, s>>>(p);
  return cudaGetLastError();
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
