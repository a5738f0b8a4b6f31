// Per-KV-head top-k of the quantized tokens under the low-bit keys.
//
// SpeCache page, "Approach": a speculative token is decoded alongside the
// output token, and its attention over the low-bit KV copy predicts the top-k
// KV pairs to fetch at 16 bits for the next step.  Scores use the summed query
// of the speculative token's heads that share the KV head.  Per key group the
// score is an exact integer dot product of the codes with the folded query
// rounded to 22-bit integers, then scaled:
//   W_d = rint(fp32(qs_d * s_d) * 2^(21-e)), S_t = sum_d W_d c_{t,d},
//   score_t = fp32(fp32(fp32(S_t) * 2^(e-21)) + beta),
//   beta = pairwise tree over 32 lane-chunks of sequential fp32 sums of fp32(qs_d * z_d).
// The dot product runs on tensor cores.  W is split into two f16-exact integer
// halves (|hi|, |lo| <= 1024, W = 2048 hi + lo).  The codes are exact f16
// values 1 + c/2^b.  Every partial sum is a multiple of 2^-b below 2^18, so the
// fp32 accumulation is exact in any order.  fp32(S_t) = fp32(2048 S_hi + S_lo) is
// then a single correctly rounded fp32 add of two exact values.
//
// One launch: B*Hkv*S CTAs, sized to run in a single wave.  Each CTA scores one
// chunk (bulk-copied tiles on an mbarrier ring, as in attention) into 32-bit
// order keys, radix-selects its top k by (score desc, index asc), and writes k
// candidates.  The last CTA of each (b, kvh), found through an atomic ticket,
// radix-selects the k best of the S*k candidates under the unique composite key
// (order key, ~index), then places each winner by counting the winners above it.
#include "kvq_modes.cuh"

namespace kvq {
namespace {

constexpr int NW = 4;
constexpr int SPW = 2;
constexpr int NSLOT = NW * SPW;
constexpr int NTHREADS = (NW + 1) * 32;

template <int MODE, int D>
struct TopkSmem {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  static constexpr int TT = M::TT;
  static constexpr int KPLANE = TT * RW::KROW;
  static constexpr int KSZ_OFF = KPLANE;                      // only the upper/only plane is read
  static constexpr int KSZ_BYTES = (TT / 32) * 2 * D * 4;
  static constexpr int SLOT = KSZ_OFF + KSZ_BYTES;
  static constexpr int SC_OFF = NSLOT * SLOT;                 // order keys / merge keys
  static constexpr int SC_BYTES = kTopkMaxCand * 8;           // >= kTopkMaxChunk * 4
  static constexpr int QS_OFF = SC_OFF + SC_BYTES;            // qs[D]
  static constexpr int HIST_OFF = QS_OFF + D * 4;             // hist[256]
  static constexpr int BAR_OFF = HIST_OFF + 256 * 4;
  static constexpr int MISC_OFF = BAR_OFF + 2 * NSLOT * 8;
  static constexpr int TOTAL = MISC_OFF + 64;
  static_assert(kTopkMaxChunk * 4 <= SC_BYTES, "chunk scores must fit");
  static_assert(SLOT % 16 == 0, "slots must stay 16-byte aligned");
  static_assert(NSLOT * SLOT >= 2 * kMaxTopk * 4, "the merge winners reuse the stage area");
};

__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t b = __float_as_uint(__fadd_rn(s, 0.0f));  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_to_score(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}

__device__ __forceinline__ float pow2f(int e) {  // 2^e for -126 <= e <= 127
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// Block-wide radix select, 8-bit digits from the most significant.  Among the
// i < n for which take(i, key) is true, it finds the kth largest key T
// (1 <= kth <= number taken).  On return st[0] = T and st[2] = how many of the
// taken keys equal to T belong to the kth largest.  Every thread of the block
// calls it; st[0..2] and hist[256] are shared memory.
template <typename F>
__device__ void radix_select(int n, int kth, F take, uint32_t* hist, int* st) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    st[0] = 0;
    st[1] = 0;
    st[2] = kth;
  }
  const int nround = (n + blockDim.x - 1) / blockDim.x * blockDim.x;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    const uint32_t prefix = static_cast<uint32_t>(st[0]), mask = static_cast<uint32_t>(st[1]);
    // warp-aggregated histogram: lanes with the same bin add once
    for (int i = tid; i < nround; i += blockDim.x) {
      uint32_t key = 0, bin = 0xFFFFFFFFu;
      bool ok = false;
      if (i < n) {
        ok = take(i, key) && (key & mask) == prefix;
        if (ok) bin = (key >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (ok && (__ffs(peers) - 1) == lane) atomicAdd(hist + bin, static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    if (warp == 0) {
      // Lane l owns bins 255-8l .. 248-8l (descending); a warp scan gives the
      // count above each lane, and the lane holding the kth key picks its digit.
      uint32_t c[8];
      uint32_t tot = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        c[k] = hist[255 - 8 * lane - k];
        tot += c[k];
      }
      uint32_t inc = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const uint32_t excl = inc - tot;
      const uint32_t remaining = static_cast<uint32_t>(st[2]);
      if (excl < remaining && remaining <= inc) {
        uint32_t cum = excl;
        int digit = 255 - 8 * lane - 7;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (cum + c[k] >= remaining) {
            digit = 255 - 8 * lane - k;
            break;
          }
          cum += c[k];
        }
        st[2] = static_cast<int>(remaining - cum);
        st[0] = static_cast<int>(prefix | (static_cast<uint32_t>(digit) << shift));
        st[1] = static_cast<int>(mask | (255u << shift));
      }
    }
    __syncthreads();
  }
}

template <int MODE, int D>
__global__ void __launch_bounds__(NTHREADS) topk_kernel(TopkParams p) {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  using L = TopkSmem<MODE, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = lane >> 2, q = lane & 3;
  const long long u = blockIdx.x / p.S;
  const int split = blockIdx.x % p.S;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  const int G = p.c.G;
  const long long t_begin = static_cast<long long>(split) * p.chunk;
  const long long t_end = min(p.c.Lq, t_begin + p.chunk);
  const int n = static_cast<int>(max(0LL, t_end - t_begin));
  const int ntiles = (n + M::TT - 1) / M::TT;
  const int per_warp = (ntiles + NW - 1) / NW;
  const int K = p.k;

  uint32_t* okeys = reinterpret_cast<uint32_t*>(smem + L::SC_OFF);
  float* qs = reinterpret_cast<float*>(smem + L::QS_OFF);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + L::HIST_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + NSLOT;
  int* misc = reinterpret_cast<int*>(smem + L::MISC_OFF);   // [0] abort, [1] flag, [2..] select state

  if (tid == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    misc[0] = 0;
    fence_mbar_init();
  }
  // summed query: ascending head order, fp32
  for (int d = tid; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int hh = 0; hh < p.HG; ++hh) {
      const long long off = (static_cast<long long>(b) * p.Hq + kvh * p.HG + hh) * D + d;
      acc = __fadd_rn(acc, bf16_to_f32(p.q[off]));
    }
    qs[d] = acc;
  }
  __syncthreads();
  volatile int* abort_flag = misc;
  const long long u_tok = u * p.c.C;

  if (warp == NW) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int j = 0; j < per_warp && !*abort_flag; ++j) {
        for (int w = 0; w < NW; ++w) {
          const int ti = w * per_warp + j;
          if (ti >= ntiles) continue;
          const int slot = w * SPW + (j % SPW);
          if (!mbar_wait_bounded(empty + slot, ((j / SPW) & 1) ^ 1, p.wait_limit)) {
            record_status(p.status, KVQ_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          const long long t0 = t_begin + static_cast<long long>(ti) * M::TT;
          const int nt = static_cast<int>(min(static_cast<long long>(M::TT), t_end - t0));
          const long long g_first = t0 / G, g_last = (t0 + nt - 1) / G;
          const uint32_t kb = nt * RW::KROW;
          const uint32_t kszb = static_cast<uint32_t>(g_last - g_first + 1) * 2 * D * 4;
          uint8_t* sbase = smem + slot * L::SLOT;
          mbar_arrive_expect_tx(full + slot, kb + kszb);
          bulk_g2s(sbase, p.c.kplane[0] + (u_tok + t0) * RW::KROW, kb, full + slot, pol);
          bulk_g2s(sbase + L::KSZ_OFF, p.c.ksz + (u * (p.c.C / G) + g_first) * 2 * D, kszb,
                   full + slot, pol);
        }
      }
    }
  } else {
    uint32_t wa[D / 16][4];
    float neg_hi = 0.f, neg_lo = 0.f, unit = 1.f, beta = 0.f;
    long long cur_grp = -1;
    const int qbase = q * (D / 4);
    const float smul = static_cast<float>(M::MULT);
    const float cbmul = static_cast<float>(1 << M::CB);
    for (int j = 0; j < per_warp; ++j) {
      const int ti = warp * per_warp + j;
      if (ti >= ntiles) break;
      const int slot = warp * SPW + (j % SPW);
      if (!mbar_wait_bounded(full + slot, (j / SPW) & 1, p.wait_limit)) {
        record_status(p.status, KVQ_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      const long long t0 = t_begin + static_cast<long long>(ti) * M::TT;
      const int nt = static_cast<int>(min(static_cast<long long>(M::TT), t_end - t0));
      const long long g_first = t0 / G;
      const uint8_t* sbase = smem + slot * L::SLOT;
      const float* ksz = reinterpret_cast<const float*>(sbase + L::KSZ_OFF);
      for (int sl = 0; sl < nt / 32; ++sl) {
        const long long tok0 = t0 + 32 * sl;
        const long long grp = tok0 / G;
        if (grp != cur_grp) {
          cur_grp = grp;
          const float* ks = ksz + (grp - g_first) * 2 * D;
          const float* kz = ks + D;
          // max |w| and beta over lane chunks of D/32 channels
          float mxw = 0.f, bp = 0.f;
          for (int d = lane * (D / 32); d < (lane + 1) * (D / 32); ++d) {
            const float w = __fmul_rn(qs[d], __fmul_rn(ks[d], smul));
            mxw = fmaxf(mxw, fabsf(w));
            bp = __fadd_rn(bp, __fmul_rn(qs[d], kz[d]));
          }
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            mxw = fmaxf(mxw, __shfl_xor_sync(0xffffffffu, mxw, o));
            bp = __fadd_rn(bp, __shfl_xor_sync(0xffffffffu, bp, o));
          }
          beta = bp;
          int e = 0;
          if (mxw > 0.f) frexpf(mxw, &e);
          e = max(e, -100);
          const float up = pow2f(21 - e);
          unit = pow2f(e - 21);
          float shi = 0.f, slo = 0.f;
#pragma unroll
          for (int pp = 0; pp < D / 8; ++pp) {
            const int2 ch = pair_chan<MODE, D>(pp);
            const int c0 = qbase + ch.x, c1 = qbase + ch.y;
            const float W0 = rintf(__fmul_rn(__fmul_rn(qs[c0], __fmul_rn(ks[c0], smul)), up));
            const float W1 = rintf(__fmul_rn(__fmul_rn(qs[c1], __fmul_rn(ks[c1], smul)), up));
            const float h0 = floorf(__fmul_rn(__fadd_rn(W0, 1024.f), 1.0f / 2048.f));
            const float h1 = floorf(__fmul_rn(__fadd_rn(W1, 1024.f), 1.0f / 2048.f));
            const float l0 = __fsub_rn(W0, __fmul_rn(2048.f, h0));
            const float l1 = __fsub_rn(W1, __fmul_rn(2048.f, h1));
            const bool mine = (g == 0);
            wa[pp / 2][(pp % 2) * 2 + 0] = mine ? pack_half2(h0, h1) : 0u;
            wa[pp / 2][(pp % 2) * 2 + 1] = mine ? pack_half2(l0, l1) : 0u;
            shi += h0 + h1;
            slo += l0 + l1;
          }
          shi += __shfl_xor_sync(0xffffffffu, shi, 1);
          shi += __shfl_xor_sync(0xffffffffu, shi, 2);
          slo += __shfl_xor_sync(0xffffffffu, slo, 1);
          slo += __shfl_xor_sync(0xffffffffu, slo, 2);
          neg_hi = -shi;
          neg_lo = -slo;
        }
        const uint8_t* kslab = sbase + (32 * sl) * RW::KROW + q * RW::KCHUNK;
        float cc[4][4];
        {
          uint32_t P[4][D / 8];
#pragma unroll
          for (int jt = 0; jt < 4; ++jt) {
            cc[jt][0] = neg_hi; cc[jt][1] = neg_hi; cc[jt][2] = neg_lo; cc[jt][3] = neg_lo;
            key_pairs<MODE, D>(kslab + (4 * g + jt) * RW::KROW, 0, P[jt]);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
            for (int jt = 0; jt < 4; ++jt) mma16816(cc[jt], wa[kk], P[jt][2 * kk], P[jt][2 * kk + 1]);
        }
#pragma unroll
        for (int jt = 0; jt < 4; ++jt) {
          const float* c = cc[jt];
          if (g == 0) {
            const int rel = static_cast<int>(tok0 - t_begin) + 8 * q + jt;
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const float shi_t = __fmul_rn(c[e2], cbmul);       // exact integer
              const float slo_t = __fmul_rn(c[2 + e2], cbmul);
              const float sf = __fadd_rn(__fmul_rn(2048.f, shi_t), slo_t);
              okeys[rel + 4 * e2] = order_key(__fadd_rn(__fmul_rn(sf, unit), beta));
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + slot);
    }
  }
  __syncthreads();
  if (*abort_flag && warp == NW && lane == 0) {
    for (int w = 0; w < NW; ++w) {
      const int issued = min(per_warp, max(0, ntiles - w * per_warp));
      for (int s2 = 0; s2 < SPW && s2 < issued; ++s2) {
        const int jl = ((issued - 1 - s2) / SPW) * SPW + s2;
        mbar_wait_bounded(full + w * SPW + s2, (jl / SPW) & 1, p.wait_limit);
      }
    }
  }
  __syncthreads();

  // ---------------- the chunk's top k: radix select on the order keys ----------------
  const int keff = min(K, n);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + L::SC_OFF);
  int* st = misc + 2;  // st[0] prefix, st[1] mask, st[2] remaining, st[3] count
  float* cs = p.cand_score + (u * p.S + split) * K;
  int32_t* ci = p.cand_idx + (u * p.S + split) * K;
  if (keff > 0) {
    radix_select(n, keff, [&](int i, uint32_t& key) { key = keys[i]; return true; }, hist, st);
    const uint32_t T = static_cast<uint32_t>(st[0]);
    const int need_eq = st[2];
    const int n_gt = keff - need_eq;
    if (tid == 0) st[3] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
      const uint32_t key = keys[i];
      if (key > T) {
        const int pos = atomicAdd(st + 3, 1);
        cs[pos] = key_to_score(key);
        ci[pos] = static_cast<int32_t>(t_begin + i);
      }
    }
    if (warp == 0) {  // ties at T: lowest indices first
      int taken = 0;
      for (int base = 0; base < n && taken < need_eq; base += 32) {
        const int i = base + lane;
        const bool eq = (i < n) && (keys[i] == T);
        const uint32_t bal = __ballot_sync(0xffffffffu, eq);
        const int before = __popc(bal & ((1u << lane) - 1u));
        if (eq && taken + before < need_eq) {
          cs[n_gt + taken + before] = key_to_score(T);
          ci[n_gt + taken + before] = static_cast<int32_t>(t_begin + i);
        }
        taken += __popc(bal);
      }
    }
  }
  for (int i = keff + tid; i < K; i += blockDim.x) {
    cs[i] = neg_inf();
    ci[i] = -1;
  }

  // ---------------- ticket: the last CTA of the unit merges ----------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(p.counters + u, 1u);
    const int last = (prev == static_cast<unsigned>(p.S - 1));
    if (last) atomicExch(p.counters + u, 0u);
    misc[1] = last;
    st[3] = 0;
  }
  __syncthreads();
  if (!misc[1]) return;
  __threadfence();
  // Candidates as unique composite keys (order key, ~index): larger is better.
  const int NC = p.S * K;
  uint32_t* khi = keys;                 // [NC] order keys, 0 for padding
  uint32_t* klo = keys + kTopkMaxCand;  // [NC] ~index
  const float* us = p.cand_score + u * p.S * K;
  const int32_t* ui = p.cand_idx + u * p.S * K;
  for (int i = tid; i < NC; i += blockDim.x) {
    const int32_t idx = __ldcg(ui + i);
    const bool ok = idx >= 0;
    khi[i] = ok ? order_key(__ldcg(us + i)) : 0u;
    klo[i] = ok ? 0xFFFFFFFFu - static_cast<uint32_t>(idx) : 0u;
    if (ok) atomicAdd(st + 3, 1);
  }
  __syncthreads();
  const int nvalid = st[3];
  const int kf = min(K, nvalid);
  uint32_t* whi = reinterpret_cast<uint32_t*>(smem);   // winners, in the (idle) stage area
  uint32_t* wlo = whi + kMaxTopk;
  if (kf > 0) {
    // order keys first, then the index among keys equal to the k-th order key
    radix_select(NC, kf, [&](int i, uint32_t& key) { key = khi[i]; return klo[i] != 0u; }, hist, st);
    const uint32_t Thi = static_cast<uint32_t>(st[0]);
    const int rem = st[2];
    __syncthreads();
    radix_select(NC, rem, [&](int i, uint32_t& key) { key = klo[i]; return klo[i] != 0u && khi[i] == Thi; },
                 hist, st);
    const uint32_t Tlo = static_cast<uint32_t>(st[0]);
    if (tid == 0) st[3] = 0;
    __syncthreads();
    for (int i = tid; i < NC; i += blockDim.x) {
      const uint32_t h = khi[i], l = klo[i];
      if (l != 0u && (h > Thi || (h == Thi && l >= Tlo))) {
        const int pos = atomicAdd(st + 3, 1);
        whi[pos] = h;
        wlo[pos] = l;
      }
    }
    __syncthreads();
    // rank sort of the kf winners (all composite keys differ)
    for (int i = tid; i < kf; i += blockDim.x) {
      const uint32_t h = whi[i], l = wlo[i];
      int rank = 0;
      for (int j = 0; j < kf; ++j) {
        const uint32_t hj = whi[j], lj = wlo[j];
        rank += (hj > h || (hj == h && lj > l)) ? 1 : 0;
      }
      const long long o = u * K + rank;
      p.idx_out[o] = static_cast<int32_t>(0xFFFFFFFFu - l);
      if (p.score_out) p.score_out[o] = key_to_score(h);
    }
  }
  for (int i = kf + tid; i < K; i += blockDim.x) {
    const long long o = u * K + i;
    p.idx_out[o] = -1;
    if (p.score_out) p.score_out[o] = neg_inf();
  }
}

template <int MODE, int D>
cudaError_t launch_t(const TopkParams& p, cudaStream_t s) {
  constexpr int smem = TopkSmem<MODE, D>::TOTAL;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(&topk_kernel<MODE, D>), smem);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.c.B) * p.c.Hkv * p.S;
  topk_kernel<MODE, D><<<static_cast<unsigned>(grid), NTHREADS, smem, s>>>(p);
  return cudaGetLastError();
}

// Resident CTAs per SM of one variant times the SM count, queried once per device.
template <int MODE, int D>
int resident_ctas_t() {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  if (cached[dev] > 0) return cached[dev];
  constexpr int smem = TopkSmem<MODE, D>::TOTAL;
  if (set_smem_once(reinterpret_cast<const void*>(&topk_kernel<MODE, D>), smem) != cudaSuccess) return 0;
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_kernel<MODE, D>, NTHREADS, smem) != cudaSuccess)
    return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cached[dev] = per_sm * sms;
  return cached[dev];
}

}  // namespace

int topk_resident_ctas(int mode, int D) {
  switch (mode) {
    case KVQ_MODE_INT4: return D == 128 ? resident_ctas_t<KVQ_MODE_INT4, 128>() : resident_ctas_t<KVQ_MODE_INT4, 64>();
    case KVQ_MODE_INT2: return D == 128 ? resident_ctas_t<KVQ_MODE_INT2, 128>() : resident_ctas_t<KVQ_MODE_INT2, 64>();
    case KVQ_MODE_INT1: return D == 128 ? resident_ctas_t<KVQ_MODE_INT1, 128>() : resident_ctas_t<KVQ_MODE_INT1, 64>();
    default: return 0;
  }
}

cudaError_t launch_topk(const TopkParams& p, int mode, cudaStream_t s) {
  const int D = p.c.D;
  switch (mode) {
    case KVQ_MODE_INT4: return D == 128 ? launch_t<KVQ_MODE_INT4, 128>(p, s) : launch_t<KVQ_MODE_INT4, 64>(p, s);
    case KVQ_MODE_INT2: return D == 128 ? launch_t<KVQ_MODE_INT2, 128>(p, s) : launch_t<KVQ_MODE_INT2, 64>(p, s);
    case KVQ_MODE_INT1: return D == 128 ? launch_t<KVQ_MODE_INT1, 128>(p, s) : launch_t<KVQ_MODE_INT1, 64>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
