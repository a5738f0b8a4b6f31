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
//   beta = fp32(Z) * 2^(f-40), Z = sum_d rint(fp32(qs_d z_d) * 2^(40-f)) (exact),
// with f the exponent of the group's largest |qs_d z_d|.  Both sums are exact
// integers, so the warp derives beta with shuffles, in any order, when it
// derives the group's weights.
// The dot product runs on tensor cores with the keys as the A operand (rows =
// tokens) in the subnormal f16 encoding of the attention (code c at mantissa
// bits k.., read as c 2^k 2^-24 with the pair's factor 2^k), and W as the B
// operand split into three integer parts, W = 2^14 h + 2^7 m + l with
// |h| <= 128 and |m|, |l| <= 64, each times 2^(SLF - k) (SLF the largest pair
// factor) an exact f16 value in columns 0, 1 and 2.  Every product is an
// integer times 2^(SLF-24) and every partial sum stays below 2^24 such units,
// so the fp32 accumulation is exact in any order; 2^14 S_h and 2^7 S_m + S_l
// are then exact fp32 values and one correctly rounded add gives fp32(S_t).
// Each warp derives W for a key group cooperatively (two key pairs per lane)
// and stages the parts in shared memory in the B fragments' order.
//
// One launch: B*Hkv*S CTAs, with S chosen on the host to balance waves against
// the merge.  Each CTA scores one chunk (bulk-copied tiles on an mbarrier ring,
// as in attention; a pre-scored launch reads the attention's scores instead)
// into 32-bit order keys and selects its top k by (score desc, index asc),
// as unique composite keys (order key, ~index) in descending order.
//
// Selection of a chunk's top k (k <= 128):
//  * a lower bound T0: the keys fall into 128 strided segments (i mod 128);
//    the k-th largest segment maximum is at most the k-th largest key, since
//    k segment maxima are k distinct keys at least that large;
//  * every warp collects the keys >= T0 of its share into its own region
//    (ballot + population count, no shared counter);
//  * the candidates (about 100 when the keys are spread out) are ranked by
//    counting, each against all, and land at their rank.
// More candidates than one per thread go through warp bitonic sorts of 128
// and a merge-path tree; more than 1024, or k > 128, through a radix
// selection of the k-th key (select_kth).
//
// Merge of a unit's S sorted lists (k <= 128): warps merge pairs of lists in
// registers (a bitonic half-cleaner and merge network), level by level; larger
// k takes a merge-path tree.
// With S <= 8 and k <= 128 the S CTAs of a unit form one thread-block cluster,
// the lists stay in shared memory and the first CTA reads them through
// distributed shared memory; otherwise every CTA writes its list to the
// workspace and the last CTA to arrive (an atomic ticket) merges.
#include <algorithm>

#include "kvq_modes.cuh"

namespace kvq {
namespace {

constexpr int NW = 8;                  // warps per CTA; each streams and scores its own tiles
constexpr int NTHREADS = NW * 32;
constexpr int kGather = 64;            // bin size below which select_kth ranks keys directly
constexpr int kSpwMax = 4;             // stage slots per warp, at most
constexpr int kRegion = 128;           // candidates per warp region
constexpr int kClusterMax = 8;         // splits that merge as one cluster, at most

// Post-scoring scratch at the start of shared memory (over the idle stage
// ring): packed candidates, the warps' candidate regions (later the sort
// lists of the merge-path fallback), select_kth's histograms.  A merge's S x k
// list entries (<= kTopkMaxCand) reuse it from offset 0.
constexpr int kPackOff = 0;                                 // [NW * kRegion + 2] u64
constexpr int kRegOff = kPackOff + (NW * kRegion + 2) * 8;  // [NW][kRegion] u64
constexpr int kListOff = kRegOff;                           // [2][NW][k <= 128] u64
constexpr int kHistOff = kListOff + 2 * NW * 128 * 8;       // [NW][256] u32 (also the 256 segment maxima)
constexpr int kScratch = kHistOff + NW * 256 * 4;
static_assert(kRegOff % 16 == 0 && kHistOff % 16 == 0 && kScratch % 16 == 0, "16-byte aligned scratch");
static_assert(kTopkMaxCand * 8 <= kScratch, "a merge's list entries fit the scratch");
static_assert(kMaxTopk * 8 <= kRegOff, "select_kth's winners fit below the regions");

template <int MODE, int D>
struct TopkTile {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  static constexpr int TT = M::TT;
  static constexpr int KPLANE = TT * RW::KROW;
  static constexpr int KSZ_OFF = KPLANE;                      // only the upper/only plane is read
  static constexpr int KSZ_BYTES = (TT / 32) * 2 * D * 4;
  static constexpr int SLOT = KSZ_OFF + KSZ_BYTES;
  static_assert(SLOT % 16 == 0, "slots must stay 16-byte aligned");
};

// Shared-memory layout of one launch: the stage ring (or the scratch, if
// larger), then the fixed parts, then the chunk's order keys (later the
// CTA's own sorted list).
struct TopkLayout {
  int qs, wb, list, red, bar, misc, sc, total;
};

__host__ __device__ constexpr long long lmax(long long a, long long b) { return a > b ? a : b; }

template <int MODE, int D>
__host__ __device__ inline TopkLayout topk_layout(bool pre, int spw, long long chunk, int k, int S) {
  const int ring = pre ? kScratch : static_cast<int>(lmax(NW * spw * TopkTile<MODE, D>::SLOT, kScratch));
  TopkLayout l;
  l.qs = ring;                                   // qs[D]
  l.wb = l.qs + D * 4;                           // per warp: weight parts [3][D/2] half2 in pair order
  l.list = l.wb + NW * 3 * (D / 2) * 4;          // gathered keys [kGather]
  l.red = l.list + kGather * 4;                  // per-warp values [2 NW]
  l.bar = l.red + 2 * NW * 4;                    // mbarriers [NW][kSpwMax]
  l.misc = l.bar + NW * kSpwMax * 8;             // [0] abort, [1] last, [2..6] select state
  l.sc = l.misc + 64;                            // order keys [chunk], then the sorted list [k] u64
  long long sc = lmax(chunk * 4, static_cast<long long>(k) * 8);
  if (k > 128) sc = lmax(sc, 2LL * S * k * 8);   // the merge-path tree's two buffers (k > 128)
  l.total = l.sc + static_cast<int>((sc + 15) / 16) * 16;
  return l;
}

__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t b = __float_as_uint(__fadd_rn(s, 0.0f));  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_to_score(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(b);
}

// Unique composite key of a candidate: order key above, ~index below (larger is
// better; 0 marks padding).
__device__ __forceinline__ uint64_t composite(uint32_t okey, uint32_t idx) {
  return (static_cast<uint64_t>(okey) << 32) | (0xFFFFFFFFu - idx);
}

__device__ __forceinline__ int32_t composite_index(uint64_t key) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

__device__ __forceinline__ float pow2f(int e) {  // 2^e for -126 <= e <= 127
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// Sorts the warp's 128 keys into descending order.  Key x = 32 r + lane sits
// in v[r]; the bitonic network pairs x with x ^ j (a shuffle for j < 32, a
// register swap otherwise).
template <typename T>
__device__ __forceinline__ void warp_sort128_desc(T (&v)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 128; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < 32) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int x = 32 * r + lane;
          const T o = __shfl_xor_sync(0xffffffffu, v[r], j);
          const bool desc = (x & k) == 0, lower = (x & j) == 0;
          const T hi = v[r] > o ? v[r] : o, lo = v[r] > o ? o : v[r];
          v[r] = (lower == desc) ? hi : lo;
        }
      } else {
        const int jr = j >> 5;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (r & jr) continue;
          const int x = 32 * r + lane;
          const bool desc = (x & k) == 0;
          const T a = v[r], b = v[r | jr];
          const T hi = a > b ? a : b, lo = a > b ? b : a;
          v[r] = desc ? hi : lo;
          v[r | jr] = desc ? lo : hi;
        }
      }
    }
  }
}

// Merge-path tree: nl lists of len keys each, in descending order, at src
// (padding 0), merged pairwise per level, each output keeping the top len of
// its two inputs (an odd list moves up unchanged).  Every thread of the block
// calls it; dst is scratch of the same size.  Returns the final list.
__device__ uint64_t* merge_tree(uint64_t* src, uint64_t* dst, int nl, int len) {
  while (nl > 1) {
    const int np = nl / 2;
    for (int t = threadIdx.x; t < np * len; t += blockDim.x) {
      const int j = t / len, i = t % len;               // output list j, position i
      const uint64_t* A = src + static_cast<long long>(2 * j) * len;
      const uint64_t* B = A + len;
      int lo = 0, hi = i;                               // elements of A among the top i
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (A[mid] > B[i - mid - 1]) lo = mid + 1;
        else hi = mid;
      }
      const uint64_t va = A[lo], vb = B[i - lo];
      dst[static_cast<long long>(j) * len + i] = va > vb ? va : vb;
    }
    if (nl & 1)
      for (int i = threadIdx.x; i < len; i += blockDim.x)
        dst[static_cast<long long>(np) * len + i] = src[static_cast<long long>(nl - 1) * len + i];
    __syncthreads();
    nl = np + (nl & 1);
    uint64_t* tmp = src;
    src = dst;
    dst = tmp;
  }
  return src;
}

// Block-wide selection of the kth largest key among the i < n for which
// take(i, key) holds (1 <= kth <= number taken).  On return st[0] = T and
// st[2] = how many of the taken keys equal to T belong to the kth largest.
// Every thread of the block calls it.  hist[NW][256] (one histogram per warp,
// so that keys crowding into a few bins do not serialize across warps),
// list[kGather], red[2 NW] and st[0..4] are shared memory.
template <typename F>
__device__ void select_kth(int n, int kth, F take, uint32_t* hist, uint32_t* list, uint32_t* red, int* st) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = (blockDim.x + 31) / 32;
  // ---- smallest and largest taken key ----
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = tid; i < n; i += blockDim.x) {
    uint32_t key;
    if (take(i, key)) {
      lo = min(lo, key);
      hi = max(hi, key);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    red[2 * warp] = lo;
    red[2 * warp + 1] = hi;
  }
  for (int i = tid; i < NW * 256; i += blockDim.x) hist[i] = 0u;
  if (tid == 0) st[4] = 0;
  __syncthreads();
  lo = red[0];
  hi = red[1];
  for (int w = 1; w < nw; ++w) {
    lo = min(lo, red[2 * w]);
    hi = max(hi, red[2 * w + 1]);
  }
  if (lo == hi) {  // every taken key is equal
    __syncthreads();
    if (tid == 0) {
      st[0] = static_cast<int>(lo);
      st[2] = kth;
    }
    __syncthreads();
    return;
  }
  const int hb = 31 - __clz(lo ^ hi);                  // highest bit where taken keys differ
  uint32_t mask = (hb == 31) ? 0u : ~((2u << hb) - 1u);
  uint32_t prefix = lo & mask;
  int shift = max(hb - 7, 0);
  int remaining = kth;
  while (true) {
    // ---- histogram of the 8 bits at `shift` among keys matching the prefix ----
    uint32_t* hw = hist + warp * 256;
    for (int i = tid; i < n; i += blockDim.x) {
      uint32_t key;
      if (take(i, key) && (key & mask) == prefix) atomicAdd(hw + ((key >> shift) & 255u), 1u);
    }
    __syncthreads();
    for (int bn = tid; bn < 256; bn += blockDim.x) {   // per-warp histograms -> hist[0]
      uint32_t c = hist[bn];
      for (int w = 1; w < nw; ++w) c += hist[w * 256 + bn];
      hist[bn] = c;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending); a warp scan gives the
      // count above each lane, and the lane holding the kth key picks its digit
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
      const uint32_t rem = static_cast<uint32_t>(remaining);
      if (excl < rem && rem <= inc) {
        uint32_t cum = excl;
        int digit = 255 - 8 * lane - 7;
        uint32_t bin = c[7];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (cum + c[k] >= rem) {
            digit = 255 - 8 * lane - k;
            bin = c[k];
            break;
          }
          cum += c[k];
        }
        st[0] = digit;
        st[1] = static_cast<int>(rem - cum);
        st[3] = static_cast<int>(bin);
      }
    }
    __syncthreads();
    const uint32_t digit = static_cast<uint32_t>(st[0]);
    remaining = st[1];
    const int bin = st[3];
    prefix |= digit << shift;
    mask |= 255u << shift;
    for (int i = tid; i < NW * 256; i += blockDim.x) hist[i] = 0u;
    if (shift == 0) {  // the key is fully determined
      __syncthreads();
      if (tid == 0) {
        st[0] = static_cast<int>(prefix);
        st[2] = remaining;
      }
      __syncthreads();
      return;
    }
    if (bin <= kGather) {
      // ---- gather the bin's keys and rank them ----
      for (int i = tid; i < n; i += blockDim.x) {
        uint32_t key;
        if (take(i, key) && (key & mask) == prefix) list[atomicAdd(st + 4, 1)] = key;
      }
      __syncthreads();
      if (warp == 0) {
        for (int j = lane; j < bin; j += 32) {
          const uint32_t kj = list[j];
          int above = 0, eq = 0;
          for (int i = 0; i < bin; ++i) {
            above += list[i] > kj;
            eq += list[i] == kj;
          }
          if (above < remaining && remaining <= above + eq) {  // every such lane writes the same
            st[0] = static_cast<int>(kj);
            st[2] = remaining - above;
          }
        }
      }
      __syncthreads();
      return;
    }
    shift = max(shift - 8, 0);
    __syncthreads();
  }
}

// Top 32 KR of two sorted lists A and B (composite keys, 0 pads) in one warp.
// a[r] holds A's position 32 r + lane (descending); b[r] holds position
// 32 r + lane of B in ascending order, i.e. B's position 32 KR - 1 - (32 r +
// lane), so that A then b is a bitonic sequence.  The half-cleaner keeps the
// larger of each pair, which are the top 32 KR as a bitonic sequence, and the
// bitonic merge network sorts them into a[] in descending order.
template <int KR>
__device__ __forceinline__ void warp_merge_top(uint64_t (&a)[KR], const uint64_t (&b)[KR]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < KR; ++r) a[r] = a[r] > b[r] ? a[r] : b[r];
#pragma unroll
  for (int jr = KR / 2; jr > 0; jr >>= 1) {
#pragma unroll
    for (int r = 0; r < KR; ++r) {
      if (r & jr) continue;
      const uint64_t x = a[r], y = a[r | jr];
      a[r] = x > y ? x : y;
      a[r | jr] = x > y ? y : x;
    }
  }
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
#pragma unroll
    for (int r = 0; r < KR; ++r) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, a[r], j);
      const bool lower = (lane & j) == 0;
      a[r] = (lower == (a[r] > o)) ? a[r] : o;
    }
  }
}

// The top K (<= 32 KR) of S sorted lists (descending, 0 pads) of K composite
// keys at M[S][K]: pairs of lists merge in warps, level by level, in place
// (the pair (i, i + st) into list i).  Every thread of the block calls it;
// the result is list 0.
template <int KR>
__device__ void warp_merge_tree(uint64_t* M, int S, int K) {
  const int lane = threadIdx.x & 31, warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 5, 0);
  constexpr int N = 32 * KR;
  for (int st = 1; st < S; st *= 2) {
    for (int i = 2 * st * warp; i + st < S; i += 2 * st * NW) {
      uint64_t* A = M + static_cast<long long>(i) * K;
      const uint64_t* B = M + static_cast<long long>(i + st) * K;
      uint64_t a[KR], b[KR];
#pragma unroll
      for (int r = 0; r < KR; ++r) {
        const int x = 32 * r + lane, y = N - 1 - x;
        a[r] = x < K ? A[x] : 0ull;
        b[r] = y < K ? B[y] : 0ull;
      }
      warp_merge_top<KR>(a, b);
      __syncwarp();
#pragma unroll
      for (int r = 0; r < KR; ++r) {
        const int x = 32 * r + lane;
        if (x < K) A[x] = a[r];
      }
    }
    __syncthreads();
  }
}

// PRE: the attention's scoring pass wrote the finished scores to p.pre;
// otherwise the kernel streams and scores the key planes itself.
template <int MODE, int D, bool PRE>
__global__ void __launch_bounds__(NTHREADS, 2) topk_kernel(TopkParams p) {
  using M = Mode<MODE>;
  using RW = Rows<MODE, D>;
  using TL = TopkTile<MODE, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  // the warp index broadcast from lane 0: a warp-uniform value for the compiler
  const int tid = threadIdx.x, lane = tid % 32, warp = __shfl_sync(0xffffffffu, tid / 32, 0);
  const int g = lane >> 2, q = lane & 3;
  const long long u = blockIdx.x / p.S;
  const int split = blockIdx.x % p.S;
  const int b = static_cast<int>(u / p.c.Hkv), kvh = static_cast<int>(u % p.c.Hkv);
  const int G = p.c.G;
  const TopkLayout L = topk_layout<MODE, D>(PRE, p.spw, p.chunk, p.k, p.S);
  // a ragged cache splits each sequence's own length over the S splits, in
  // multiples of the plan's alignment (the length is broadcast from lane 0 so
  // that the copy operands below are warp-uniform values for the compiler)
  const long long lq_b = __shfl_sync(0xffffffffu, seq_lq(p.c, b), 0);
  const long long chunk =
      p.c.ragged ? ((lq_b + p.S - 1) / p.S + p.align - 1) / p.align * p.align : p.chunk;
  const long long t_begin = static_cast<long long>(split) * chunk;
  const long long t_end = min(lq_b, t_begin + chunk);
  const int n = static_cast<int>(max(0LL, t_end - t_begin));
  const int ntiles = PRE ? 0 : (n + M::TT - 1) / M::TT;   // a pre-scored launch streams nothing
  const int per_warp = (ntiles + NW - 1) / NW;
  const int K = p.k;
  const int spw = p.spw;

  uint32_t* okeys = reinterpret_cast<uint32_t*>(smem + L.sc);
  float* qs = reinterpret_cast<float*>(smem + L.qs);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kHistOff);
  uint32_t* list = reinterpret_cast<uint32_t*>(smem + L.list);
  uint32_t* red = reinterpret_cast<uint32_t*>(smem + L.red);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  int* misc = reinterpret_cast<int*>(smem + L.misc);   // [0] abort, [1] last, [2..6] select state
  const long long u_tok = u * p.c.C;
  // this warp's tiles: a contiguous run of the chunk
  const int my_first = warp * per_warp;
  const int my_tiles = max(0, min(per_warp, ntiles - my_first));
  // Each warp streams its own tiles: one elected lane puts tile j into slot
  // j % spw of the warp's ring with 1-D bulk copies that complete on the slot's
  // mbarrier.  The whole (converged) warp computes the copy operands from
  // warp-uniform values only.
  const uint64_t pol = __shfl_sync(0xffffffffu, policy_evict_first(), 0);
  auto issue = [&](int j) {
    const int slot = warp * spw + (j % spw);
    const int rel = (my_first + j) * M::TT;                 // chunk-relative first token
    const int nt = min(M::TT, n - rel);
    const long long t0 = t_begin + rel;
    // a tile loads key scales only when it starts a key group (or the run)
    const bool new_grp = (j == 0) || (M::TT > G) || (t0 % G == 0);
    const uint32_t kb = nt * RW::KROW;
    const uint32_t kszb = new_grp ? static_cast<uint32_t>((nt + G - 1) / G) * 2 * D * 4 : 0u;
    uint8_t* sbase = smem + slot * TL::SLOT;
    uint64_t* bar = full + warp * kSpwMax + (j % spw);
    if (elect_one()) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(bar, kb + kszb);
      bulk_g2s(sbase, p.c.kplane[0] + (u_tok + t0) * RW::KROW, kb, bar, pol);
      if (new_grp)
        bulk_g2s(sbase + TL::KSZ_OFF, p.c.ksz + (u * (p.c.C / G) + t0 / G) * 2 * D, kszb, bar, pol);
    }
    __syncwarp();
  };
  int issued = 0, consumed = 0;
  if (tid == 0) misc[0] = 0;
  volatile int* abort_flag = misc;
  if constexpr (PRE) {
    __syncthreads();
    // the attention's scoring pass wrote the finished scores: n is a multiple
    // of 128 tokens, so each thread takes float4 runs, all loads in flight
    static_assert(kTopkMaxChunk % (4 * NTHREADS) == 0, "whole float4 runs per thread");
    const float4* src = reinterpret_cast<const float4*>(p.pre + u * p.c.C + t_begin);
    constexpr int kRuns = kTopkMaxChunk / (4 * NTHREADS);
    float4 v[kRuns];
#pragma unroll
    for (int r = 0; r < kRuns; ++r) {
      const int i4 = tid + r * NTHREADS;
      if (4 * i4 < n) v[r] = __ldcg(src + i4);
    }
#pragma unroll
    for (int r = 0; r < kRuns; ++r) {
      const int i4 = tid + r * NTHREADS;
      if (4 * i4 < n) {
        okeys[4 * i4] = order_key(v[r].x);
        okeys[4 * i4 + 1] = order_key(v[r].y);
        okeys[4 * i4 + 2] = order_key(v[r].z);
        okeys[4 * i4 + 3] = order_key(v[r].w);
      }
    }
  } else {
    // the first heads' query values are loaded before the first copies issue
    constexpr int kQPre = 8;
    static_assert(D <= NTHREADS, "one query channel per thread");
    uint16_t qpre[kQPre];
    const long long qoff = static_cast<long long>(b) * p.q_bstride + static_cast<long long>(kvh) * p.HG * D + tid;
#pragma unroll
    for (int hh = 0; hh < kQPre; ++hh) qpre[hh] = (tid < D && hh < p.HG) ? p.q[qoff + hh * D] : 0;
    if (lane == 0) {
      for (int s2 = 0; s2 < spw; ++s2) mbar_init(full + warp * kSpwMax + s2, 1);
      fence_mbar_init();
    }
    __syncwarp();
    for (int j = 0; j < min(spw, my_tiles); ++j) issue(j);
    issued = min(spw, my_tiles);
    // summed query (ascending head order, fp32) while the first tiles load
    if (tid < D) {
      float acc = 0.f;
#pragma unroll
      for (int hh = 0; hh < kQPre; ++hh)
        if (hh < p.HG) acc = __fadd_rn(acc, bf16_to_f32(qpre[hh]));
      for (int hh = kQPre; hh < p.HG; ++hh) acc = __fadd_rn(acc, bf16_to_f32(p.q[qoff + hh * D]));
      qs[tid] = acc;
    }
    __syncthreads();

    // Lane (g, q) reads column g of the weight parts (zero past column 2) from
    // the warp's staging area at each k-step.
    float unit = 1.f, beta = 0.f;
    long long cur_grp = -1;
    const float smul = static_cast<float>(M::MULT) * (MODE == KVQ_MODE_INT1 ? p.smul : 1.0f);
    uint32_t* whs = reinterpret_cast<uint32_t*>(smem + L.wb) + warp * 3 * (D / 2);   // [3][D/2]
    const uint2* wsrc = reinterpret_cast<const uint2*>(whs + min(g, 2) * (D / 2) + q * (D / 8));
    constexpr int NIT = D / 64;                  // key pairs per lane in the derivation
    constexpr int SLF = score_log2fac_max<MODE, D>();
    constexpr float INV = static_cast<float>(1 << (24 - SLF));
    constexpr float kRnd = 12582912.0f;          // 1.5 * 2^23: x + kRnd - kRnd = rint(x) for |x| < 2^22
    const int pp = lane % (D / 8);
    const int c0 = kx_chan<MODE, D>(pp, 0), c1 = kx_chan<MODE, D>(pp, 1);
    const float fsh = pow2f(SLF - ks_log2fac<MODE, D>(pp));
    for (int j = 0; j < my_tiles; ++j) {
      const int ti = my_first + j;
      const int slot = warp * spw + (j % spw);
      if (!mbar_wait_bounded(full + warp * kSpwMax + (j % spw), (j / spw) & 1, p.wait_limit)) {
        record_status(p.status, KVQ_ERR_DEVICE_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      const long long t0 = t_begin + static_cast<long long>(ti) * M::TT;
      const int nt = static_cast<int>(min(static_cast<long long>(M::TT), t_end - t0));
      const long long g_first = t0 / G;
      const uint8_t* sbase = smem + slot * TL::SLOT;
      const float* ksz = reinterpret_cast<const float*>(sbase + TL::KSZ_OFF);
      for (int sl = 0; sl < nt / 32; ++sl) {
        const long long tok0 = t0 + 32 * sl;
        const long long grp = tok0 / G;
        if (grp != cur_grp) {
          // ---- W of this group: lane l derives key pairs l and l + 32 ----
          // w_d = fp32(qs_d * fp32(MULT s_d)); e with max|w| < 2^e (floored
          // at -100); W_d = rint(w_d 2^(21-e)); h = rint(W 2^-14), r = W - 2^14 h,
          // m = rint(r 2^-7), l = r - 2^7 m, all exact fp32 steps.
          cur_grp = grp;
          __syncwarp();                          // every lane is done with the previous group's parts
          const float* ks = ksz + (grp - g_first) * 2 * D;
          const float* kz = ks + D;
          float wv[2 * NIT], zp[2 * NIT];
          float mxw = 0.f;
#pragma unroll
          for (int i = 0; i < NIT; ++i) {
            const int base = ((lane + 32 * i) / (D / 8)) * (D / 4);
            const int d0 = base + c0, d1 = base + c1;
            wv[2 * i] = __fmul_rn(qs[d0], __fmul_rn(ks[d0], smul));
            wv[2 * i + 1] = __fmul_rn(qs[d1], __fmul_rn(ks[d1], smul));
            // zero points as the mode reads them: fp32(z + zshift * s)
            zp[2 * i] = __fmul_rn(qs[d0], fmaf(p.zshift, ks[d0], kz[d0]));
            zp[2 * i + 1] = __fmul_rn(qs[d1], fmaf(p.zshift, ks[d1], kz[d1]));
            mxw = fmaxf(mxw, fmaxf(fabsf(wv[2 * i]), fabsf(wv[2 * i + 1])));
          }
          mxw = warp_max_nonneg(mxw);
          beta = zero_term_warp<2 * NIT>(zp);
          int e = 0;
          if (mxw > 0.f) frexpf(mxw, &e);
          e = max(e, -100);
          const float up = pow2f(21 - e);
          unit = pow2f(e - 21);
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
#pragma unroll
            for (int k3 = 0; k3 < 3; ++k3) whs[k3 * (D / 2) + lane + 32 * i] = pack_half2(v[0][k3], v[1][k3]);
          }
          __syncwarp();
        }
        const uint8_t* kslab = sbase + (32 * sl) * RW::KROW + q * RW::KCHUNK;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          uint32_t PA[D / 8], PB[D / 8];
          key_pairs_s<MODE, D>(kslab + (16 * s + g) * RW::KROW, 0, PA);
          key_pairs_s<MODE, D>(kslab + (16 * s + g + 8) * RW::KROW, 0, PB);
          // two independent chains over the k-steps (every partial sum is exact)
          float cc[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < D / 16; kk += 2) {
            const uint32_t a[4] = {PA[2 * kk], PB[2 * kk], PA[2 * kk + 1], PB[2 * kk + 1]};
            const uint32_t a2[4] = {PA[2 * kk + 2], PB[2 * kk + 2], PA[2 * kk + 3], PB[2 * kk + 3]};
            const uint2 w0 = wsrc[kk], w1 = wsrc[kk + 1];
            mma16816(cc, a, g < 3 ? w0.x : 0u, g < 3 ? w0.y : 0u);
            mma16816(c2, a2, g < 3 ? w1.x : 0u, g < 3 ? w1.y : 0u);
          }
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) cc[e2] += c2[e2];
          // columns 0, 1 (lanes q = 0) hold the h and m part sums, column 2
          // (lanes q = 1) the l part sum
          const float lA = __shfl_down_sync(0xffffffffu, cc[0], 1);
          const float lB = __shfl_down_sync(0xffffffffu, cc[2], 1);
          if (q == 0) {
            const int rel = static_cast<int>(tok0 - t_begin) + 16 * s + g;
            const float SA = __fadd_rn(__fmul_rn(cc[0], INV * 16384.f), __fmaf_rn(cc[1], INV * 128.f, __fmul_rn(lA, INV)));
            const float SB = __fadd_rn(__fmul_rn(cc[2], INV * 16384.f), __fmaf_rn(cc[3], INV * 128.f, __fmul_rn(lB, INV)));
            okeys[rel] = order_key(__fadd_rn(__fmul_rn(SA, unit), beta));
            okeys[rel + 8] = order_key(__fadd_rn(__fmul_rn(SB, unit), beta));
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
        mbar_wait_bounded(full + warp * kSpwMax + (jj % spw), (jj / spw) & 1, p.wait_limit);
    }
    __syncwarp();
  }
  __syncthreads();

  // ---------------- the chunk's top k, sorted, into `mine` ----------------
  const int keff = min(K, n);
  int* st = misc + 2;  // st[0] T, st[1] remaining, st[2] ties taken, st[3] bin / count, st[4] gather count
  uint64_t* mine = reinterpret_cast<uint64_t*>(smem + L.sc);   // [K] over the order keys, once they are read
  uint64_t* pk = reinterpret_cast<uint64_t*>(smem + kPackOff);
  bool selected = keff == 0;
  if (keff > 0 && K <= 128) {
    // ---- lower bound T0 (all keys when the chunk is short) ----
    uint32_t T0 = 0u;
    if (n > 2 * 128) {
      uint32_t* segmax = hist;                              // [256]
      uint32_t mx = 0u;
      for (int i = tid; i < n; i += NTHREADS) mx = max(mx, okeys[i]);   // segment tid % 128
      segmax[tid] = mx;
      __syncthreads();
      if (warp == 0) {
        uint32_t v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int sg = 32 * r + lane;
          v[r] = max(segmax[sg], segmax[sg + 128]);
        }
        warp_sort128_desc(v);
#pragma unroll
        for (int r = 0; r < 4; ++r)
          if (32 * r + lane == keff - 1) st[0] = static_cast<int>(v[r]);
      }
      __syncthreads();
      T0 = static_cast<uint32_t>(st[0]);
    }
    // ---- each warp's keys >= T0 into its region ----
    uint64_t* reg = reinterpret_cast<uint64_t*>(smem + kRegOff) + warp * kRegion;
    int cnt = 0;
    for (int base = warp * 32; base < n; base += NTHREADS) {   // the same trip count in every lane
      const int i = base + lane;
      const uint32_t key = (i < n) ? okeys[i] : 0u;
      const bool take = (i < n) && key >= T0;
      const uint32_t bal = __ballot_sync(0xffffffffu, take);
      const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
      if (take && pos < kRegion) reg[pos] = composite(key, static_cast<uint32_t>(t_begin + i));
      cnt += __popc(bal);
    }
    if (lane == 0) red[warp] = static_cast<uint32_t>(cnt);
    __syncthreads();
    int total = 0, off = 0;
    bool over = false;
    for (int w = 0; w < NW; ++w) {
      const int c = static_cast<int>(red[w]);
      off += (w < warp) ? c : 0;
      total += c;
      over = over || c > kRegion;
    }
    if (!over && total <= NW * kRegion) {
      // ---- pack the regions ----
      for (int j = lane; j < cnt; j += 32) pk[off + j] = reg[j];
      if (tid == 0) {
        pk[total] = 0ull;
        pk[total + 1] = 0ull;
      }
      __syncthreads();
      if (total <= NTHREADS) {
        // ---- rank by counting: every composite key is unique ----
        if (tid < total) {
          const uint64_t x = pk[tid];
          const ulonglong2* p2 = reinterpret_cast<const ulonglong2*>(pk);
          int rank = 0;
          for (int j = 0; j < (total + 1) / 2; ++j) {
            const ulonglong2 y = p2[j];
            rank += (y.x > x) + (y.y > x);
          }
          if (rank < keff) mine[rank] = x;
        }
      } else {
        // ---- warp sorts of 128 and a merge-path tree ----
        const int nl = (total + 127) / 128;
        uint64_t* la = reinterpret_cast<uint64_t*>(smem + kListOff);   // [nl][K]
        uint64_t* lb = la + NW * K;
        if (warp < nl) {
          uint64_t v[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int i = warp * 128 + 32 * r + lane;
            v[r] = (i < total) ? pk[i] : 0ull;
          }
          warp_sort128_desc(v);
#pragma unroll
          for (int r = 0; r < 4; ++r)
            if (32 * r + lane < K) la[warp * K + 32 * r + lane] = v[r];
        }
        __syncthreads();
        const uint64_t* top = merge_tree(la, lb, nl, K);
        for (int i = tid; i < keff; i += NTHREADS) mine[i] = top[i];
      }
      selected = true;
    }
  }
  if (!selected) {
    // ---- radix selection of the k-th key, then the winners ranked ----
    select_kth(n, keff, [&](int i, uint32_t& key) { key = okeys[i]; return true; }, hist, list, red, st);
    const uint32_t T = static_cast<uint32_t>(st[0]);
    const int need_eq = st[2];
    const int n_gt = keff - need_eq;
    __syncthreads();
    if (tid == 0) st[3] = 0;
    __syncthreads();
    // The winners go to shared memory as composite keys (order key, ~index):
    // keys above T anywhere in [0, n_gt), then the need_eq ties at T with the
    // lowest indices (each warp scans a contiguous segment, counts its ties,
    // and places its own after those of the warps before it).
    uint64_t* wk = pk;   // [keff]
    const int seg = (n + NW - 1) / NW;
    const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
    int myeq = 0;
    for (int base = s0; base < s1; base += 32) {
      const int i = base + lane;
      const uint32_t key = (i < s1) ? okeys[i] : 0u;
      const bool sel = (i < s1) && key > T;
      const uint32_t bal = __ballot_sync(0xffffffffu, sel);
      myeq += __popc(__ballot_sync(0xffffffffu, (i < s1) && key == T));
      int pbase = 0;
      if (lane == 0 && bal) pbase = atomicAdd(st + 3, __popc(bal));
      pbase = __shfl_sync(0xffffffffu, pbase, 0);
      if (sel) {
        const int pos = pbase + __popc(bal & ((1u << lane) - 1u));
        wk[pos] = composite(key, static_cast<uint32_t>(t_begin + i));
      }
    }
    if (lane == 0) red[warp] = static_cast<uint32_t>(myeq);
    __syncthreads();
    int taken = 0;
    for (int w = 0; w < warp; ++w) taken += static_cast<int>(red[w]);
    for (int base = s0; base < s1 && taken < need_eq; base += 32) {
      const int i = base + lane;
      const bool eq = (i < s1) && (okeys[i] == T);
      const uint32_t bal = __ballot_sync(0xffffffffu, eq);
      const int before = __popc(bal & ((1u << lane) - 1u));
      if (eq && taken + before < need_eq) wk[n_gt + taken + before] = composite(T, static_cast<uint32_t>(t_begin + i));
      taken += __popc(bal);
    }
    __syncthreads();
    // the winners in descending order (composite keys are unique): four lanes
    // count the larger keys of one winner
    for (int e0 = tid >> 2; e0 < ((keff + NW * 8 - 1) / (NW * 8)) * (NW * 8); e0 += NW * 8) {
      const int e = min(e0, keff - 1);
      const uint64_t key = wk[e];
      int rank = 0;
      for (int j = (tid & 3); j < keff; j += 4) rank += wk[j] > key;
      rank += __shfl_xor_sync(0xffffffffu, rank, 1);
      rank += __shfl_xor_sync(0xffffffffu, rank, 2);
      if ((tid & 3) == 0 && e0 < keff) mine[rank] = key;
    }
  }
  for (int i = keff + tid; i < K; i += NTHREADS) mine[i] = 0ull;
  __syncthreads();

  // ---------------- the unit's top k ----------------
  if (p.S == 1) {
    for (int i = tid; i < K; i += NTHREADS) {
      const uint64_t x = mine[i];
      const long long o = u * K + i;
      p.idx_out[o] = x ? composite_index(x) : -1;
      if (p.score_out) p.score_out[o] = x ? key_to_score(static_cast<uint32_t>(x >> 32)) : neg_inf();
    }
    return;
  }
  // the unit's S lists: in the scratch for k <= 128, else in the order-key area
  // (free once this CTA's list left it) with room for the merge-path tree
  uint64_t* mb = reinterpret_cast<uint64_t*>(K <= 128 ? smem : smem + L.sc);   // [S][K]
  if (p.cluster) {
    // The lists stay in shared memory; the unit's first CTA copies them
    // through distributed shared memory.  The second barrier keeps every
    // CTA's list alive until the copy is done.
    cluster_sync();
    const bool leader = cluster_rank() == 0;
    if (leader) {
      for (int c = tid; c < p.S * K; c += NTHREADS)
        mb[c] = ld_dsmem_u64(dsmem_addr(mine + c % K, static_cast<uint32_t>(c / K)));
    }
    __syncthreads();
    cluster_sync();
    if (!leader) return;
  } else {
    float* cs = p.cand_score + (u * p.S + split) * K;
    int32_t* ci = p.cand_idx + (u * p.S + split) * K;
    for (int i = tid; i < K; i += NTHREADS) {
      const uint64_t x = mine[i];
      cs[i] = x ? key_to_score(static_cast<uint32_t>(x >> 32)) : neg_inf();
      ci[i] = x ? composite_index(x) : -1;
    }
    // ticket: the last CTA of the unit merges
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const unsigned prev = atomicAdd(p.counters + u, 1u);
      const int last = (prev == static_cast<unsigned>(p.S - 1));
      if (last) atomicExch(p.counters + u, 0u);
      misc[1] = last;
    }
    __syncthreads();
    if (!misc[1]) return;
    __threadfence();
    const int NC = p.S * K;
    const float* us = p.cand_score + u * p.S * K;
    const int32_t* ui = p.cand_idx + u * p.S * K;
    for (int i0 = tid; i0 < NC; i0 += 4 * NTHREADS) {
      int32_t idx[4];
      float sc[4];
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {   // four entries in flight per thread
        const int i = i0 + k2 * NTHREADS;
        idx[k2] = (i < NC) ? __ldcg(ui + i) : -1;
        sc[k2] = (i < NC) ? __ldcg(us + i) : 0.f;
      }
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        const int i = i0 + k2 * NTHREADS;
        if (i < NC) mb[i] = idx[k2] >= 0 ? composite(order_key(sc[k2]), static_cast<uint32_t>(idx[k2])) : 0ull;
      }
    }
  }
  __syncthreads();
  const uint64_t* top = mb;
  if (K <= 32) warp_merge_tree<1>(mb, p.S, K);
  else if (K <= 64) warp_merge_tree<2>(mb, p.S, K);
  else if (K <= 128) warp_merge_tree<4>(mb, p.S, K);
  else top = merge_tree(mb, mb + p.S * K, p.S, K);
  for (int i = tid; i < K; i += NTHREADS) {
    const uint64_t x = top[i];
    const long long o = u * K + i;
    p.idx_out[o] = x ? composite_index(x) : -1;
    if (p.score_out) p.score_out[o] = x ? key_to_score(static_cast<uint32_t>(x >> 32)) : neg_inf();
  }
}

template <int MODE, int D, bool PRE>
int smem_t(const TopkParams& p) {
  return topk_layout<MODE, D>(PRE, p.spw, p.chunk, p.k, p.S).total;
}

template <int MODE, int D, bool PRE>
cudaError_t set_max_smem() {
  const TopkLayout l = topk_layout<MODE, D>(PRE, kSpwMax, kTopkMaxChunk, kMaxTopk, kTopkMaxCand / kMaxTopk);
  return set_smem_once(reinterpret_cast<const void*>(&topk_kernel<MODE, D, PRE>), l.total);
}

template <int MODE, int D, bool PRE>
cudaError_t launch_t(const TopkParams& p, cudaStream_t s) {
  const int smem = smem_t<MODE, D, PRE>(p);
  cudaError_t e = set_max_smem<MODE, D, PRE>();
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.c.B) * p.c.Hkv * p.S;
  if (!p.cluster) {
    topk_kernel<MODE, D, PRE><<<static_cast<unsigned>(grid), NTHREADS, smem, s>>>(p);
    return cudaGetLastError();
  }
  if (p.S < 2 || p.S > kClusterMax || p.k > 128) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute at{};
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = static_cast<unsigned>(p.S);
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel<MODE, D, PRE>, p);
}

template <int MODE>
cudaError_t launch_m(const TopkParams& p, bool pre, cudaStream_t s) {
  if (p.c.D == 128) return pre ? launch_t<MODE, 128, true>(p, s) : launch_t<MODE, 128, false>(p, s);
  return pre ? launch_t<MODE, 64, true>(p, s) : launch_t<MODE, 64, false>(p, s);
}

// CTAs per SM of one variant at `smem` bytes of dynamic shared memory, cached
// per device in 1 KB steps (0 if unknown).
template <int MODE, int D, bool PRE>
int per_sm_t(int smem) {
  constexpr int kMaxDev = 64;
  constexpr int kSteps = 240;
  static int cached[kMaxDev][kSteps] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  const int step = (smem + 1023) / 1024;
  if (step >= kSteps) return 0;
  if (cached[dev][step] > 0) return cached[dev][step];
  if (set_max_smem<MODE, D, PRE>() != cudaSuccess) return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_kernel<MODE, D, PRE>, NTHREADS, step * 1024) !=
      cudaSuccess)
    return 0;
  cached[dev][step] = per_sm;
  return per_sm;
}

// Clusters of `size` CTAs of one variant at `smem` bytes that fit on the
// device at once, cached per device, size and 1 KB step (0: none or unknown).
template <int MODE, int D, bool PRE>
int clusters_t(int size, int smem) {
  constexpr int kMaxDev = 64;
  constexpr int kSteps = 240;
  static int cached[kMaxDev][kClusterMax + 1][kSteps] = {};   // 0: not queried, -1: none
  int dev = 0;
  if (size < 2 || size > kClusterMax) return 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  const int step = (smem + 1023) / 1024;
  if (step >= kSteps) return 0;
  int& c = cached[dev][size][step];
  if (c != 0) return c > 0 ? c : 0;
  if (set_max_smem<MODE, D, PRE>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(size), 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(step) * 1024;
  cudaLaunchAttribute at{};
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = static_cast<unsigned>(size);
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, topk_kernel<MODE, D, PRE>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    c = -1;
    return 0;
  }
  c = n;
  return n;
}

long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

// Split plan: over S from the fewest splits the chunk limit allows to the most
// that the candidate limit and the chunk alignment allow, minimise
// waves x (chunk x per-token cost + fixed per-CTA cost) + merge cost.  Chunks
// are multiples of NW x max(G, tile) tokens, so each consumer warp scores
// whole key groups.  The streaming variant keeps kSpwMax tiles per warp in
// flight when two CTAs still fit on an SM, else two.
template <int MODE>
long long align_t(int G) {
  return std::max<long long>(kChunkAlign, static_cast<long long>(NW) * std::max(G, Mode<MODE>::TT));
}

template <int MODE, int D, bool PRE>
TopkPlan plan_t(long long Lq, long long U, int G, int k) {
  constexpr int kTwoPerSm = 112 * 1024;   // dynamic shared memory that still lets two CTAs share an SM
  const long long align = align_t<MODE>(G);
  const long long s_lo = std::max(1LL, ceil_div_ll(Lq, kTopkMaxChunk));
  const long long s_hi = std::max(s_lo, std::min(ceil_div_ll(Lq, align), static_cast<long long>(kTopkMaxCand / k)));
  const int sms = device_sm_count();
  const double per_token = PRE ? 0.125 : 1.0;
  TopkPlan best{0, 0, 2, 0};
  double best_cost = 0.0;
  for (long long S = s_lo; S <= s_hi; ++S) {
    const long long ch = ceil_div_ll(ceil_div_ll(Lq, S), align) * align;
    if (ch > kTopkMaxChunk && S < s_hi) continue;
    const long long s_eff = ceil_div_ll(Lq, ch);
    if (s_eff != S) continue;
    int spw = kSpwMax;
    if (!PRE && topk_layout<MODE, D>(false, spw, ch, k, static_cast<int>(S)).total > kTwoPerSm) spw = 2;
    const int smem = topk_layout<MODE, D>(PRE, spw, ch, k, static_cast<int>(S)).total;
    const int per_sm = per_sm_t<MODE, D, PRE>(smem);
    const long long slots = (per_sm > 0 && sms > 0) ? static_cast<long long>(per_sm) * sms : target_ctas();
    const long long waves = ceil_div_ll(U * S, slots);
    const double cost = static_cast<double>(waves) * (static_cast<double>(ch) * per_token + 1024.0) +
                        0.25 * static_cast<double>(S * k);
    if (best.S == 0 || cost < best_cost) {
      best = TopkPlan{static_cast<int>(S), ch, spw, 0};
      best_cost = cost;
    }
  }
  if (best.S == 0) {  // the chunk limit alone
    best.chunk = std::min<long long>(kTopkMaxChunk, ceil_div_ll(ceil_div_ll(Lq, s_lo), kChunkAlign) * kChunkAlign);
    best.S = static_cast<int>(ceil_div_ll(Lq, best.chunk));
    best.spw = 2;
  }
  if (best.S >= 2 && best.S <= kClusterMax && k <= 128) {
    const int smem = topk_layout<MODE, D>(PRE, best.spw, best.chunk, k, best.S).total;
    best.cluster = clusters_t<MODE, D, PRE>(best.S, smem) > 0 ? 1 : 0;
  }
  return best;
}

template <int MODE>
TopkPlan plan_m(int D, long long Lq, long long U, int G, int k, bool pre) {
  if (D == 128) return pre ? plan_t<MODE, 128, true>(Lq, U, G, k) : plan_t<MODE, 128, false>(Lq, U, G, k);
  return pre ? plan_t<MODE, 64, true>(Lq, U, G, k) : plan_t<MODE, 64, false>(Lq, U, G, k);
}

}  // namespace

TopkPlan topk_plan(int mode, int D, int G, long long Lq, long long U, int k, bool pre) {
  if (Lq <= 0) return TopkPlan{1, 0, 2, 0};
  switch (mode) {
    case KVQ_MODE_INT4: return plan_m<KVQ_MODE_INT4>(D, Lq, U, G, k, pre);
    case KVQ_MODE_INT2: return plan_m<KVQ_MODE_INT2>(D, Lq, U, G, k, pre);
    case KVQ_MODE_INT1: return plan_m<KVQ_MODE_INT1>(D, Lq, U, G, k, pre);
    default: return TopkPlan{0, 0, 2, 0};
  }
}

long long topk_align(int mode, int /*D*/, int G) {
  switch (mode) {
    case KVQ_MODE_INT4: return align_t<KVQ_MODE_INT4>(G);
    case KVQ_MODE_INT2: return align_t<KVQ_MODE_INT2>(G);
    case KVQ_MODE_INT1: return align_t<KVQ_MODE_INT1>(G);
    default: return kChunkAlign;
  }
}

cudaError_t launch_topk(const TopkParams& p, int mode, bool pre, cudaStream_t s) {
  switch (mode) {
    case KVQ_MODE_INT4: return launch_m<KVQ_MODE_INT4>(p, pre, s);
    case KVQ_MODE_INT2: return launch_m<KVQ_MODE_INT2>(p, pre, s);
    case KVQ_MODE_INT1: return launch_m<KVQ_MODE_INT1>(p, pre, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
