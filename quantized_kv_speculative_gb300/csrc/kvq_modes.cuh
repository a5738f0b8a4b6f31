// Read modes and the register-level fragment builders for the quantized planes.
//
// Storage (see kvq.h): key planes are token-major with channels packed; value
// planes are 32-token slabs with rows = channels and tokens packed.  Read modes
// (QuantSpec page, "Approach"; SpeCache page, "Approach"):
//   INT8: both nibble planes of the hierarchical code, 8-bit codes, scale x1
//   INT4: the upper nibble plane only (the draft code), scale x16
//   INT2 / INT1: the 2-/1-bit planes, scale x1
//
// Tensor-core mapping (m16n8k16, see kvq_device.cuh).  Lane = 4*g + q.
// Logits are S = K x W:
//  * A = key codes (rows = 16 tokens of an m-tile, k = 16 channels of a k-step)
//  * B = folded query weights (column = query row and high / low f16 part)
// Thread q owns channels [q*D/4, (q+1)*D/4) of every token row.  It turns them
// into D/8 half2 "pairs" P[p]; k-step kk consumes P[2kk] and P[2kk+1].
// kx_chan() gives the channels of pair p, so the weights are laid out over the
// same permutation.  The token each lane's A rows hold is chosen (xpair_a /
// xpair_b below) so that the logit registers a lane ends up with are, after one
// shuffle, a whole B register of P.V, whose A operand is the value codes
// (rows = channels, k = tokens).
#pragma once

#include "kvq_device.cuh"

namespace kvq {

template <int MODE>
struct Mode;
template <>
struct Mode<KVQ_MODE_INT8> {
  static constexpr int NP = 2, PB = 4, CB = 8, MULT = 1, TT = 32;
};
template <>
struct Mode<KVQ_MODE_INT4> {
  static constexpr int NP = 1, PB = 4, CB = 4, MULT = 16, TT = 32;
};
template <>
struct Mode<KVQ_MODE_INT2> {
  static constexpr int NP = 1, PB = 2, CB = 2, MULT = 1, TT = 64;
};
template <>
struct Mode<KVQ_MODE_INT1> {
  static constexpr int NP = 1, PB = 1, CB = 1, MULT = 1, TT = 64;
};

// Bytes of one key row per plane, and of one value slab row per plane.
template <int MODE, int D>
struct Rows {
  static constexpr int KROW = D * Mode<MODE>::PB / 8;
  static constexpr int VROW = 32 * Mode<MODE>::PB / 8;
  static constexpr int KCHUNK = KROW / 4;  // bytes of a key row owned by one lane
};

// ------------------------------------------------------------------------------
// Subnormal encoding (attention and top-k).  An f16 whose exponent field is 0
// is the subnormal m * 2^-24, m its 10-bit mantissa field, and the tensor cores take
// it exactly.  A b-bit code c whose bits sit at mantissa positions k..k+b-1
// (k + b <= 10) therefore reads as exactly c * 2^k * 2^-24: no offset to
// remove afterwards.  Two codes 16 bits apart in a 32-bit word become one half2
// with a single AND, and a word's codes above mantissa bit 9 need one shift
// first.  The power of two 2^k a pair carries (its factor) is divided out of
// the other operand: out of the folded query weights for keys, out of the
// folded probabilities for values.  The 8-bit target code first merges its two
// nibble planes into bytes (shift + LOP3 per four codes), then a PRMT puts each
// byte into the low half of an f16 (factor 1).
//
// For values, a lane reads 8 consecutive tokens 8q..8q+7 of a channel row;
// pair i covers tokens 8q + xpair_a(i), 8q + xpair_b(i) with factor
// 2^vs_log2fac(i).  For the key chunk of a lane (D/4 channels of a token row),
// pair p covers channels kx_chan(p, 0) and kx_chan(p, 1), with factor
// 2^ks_log2fac(p).
// ------------------------------------------------------------------------------

// Value token pair i of a lane's 8 tokens 8q..8q+7: tokens 8q + xpair_a(i)
// and 8q + xpair_b(i).  INT8: the merged nibble planes give the even tokens'
// bytes in one word and the odd tokens' in another; pairs (0,2), (1,3), (4,6),
// (5,7) keep the key rows that the two lanes of a quarter-warp read one row
// apart (no shared-memory bank conflict).  Others: (0,4), (1,5), (2,6), (3,7).
template <int MODE>
__host__ __device__ constexpr int xpair_a(int i) {
  return MODE == KVQ_MODE_INT8 ? 4 * (i >> 1) + (i & 1) : i;
}
template <int MODE>
__host__ __device__ constexpr int xpair_b(int i) {
  return xpair_a<MODE>(i) + (MODE == KVQ_MODE_INT8 ? 2 : 4);
}

// log2 of value pair i's factor.
template <int MODE>
__host__ __device__ constexpr int vs_log2fac(int i) {
  if constexpr (MODE == KVQ_MODE_INT8) return 0;
  else if constexpr (MODE == KVQ_MODE_INT4) return (i & 1) ? 4 : 0;
  else if constexpr (MODE == KVQ_MODE_INT2) return 2 * i;
  else return i;
}

// Channels (relative to the lane chunk) of key pair p.
template <int MODE, int D>
__host__ __device__ constexpr int kx_chan(int p, int e) {
  if constexpr (MODE == KVQ_MODE_INT8) {
    constexpr int A8[4] = {0, 4, 1, 5};
    return 8 * (p / 4) + A8[p % 4] + 2 * e;
  } else if constexpr (MODE == KVQ_MODE_INT4) {
    return 8 * (p / 4) + p % 4 + 4 * e;
  } else if constexpr (MODE == KVQ_MODE_INT2) {
    return 16 * (p / 8) + p % 8 + 8 * e;
  } else {
    return p + e * (D == 128 ? 16 : 8);
  }
}

// Position of lane-chunk channel `cl` among the chunk's key pairs, in halves:
// 2 * pair + (0: first channel of the pair, 1: second), the inverse of kx_chan.
template <int MODE, int D>
__host__ __device__ constexpr int kx_slot(int cl) {
  if constexpr (MODE == KVQ_MODE_INT8) {
    constexpr int SL8[8] = {0, 4, 1, 5, 2, 6, 3, 7};   // 2 * (pair within the octet) + e, per channel of the octet
    return 8 * (cl / 8) + SL8[cl % 8];
  } else if constexpr (MODE == KVQ_MODE_INT4) {
    return 2 * (4 * (cl / 8) + cl % 4) + (cl % 8) / 4;
  } else if constexpr (MODE == KVQ_MODE_INT2) {
    return 2 * (8 * (cl / 16) + cl % 8) + (cl % 16) / 8;
  } else {
    constexpr int HALF = D == 128 ? 16 : 8;
    return 2 * (cl % HALF) + cl / HALF;
  }
}

template <int MODE, int D>
__host__ __device__ constexpr bool kx_slot_inverts_chan() {
  for (int p = 0; p < D / 8; ++p)
    for (int e = 0; e < 2; ++e)
      if (kx_slot<MODE, D>(kx_chan<MODE, D>(p, e)) != 2 * p + e) return false;
  return true;
}
static_assert(kx_slot_inverts_chan<KVQ_MODE_INT8, 128>() && kx_slot_inverts_chan<KVQ_MODE_INT8, 64>(), "INT8 slots");
static_assert(kx_slot_inverts_chan<KVQ_MODE_INT4, 128>() && kx_slot_inverts_chan<KVQ_MODE_INT4, 64>(), "INT4 slots");
static_assert(kx_slot_inverts_chan<KVQ_MODE_INT2, 128>() && kx_slot_inverts_chan<KVQ_MODE_INT2, 64>(), "INT2 slots");
static_assert(kx_slot_inverts_chan<KVQ_MODE_INT1, 128>() && kx_slot_inverts_chan<KVQ_MODE_INT1, 64>(), "INT1 slots");

// log2 of key pair p's factor.  The factors repeat with a period that divides
// D/16, so both halves of a lane chunk see the same ones.
template <int MODE, int D>
__host__ __device__ constexpr int ks_log2fac(int p) {
  if constexpr (MODE == KVQ_MODE_INT8) return 0;
  else if constexpr (MODE == KVQ_MODE_INT4) return (p & 1) ? 4 : 0;
  else if constexpr (MODE == KVQ_MODE_INT2) return 2 * (p % 4);
  else return D == 128 ? p % 8 : p % 4;
}

// The largest key pair factor's log2 (the scoring weights are scaled to it).
template <int MODE, int D>
__host__ __device__ constexpr int score_log2fac_max() {
  int m = 0;
  for (int p = 0; p < D / 8; ++p) m = ks_log2fac<MODE, D>(p) > m ? ks_log2fac<MODE, D>(p) : m;
  return m;
}

template <int MODE, int D>
__host__ __device__ constexpr float ks_inv_fac(int p) {
  return 1.0f / static_cast<float>(1 << ks_log2fac<MODE, D>(p));
}

// The lane's key chunk of one token row as D/8 subnormal f16 pairs.  `k0`
// points at the chunk in plane 0; plane 1 (INT8 lower nibbles) lies
// `plane_stride` bytes further.
template <int MODE, int D>
__device__ __forceinline__ void key_pairs_s(const uint8_t* k0, int plane_stride, uint32_t (&P)[D / 8]) {
  if constexpr (MODE == KVQ_MODE_INT8) {
    constexpr int NWD = D / 32;
    uint32_t h[NWD], l[NWD];
    if constexpr (NWD == 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(k0);
      const uint4 w = *reinterpret_cast<const uint4*>(k0 + plane_stride);
      h[0] = v.x; h[1] = v.y; h[2] = v.z; h[3] = v.w;
      l[0] = w.x; l[1] = w.y; l[2] = w.z; l[3] = w.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(k0);
      const uint2 w = *reinterpret_cast<const uint2*>(k0 + plane_stride);
      h[0] = v.x; h[1] = v.y;
      l[0] = w.x; l[1] = w.y;
    }
#pragma unroll
    for (int w = 0; w < NWD; ++w) {
      const uint32_t E = ((h[w] << 4) & 0xF0F0F0F0u) | (l[w] & 0x0F0F0F0Fu);
      const uint32_t O = (h[w] & 0xF0F0F0F0u) | ((l[w] >> 4) & 0x0F0F0F0Fu);
      P[4 * w + 0] = __byte_perm(E, 0u, 0x4140);
      P[4 * w + 1] = __byte_perm(E, 0u, 0x4342);
      P[4 * w + 2] = __byte_perm(O, 0u, 0x4140);
      P[4 * w + 3] = __byte_perm(O, 0u, 0x4342);
    }
  } else if constexpr (MODE == KVQ_MODE_INT4) {
    // nibble n of word w is channel 8w + n; pairs (n, n + 4)
    constexpr int NWD = D / 32;
    uint32_t h[NWD];
    if constexpr (NWD == 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(k0);
      h[0] = v.x; h[1] = v.y; h[2] = v.z; h[3] = v.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(k0);
      h[0] = v.x; h[1] = v.y;
    }
#pragma unroll
    for (int w = 0; w < NWD; ++w) {
      const uint32_t t = h[w] >> 8;
      P[4 * w + 0] = h[w] & 0x000F000Fu;
      P[4 * w + 1] = h[w] & 0x00F000F0u;
      P[4 * w + 2] = t & 0x000F000Fu;
      P[4 * w + 3] = t & 0x00F000F0u;
    }
  } else if constexpr (MODE == KVQ_MODE_INT2) {
    // code n of word w (bits 2n) is channel 16w + n; pairs (n, n + 8)
    constexpr int NWD = D / 64;
    uint32_t h[NWD];
    if constexpr (NWD == 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(k0);
      h[0] = v.x; h[1] = v.y;
    } else {
      h[0] = *reinterpret_cast<const uint32_t*>(k0);
    }
#pragma unroll
    for (int w = 0; w < NWD; ++w) {
      const uint32_t t = h[w] >> 8;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        P[8 * w + n] = h[w] & (0x00030003u << (2 * n));
        P[8 * w + 4 + n] = t & (0x00030003u << (2 * n));
      }
    }
  } else {
    if constexpr (D == 128) {
      // bit n is channel n; pairs (n, n + 16)
      const uint32_t w = *reinterpret_cast<const uint32_t*>(k0);
      const uint32_t t = w >> 8;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        P[n] = w & (0x00010001u << n);
        P[8 + n] = t & (0x00010001u << n);
      }
    } else {
      // channels 0-7 at bits 0-7, 8-15 at bits 16-23; pairs (n, n + 8)
      const uint32_t h = *reinterpret_cast<const uint16_t*>(k0);
      const uint32_t w = (h & 0xFFu) | ((h & 0xFF00u) << 8);
      const uint32_t t = w >> 4;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        P[n] = w & (0x00010001u << n);
        P[4 + n] = t & (0x00010001u << n);
      }
    }
  }
}

// A fragments of P.V for one channel m-tile (rows ca = 16mt+g and cb = ca+8) of
// one 32-token slab, as subnormal f16 values code * 2^vs_log2fac(i) * 2^-24.
// a[s] serves k-step s: a[s][0..1] are pair 2s of rows ca/cb (k = 2q, 2q+1),
// a[s][2..3] pair 2s+1 (k = 2q+8, 2q+9).  `va`/`vb` point at rows ca/cb of
// plane 0.
template <int MODE>
__device__ __forceinline__ void value_frags_s(const uint8_t* va, const uint8_t* vb, int plane_stride, int q,
                                              uint32_t (&a)[2][4]) {
  uint32_t pa[4], pb[4];
  if constexpr (MODE == KVQ_MODE_INT8) {
    const uint32_t ha = *reinterpret_cast<const uint32_t*>(va + 4 * q);
    const uint32_t hb = *reinterpret_cast<const uint32_t*>(vb + 4 * q);
    const uint32_t la = *reinterpret_cast<const uint32_t*>(va + plane_stride + 4 * q);
    const uint32_t lb = *reinterpret_cast<const uint32_t*>(vb + plane_stride + 4 * q);
    const uint32_t Ea = ((ha << 4) & 0xF0F0F0F0u) | (la & 0x0F0F0F0Fu);
    const uint32_t Oa = (ha & 0xF0F0F0F0u) | ((la >> 4) & 0x0F0F0F0Fu);
    const uint32_t Eb = ((hb << 4) & 0xF0F0F0F0u) | (lb & 0x0F0F0F0Fu);
    const uint32_t Ob = (hb & 0xF0F0F0F0u) | ((lb >> 4) & 0x0F0F0F0Fu);
    // E byte k = token 2k, O byte k = token 2k + 1 (pairs per xpair_a / xpair_b)
    pa[0] = __byte_perm(Ea, 0u, 0x4140); pa[1] = __byte_perm(Oa, 0u, 0x4140);
    pa[2] = __byte_perm(Ea, 0u, 0x4342); pa[3] = __byte_perm(Oa, 0u, 0x4342);
    pb[0] = __byte_perm(Eb, 0u, 0x4140); pb[1] = __byte_perm(Ob, 0u, 0x4140);
    pb[2] = __byte_perm(Eb, 0u, 0x4342); pb[3] = __byte_perm(Ob, 0u, 0x4342);
  } else if constexpr (MODE == KVQ_MODE_INT4) {
    // nibble i of the word is token 8q + i
    const uint32_t wa = *reinterpret_cast<const uint32_t*>(va + 4 * q);
    const uint32_t wb = *reinterpret_cast<const uint32_t*>(vb + 4 * q);
    const uint32_t ta = wa >> 8, tb = wb >> 8;
    pa[0] = wa & 0x000F000Fu; pa[1] = wa & 0x00F000F0u; pa[2] = ta & 0x000F000Fu; pa[3] = ta & 0x00F000F0u;
    pb[0] = wb & 0x000F000Fu; pb[1] = wb & 0x00F000F0u; pb[2] = tb & 0x000F000Fu; pb[3] = tb & 0x00F000F0u;
  } else if constexpr (MODE == KVQ_MODE_INT2) {
    const uint32_t xa = *reinterpret_cast<const uint16_t*>(va + 2 * q);
    const uint32_t xb = *reinterpret_cast<const uint16_t*>(vb + 2 * q);
    const uint32_t y = __byte_perm(xa, xb, 0x5140);   // [a.b0, b.b0, a.b1, b.b1]
    // token j of row a sits at bits 2j and 16+2j, of row b 8 bits higher
    const uint32_t yb = y >> 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pa[j] = y & (0x00030003u << (2 * j));
      pb[j] = yb & (0x00030003u << (2 * j));
    }
  } else {
    const uint32_t x = static_cast<uint32_t>(va[q]) | (static_cast<uint32_t>(vb[q]) << 8);
    const uint32_t y = (x & 0x0F0Fu) | ((x & 0xF0F0u) << 12);
    // token j of row a at bits j and 16+j, of row b 8 bits higher
    const uint32_t yb = y >> 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pa[j] = y & (0x00010001u << j);
      pb[j] = yb & (0x00010001u << j);
    }
  }
  a[0][0] = pa[0]; a[0][1] = pb[0]; a[0][2] = pa[1]; a[0][3] = pb[1];
  a[1][0] = pa[2]; a[1][1] = pb[2]; a[1][2] = pa[3]; a[1][3] = pb[3];
}

}  // namespace kvq
