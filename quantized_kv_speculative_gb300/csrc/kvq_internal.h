// Internal declarations shared by the host API (kvq_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int kMaxRows = 8;            // rows (gamma x query heads per KV head) per kernel
constexpr int kChunkAlign = 128;       // split boundaries are multiples of this many tokens
constexpr int kMaxChunk = 8192;        // tokens per attention split, up to four rows (bounds the selection bitmap)
constexpr int kMaxChunkWide = 16384;   // the same for the eight-row variants
__host__ __device__ constexpr int max_chunk_for_rows(int R) { return R > 4 ? kMaxChunkWide : kMaxChunk; }
constexpr int kCtasPerSmTarget = 4;   // split-count target per launch: this many CTAs per SM
constexpr int kTopkMaxChunk = 8192;    // tokens per top-k split (scores held in shared memory)
constexpr int kTopkMaxCand = 4096;     // splits x k candidates merged by the last CTA
constexpr int kMaxTopk = 1024;
constexpr int kMaxTailSplits = 8;      // CTAs per (b, kvh) for the bf16 tail
constexpr int kMaxCombine = 256;       // partials per (b, kvh) merged by the combine
constexpr int kMaxQuantSplits = kMaxCombine - kMaxTailSplits;
constexpr int kTailTokensPerSplit = 320;  // bf16 tail tokens per tail CTA (usually one per (b, kvh))
constexpr int kMaxClusterCtas = 16;   // CTAs per (b, kvh) that may combine as one thread-block cluster
constexpr int kStatusBytes = 256;      // workspace header (status word)
constexpr long long kDefaultWaitLimit = 4000000000LL;  // ~2 s at 2 GHz
constexpr int kMaxRaggedBatch = 64;    // sequences of a ragged cache (their lengths ride in the kernel parameters)
__host__ __device__ constexpr int kPartialFloats(int D) { return 2 * kMaxRows + kMaxRows * D; }

// Device view of one cache (all pointers already offset to the regions).
struct CacheView {
  const uint8_t* kplane[2];
  const uint8_t* vplane[2];
  const float* ksz;   // [u][C/G][2][D]
  const float* vsz;   // [u][C][2][D/G]
  const uint16_t* res_k;  // [u][2G][D] bf16
  const uint16_t* res_v;
  int B, Hkv, D, G, fmt;
  long long C;        // capacity tokens
  long long Lq;       // ragged: the largest sequence's
  int r, res_start;
  // Ragged cache: each sequence's own quantized length, residual fill and
  // residual start (read through seq_lq / seq_r / seq_start below).
  int ragged;
  int32_t rag_lq[kMaxRaggedBatch];
  int16_t rag_r[kMaxRaggedBatch];
  int16_t rag_start[kMaxRaggedBatch];
};

__host__ __device__ inline long long seq_lq(const CacheView& c, int b) { return c.ragged ? c.rag_lq[b] : c.Lq; }
__host__ __device__ inline int seq_r(const CacheView& c, int b) { return c.ragged ? c.rag_r[b] : c.r; }
__host__ __device__ inline int seq_start(const CacheView& c, int b) { return c.ragged ? c.rag_start[b] : c.res_start; }

// One sequence's part of an append: its state before the call, the groups it
// flushes, and the new tokens that land in its residual buffer.
struct SeqAppend {
  int32_t lq;               // quantized tokens before this call
  int16_t r, start;         // residual fill and start before this call
  int32_t n;                // tokens this sequence appends (<= the launch's row stride n)
  int32_t nflush;           // groups quantized by this call
  int32_t first_new;        // first stream position (>= r) kept in the residual
  int32_t res_count;        // new tokens written into the residual buffer
};

struct AttendParams {
  CacheView c;
  const uint16_t* q;        // [B][gamma][Hq][D]
  int Hq, gamma, HG, R;
  const uint16_t* pend_k;   // [B][Hkv][P][D]
  const uint16_t* pend_v;
  int P;
  const int32_t* sel_idx;   // [B][Hkv][top_k]
  const uint16_t* sel_k;
  const uint16_t* sel_v;
  int top_k;
  float qscale;             // sm_scale * log2(e)
  float zshift;             // zero points read as z + zshift * s (8: the INT4 midpoint reading)
  float smul;               // INT1 variants: scales read as smul * s (1/2: the centred 1-bit reading)
  uint16_t* out;            // [B][gamma][Hq][D]
  float* lse;               // [B][gamma][Hq] or null
  int* status;
  unsigned* counters;       // [B*Hkv]
  float* partials;          // [B*Hkv][S_q+S_t][kPartialFloats(D)]
  int S_q;                  // quantized splits per (b, kvh)
  int S_t;                  // tail splits per (b, kvh): residual + pending + selected tokens
  long long chunk;          // tokens per split (multiple of kChunkAlign)
  long long wait_limit;
  int cluster;              // 1: the S_q + S_t CTAs of a unit form one cluster and combine in shared memory
  // Scoring variants only: query row whose heads' summed query scores every
  // quantized token, and where each token's finished top-k score goes.
  int score_row;
  float* pre;               // [B*Hkv][C]
};

struct TopkParams {
  CacheView c;
  const uint16_t* q;        // query row of sequence b at q + b * q_bstride: [Hq][D]
  long long q_bstride;      // elements between sequences' query rows
  const float* pre;         // pre-scored launch: [B*Hkv][C] finished scores from the attention's scoring pass
  int Hq, HG, k;
  float zshift;             // key zero points read as fp32(z + zshift * s)
  float smul;               // INT1 variants: key scales read as smul * s
  int32_t* idx_out;         // [B][Hkv][k]
  float* score_out;         // [B][Hkv][k] or null
  int* status;
  unsigned* counters;       // [B*Hkv]
  float* cand_score;        // [B*Hkv][S][k]
  int32_t* cand_idx;
  int S;
  long long chunk;
  long long align;          // chunk alignment of the plan (per-sequence chunks of a ragged cache)
  int spw;                  // stage slots per warp (streaming variant)
  int cluster;              // 1: the S CTAs of a (b, kv head) form one cluster and merge through shared memory
  long long wait_limit;
};

// A top-k launch plan.
struct TopkPlan {
  int S;                    // splits per (b, kv head)
  long long chunk;          // tokens per split
  int spw;                  // stage slots per warp of the streaming variant
  int cluster;              // 1: one thread-block cluster per (b, kv head)
};

struct FlushParams {
  // writable views of the cache regions
  uint8_t* kplane[2];
  uint8_t* vplane[2];
  float* ksz;
  float* vsz;
  const uint16_t* res_k;
  const uint16_t* res_v;
  const uint16_t* k_new;    // [B][Hkv][n][D]
  const uint16_t* v_new;
  int B, Hkv, D, G, fmt;
  long long C, Lq;          // Lq before this call
  int r, res_start, n;      // residual state before this call, tokens in this call
  int nflush;               // groups quantized by this launch (ragged: the most any sequence flushes)
  // New tokens written into the residual buffer by the same launch: the CTA
  // that arrives last at the head's counter (after every CTA of the head has
  // read its old slots) writes them and resets the counter.
  uint16_t* res_k_w;
  uint16_t* res_v_w;
  int first_new, res_count;
  unsigned* ctr;            // [B * Hkv] arrival counters, zero between launches
  int ragged;               // 1: per-sequence parts in seq[] (the scalars above are unused)
  SeqAppend seq[kMaxRaggedBatch];
};

// The CTAs of one flushed group: key parts over 32-channel ranges, then value
// parts over one block of G channels (all G tokens) or, when the block is all
// D channels, over one 32-token slab.
struct FlushSplit {
  int npk, npv, tv, cv;
};
__host__ __device__ inline FlushSplit flush_split(int D, int G) {
  FlushSplit s{};
  s.npk = D / 32;
  if (D / G >= 2) {
    s.npv = D / G;
    s.tv = G;
    s.cv = G;
  } else {
    s.npv = G / 32;
    s.tv = 32;
    s.cv = D;
  }
  return s;
}

struct ResidualWriteParams {
  uint16_t* res_k;
  uint16_t* res_v;
  const uint16_t* k_new;
  const uint16_t* v_new;
  int B, Hkv, D, G, n;
  int r, res_start;         // before this call
  int first_new;            // first stream position (>= r) kept in the residual
  int count;                // tokens to write (ragged: the most any sequence writes)
  int ragged;               // 1: per-sequence r, start, first_new and count (res_count) in seq[]
  SeqAppend seq[kMaxRaggedBatch];
};

// The kernel variant a read mode runs (the INT4 midpoint reading runs the INT4
// kernels with a zero shift) and that shift.
// A read mode's kernel variant, and its zero-point shift and scale multiplier
// on top of the variant's own: INT4_MID reads zero point z + 8 s; INT1_CENTER
// reads zero point z + s/4 and scale s/2.
inline int kernel_mode(int mode) {
  return mode == KVQ_MODE_INT4_MID ? KVQ_MODE_INT4 : (mode == KVQ_MODE_INT1_CENTER ? KVQ_MODE_INT1 : mode);
}
inline float mode_zero_shift(int mode) {
  return mode == KVQ_MODE_INT4_MID ? 8.0f : (mode == KVQ_MODE_INT1_CENTER ? 0.25f : 0.0f);
}
inline float mode_scale_mul(int mode) { return mode == KVQ_MODE_INT1_CENTER ? 0.5f : 1.0f; }

cudaError_t launch_flush(const FlushParams& p, cudaStream_t s);
cudaError_t launch_residual_write(const ResidualWriteParams& p, cudaStream_t s);
// `score`: the variant that also scores every quantized token for the next
// step's top-k (p.pre, p.score_row).
cudaError_t launch_attend(const AttendParams& p, int mode, bool score, cudaStream_t s);
// CTAs of the attention kernel variant that fit on the current device at once
// (0 if unknown).
int attend_resident_ctas(int mode, int D, int G, int R, bool score);
// Clusters of `size` CTAs of that variant that fit on the current device at
// once (0 if unknown or if the size cannot be launched).
int attend_resident_clusters(int mode, int D, int G, int R, int size, bool score);
// `pre`: select from the scores the attention's scoring variant wrote (p.pre)
// instead of scoring the key planes.
cudaError_t launch_topk(const TopkParams& p, int mode, bool pre, cudaStream_t s);
// Top-k plan for the current device (`pre`: the pre-scored variant).
TopkPlan topk_plan(int mode, int D, int G, long long Lq, long long U, int k, bool pre);
// The chunk alignment topk_plan uses for a variant (whole key groups per warp).
long long topk_align(int mode, int D, int G);
cudaError_t launch_wait_selftest(int* status, long long limit, cudaStream_t s);
// SMs of the current device (cached per device; 0 if unknown).
int device_sm_count();
// Split-count target of one launch on the current device: kCtasPerSmTarget x
// its SM count (152 SMs assumed when the count is unknown).
long long target_ctas();
// kvq_attend's argument checks (all but the workspace), with kvq_attend's
// status codes; on KVQ_OK *ws_need holds the workspace bytes the call needs.
kvq_status attend_check(const kvq_cache* cache, int mode, const void* q, int num_q_heads, int gamma,
                        const void* pend_k, const void* pend_v, int n_pend, const int32_t* sel_idx,
                        const void* sel_k, const void* sel_v, int top_k, const void* out, const float* lse,
                        size_t* ws_need);

}  // namespace kvq
