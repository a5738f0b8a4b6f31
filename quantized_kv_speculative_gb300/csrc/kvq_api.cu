// Host side of the C ABI declared in include/kvq.h: argument validation, the
// 2G double-buffer state machine, split sizing, workspace layout and launches.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "kvq_internal.h"

using namespace kvq;

namespace {

constexpr uint32_t kMagic = 0x4B565131u;  // "KVQ1"
constexpr uint32_t kFlagCountersZeroed = 1u;   // kvq_cache.flags: flush counters zeroed on the device

// The flush kernel's arrival counters start at zero: zeroed on the stream
// before the cache's first flush, whatever was appended before it.
kvq_status zero_counters_once(kvq_cache* cache, unsigned* ctr, cudaStream_t s);

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A split CTA's fixed cost in the attention split planner, in tokens of its
// chunk: set-up, first copies, merge and combine.  Measured on the GB300 at
// the 128K verify call: with 1024 the planner keeps one wave of 8 splits per
// head (0.231 ms) instead of two waves of 17 (0.236 ms); no other workload's
// plan changes between 256 and 2048.
constexpr long long kSplitOverheadTokens = 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_desc(const kvq_cache_desc* d) {
  if (!d) return false;
  if (d->batch < 1 || d->num_kv_heads < 1) return false;
  if (d->head_dim != 64 && d->head_dim != 128) return false;
  if (d->group_size != 32 && d->group_size != 64 && d->group_size != 128) return false;
  if (d->head_dim % d->group_size) return false;
  if (d->format != KVQ_FMT_HIER8 && d->format != KVQ_FMT_INT2 && d->format != KVQ_FMT_INT1) return false;
  if (d->reserved0 != 0) return false;
  if (d->capacity_tokens < 0 || d->capacity_tokens % d->group_size) return false;
  if (d->capacity_tokens > static_cast<long long>(kMaxQuantSplits) * kMaxChunk) return false;
  const long long units = static_cast<long long>(d->batch) * d->num_kv_heads;
  if (units > (1LL << 24)) return false;
  return true;
}

struct Regions {
  int np;
  size_t k_plane, v_plane, k_sz, v_sz, res, ctr, total;
};

Regions regions(const kvq_cache_desc* d) {
  Regions r{};
  const size_t U = static_cast<size_t>(d->batch) * d->num_kv_heads;
  const size_t C = static_cast<size_t>(d->capacity_tokens);
  const size_t D = d->head_dim, G = d->group_size;
  const size_t pb = (d->format == KVQ_FMT_HIER8) ? 4 : static_cast<size_t>(d->format);
  r.np = (d->format == KVQ_FMT_HIER8) ? 2 : 1;
  r.k_plane = align256(U * C * D * pb / 8);
  r.v_plane = align256(U * C * D * pb / 8);
  r.k_sz = align256(U * (C / G) * 2 * D * 4);
  r.v_sz = align256(U * C * 2 * (D / G) * 4);
  r.res = align256(U * 2 * G * D * 2);
  r.ctr = align256(U * 4);
  r.total = r.np * (r.k_plane + r.v_plane) + r.k_sz + r.v_sz + 2 * r.res + r.ctr;
  return r;
}

bool cache_ok(const kvq_cache* c) { return c && c->magic == kMagic && valid_desc(&c->desc); }

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

long long units_of(const kvq_cache* c) {
  return static_cast<long long>(c->desc.batch) * c->desc.num_kv_heads;
}

// Quantized splits per (b, kvh) for attention, and the chunk size.  `slots` is
// how many CTAs of the kernel fit on the device at once.  Over the split counts
// from the fewest the chunk limit allows to the target_ctas() share, pick the one
// with the smallest waves x (chunk + per-split overhead), the `tail` CTAs per
// (b, kvh) counted in the waves; chunks are multiples of kChunkAlign.
int attend_splits(long long Lq, long long U, long long slots, long long tail, long long max_chunk, long long* chunk) {
  if (Lq <= 0) {
    *chunk = 0;
    return 0;
  }
  const long long s_min = std::max(1LL, ceil_div(Lq, max_chunk));
  const long long s_cap = std::max(
      s_min, std::min<long long>(kMaxQuantSplits, std::min(ceil_div(Lq, kChunkAlign), std::max(1LL, ceil_div(target_ctas(), U)))));
  long long best_s = 0, best_ch = 0, best_cost = 0;
  for (long long S = s_min; S <= s_cap; ++S) {
    const long long ch = ceil_div(ceil_div(Lq, S), kChunkAlign) * kChunkAlign;
    if (ch > max_chunk || ceil_div(Lq, ch) != S) continue;
    const long long waves = slots > 0 ? ceil_div(U * (S + tail), slots) : 1;
    const long long cost = waves * (ch + kSplitOverheadTokens);
    if (best_s == 0 || cost < best_cost || (slots <= 0 && S > best_s)) {
      best_s = S;
      best_ch = ch;
      best_cost = cost;
    }
  }
  if (best_s == 0) {   // no split count meets both limits exactly: the chunk limit wins
    best_ch = std::min(max_chunk, ceil_div(ceil_div(Lq, s_min), kChunkAlign) * kChunkAlign);
    best_s = ceil_div(Lq, best_ch);
  }
  *chunk = best_ch;
  return static_cast<int>(best_s);
}

// The cluster combine is on unless the environment sets KVQ_ATTEND_CLUSTERS=0
// (read on every call; the ticket combine then serves every launch).
bool clusters_enabled() {
  const char* v = std::getenv("KVQ_ATTEND_CLUSTERS");
  return !(v && v[0] == '0' && v[1] == '\0');
}

int attend_splits_max(const kvq_cache_desc* d) {
  const long long U = static_cast<long long>(d->batch) * d->num_kv_heads;
  const long long Lq = d->capacity_tokens;
  if (Lq <= 0) return 0;
  const long long target = std::min<long long>(kMaxQuantSplits, std::max(1LL, ceil_div(target_ctas(), U)));
  long long S = std::min(ceil_div(Lq, kChunkAlign), target);
  S = std::max(S, ceil_div(Lq, kMaxChunk));
  return static_cast<int>(std::max(S, 1LL));
}

// Largest split count topk_plan can return for this cache and k (any fill,
// any device): its chunks are multiples of kChunkAlign tokens and at most
// kTopkMaxChunk, and S * k stays within kTopkMaxCand unless the chunk limit
// alone needs more splits.
int topk_splits_max(const kvq_cache_desc* d, int k) {
  const long long Lq = d->capacity_tokens;
  if (Lq <= 0) return 1;
  long long S = std::min(ceil_div(Lq, kChunkAlign), std::max(1LL, static_cast<long long>(kTopkMaxCand / k)));
  S = std::max(S, ceil_div(Lq, kTopkMaxChunk));
  return static_cast<int>(std::max(S, 1LL));
}

size_t attend_ws_bytes(const kvq_cache_desc* d) {
  const size_t U = static_cast<size_t>(d->batch) * d->num_kv_heads;
  const size_t S = static_cast<size_t>(attend_splits_max(d)) + kMaxTailSplits;
  return align256(U * 4) + align256(U * S * kPartialFloats(d->head_dim) * 4);
}

size_t topk_ws_bytes(const kvq_cache_desc* d, int k) {
  const size_t U = static_cast<size_t>(d->batch) * d->num_kv_heads;
  const size_t S = static_cast<size_t>(topk_splits_max(d, k));
  return align256(U * 4) + 2 * align256(U * S * static_cast<size_t>(k) * 4);
}

CacheView view_of(const kvq_cache* c) {
  CacheView v{};
  uint8_t* base = static_cast<uint8_t*>(c->base);
  v.kplane[0] = base + c->off_k_plane[0];
  v.kplane[1] = base + c->off_k_plane[1];
  v.vplane[0] = base + c->off_v_plane[0];
  v.vplane[1] = base + c->off_v_plane[1];
  v.ksz = reinterpret_cast<const float*>(base + c->off_k_sz);
  v.vsz = reinterpret_cast<const float*>(base + c->off_v_sz);
  v.res_k = reinterpret_cast<const uint16_t*>(base + c->off_res_k);
  v.res_v = reinterpret_cast<const uint16_t*>(base + c->off_res_v);
  v.B = c->desc.batch;
  v.Hkv = c->desc.num_kv_heads;
  v.D = c->desc.head_dim;
  v.G = c->desc.group_size;
  v.fmt = c->desc.format;
  v.C = c->desc.capacity_tokens;
  v.Lq = c->quantized_len;
  v.r = c->residual_len;
  v.res_start = c->residual_start;
  v.ragged = c->seqs != nullptr;
  if (v.ragged) {
    for (int b = 0; b < c->desc.batch; ++b) {
      v.rag_lq[b] = static_cast<int32_t>(c->seqs[b].quantized_len);
      v.rag_r[b] = static_cast<int16_t>(c->seqs[b].residual_len);
      v.rag_start[b] = static_cast<int16_t>(c->seqs[b].residual_start);
    }
  }
  return v;
}

// One sequence's part of an append of n tokens to state (lq, r, start), as
// the 2G double buffer runs it token by token: f groups flush, and the new
// tokens from stream position first_new on stay in the residual buffer.
SeqAppend plan_seq_append(long long lq, int r, int start, int n, int G) {
  SeqAppend a{};
  const long long T = static_cast<long long>(r) + n;
  const long long f = (T < 2LL * G) ? 0 : T / G - 1;
  const long long first_new = std::max<long long>(r, f * G);
  a.lq = static_cast<int32_t>(lq);
  a.r = static_cast<int16_t>(r);
  a.start = static_cast<int16_t>(start);
  a.n = n;
  a.nflush = static_cast<int32_t>(f);
  a.first_new = static_cast<int32_t>(first_new);
  a.res_count = static_cast<int32_t>(T - first_new);
  return a;
}

bool mode_reads(int mode, int fmt) {
  switch (mode) {
    case KVQ_MODE_INT8:
    case KVQ_MODE_INT4:
    case KVQ_MODE_INT4_MID: return fmt == KVQ_FMT_HIER8;
    case KVQ_MODE_INT2: return fmt == KVQ_FMT_INT2;
    case KVQ_MODE_INT1:
    case KVQ_MODE_INT1_CENTER: return fmt == KVQ_FMT_INT1;
    default: return false;
  }
}

// The attention launch plan: quantized splits and chunk, tail CTAs, and
// whether each (b, kvh) runs as one thread-block cluster.
struct AttendPlan {
  int S_q, S_t;
  long long chunk;
  int cluster;
};

AttendPlan plan_attend(const kvq_cache* cache, int mode, int R, int n_pend, int top_k, bool score = false) {
  AttendPlan pl{};
  const long long U = units_of(cache);
  const long long slots =
      attend_resident_ctas(kernel_mode(mode), cache->desc.head_dim, cache->desc.group_size, R, score);
  const long long max_chunk = max_chunk_for_rows(R);
  // The bf16 tail (residual, pending and selected tokens) goes to CTAs of its
  // own when they fit in the first wave beside the quantized splits without
  // making the chunks longer, or (below) when they would not fit beside the
  // splits at all; otherwise each quantized split takes a slice of it after
  // its own tokens.
  const long long ntail = static_cast<long long>(cache->residual_len) + n_pend + top_k;
  const int S_t = static_cast<int>(std::min<long long>(kMaxTailSplits, std::max(1LL, ceil_div(ntail, kTailTokensPerSplit))));
  if (cache->quantized_len > 0) {
    long long ch_fused = 0, ch_sep = 0;
    const int sq_fused = attend_splits(cache->quantized_len, U, slots, 0, max_chunk, &ch_fused);
    const int sq_sep = attend_splits(cache->quantized_len, U, slots, S_t, max_chunk, &ch_sep);
    const bool sep = slots > 0 && (sq_sep + S_t) * U <= slots && ch_sep <= ch_fused;
    pl.S_t = sep ? S_t : 0;
    pl.S_q = sep ? sq_sep : sq_fused;
    pl.chunk = sep ? ch_sep : ch_fused;
  } else {
    pl.S_t = S_t;
    pl.S_q = attend_splits(cache->quantized_len, U, slots, pl.S_t, max_chunk, &pl.chunk);
  }
  // When the tail CTAs would not fit in the first wave beside the quantized
  // splits, they still run, launched after the splits and combining through
  // the workspace: they take free slots and those of the first splits to
  // finish (a unit's last split is usually shorter, and the CTAs
  // that started first on an SM stream fastest), and no split ends with a
  // share of the tail.  Measured: 32K and 128K draft calls 8% and 3% faster,
  // the SpeCache batch (two waves of three-CTA clusters before) 1.7% faster.
  if (pl.S_t == 0 && cache->quantized_len > 0 && slots > 0 && (pl.S_q + S_t) * U > slots) {
    pl.S_t = S_t;
    return pl;
  }
  // One cluster per (b, kvh), combining in shared memory, when its CTAs fit
  // the cluster limit and the clusters fill no more waves than the plan counted.
  const int S_all = pl.S_q + pl.S_t;
  if (S_all >= 1 && S_all <= kMaxClusterCtas && slots > 0 && clusters_enabled()) {
    const long long cap =
        attend_resident_clusters(kernel_mode(mode), cache->desc.head_dim, cache->desc.group_size, R, S_all, score);
    if (cap > 0 && ceil_div(U, cap) <= ceil_div(U * S_all, slots)) pl.cluster = 1;
  }
  return pl;
}

kvq_status zero_counters_once(kvq_cache* cache, unsigned* ctr, cudaStream_t s) {
  if (cache->flags & kFlagCountersZeroed) return KVQ_OK;
  if (cudaMemsetAsync(ctr, 0, static_cast<size_t>(units_of(cache)) * 4, s) != cudaSuccess) return KVQ_ERR_CUDA;
  cache->flags |= kFlagCountersZeroed;
  return KVQ_OK;
}

// Per-token scores that kvq_attend_topk's attention pass writes for its
// selection pass: [B*Hkv][C] fp32.
size_t pre_score_bytes(const kvq_cache_desc* d) {
  return align256(static_cast<size_t>(d->batch) * d->num_kv_heads * static_cast<size_t>(d->capacity_tokens) * 4);
}

// Launch parameters of an attention call whose arguments are checked.
AttendParams make_attend_params(const kvq_cache* cache, int mode, const void* q, int num_q_heads, int gamma,
                                const void* pend_k, const void* pend_v, int n_pend, const int32_t* sel_idx,
                                const void* sel_k, const void* sel_v, int top_k, float sm_scale, void* out, float* lse,
                                uint8_t* ws, bool score) {
  const int HG = num_q_heads / cache->desc.num_kv_heads;
  if (!(sm_scale > 0.f)) sm_scale = 1.0f / std::sqrt(static_cast<float>(cache->desc.head_dim));
  AttendParams p{};
  p.c = view_of(cache);
  p.q = static_cast<const uint16_t*>(q);
  p.Hq = num_q_heads;
  p.gamma = gamma;
  p.HG = HG;
  p.R = gamma * HG;
  p.pend_k = static_cast<const uint16_t*>(pend_k);
  p.pend_v = static_cast<const uint16_t*>(pend_v);
  p.P = n_pend;
  p.sel_idx = sel_idx;
  p.sel_k = static_cast<const uint16_t*>(sel_k);
  p.sel_v = static_cast<const uint16_t*>(sel_v);
  p.top_k = top_k;
  p.qscale = sm_scale * 1.4426950408889634f;
  p.zshift = mode_zero_shift(mode);
  p.smul = mode_scale_mul(mode);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  const long long U = units_of(cache);
  p.status = reinterpret_cast<int*>(ws);
  p.counters = reinterpret_cast<unsigned*>(ws + kStatusBytes);
  p.partials = reinterpret_cast<float*>(ws + kStatusBytes + align256(U * 4));
  const AttendPlan pl = plan_attend(cache, mode, gamma * HG, n_pend, top_k, score);
  p.S_q = pl.S_q;
  p.S_t = pl.S_t;
  p.chunk = pl.chunk;
  p.cluster = pl.cluster;
  p.wait_limit = kDefaultWaitLimit;
  return p;
}

// Launch parameters of a top-k selection (arguments and plan checked).  The
// query row of sequence b sits at q + b * q_bstride.
TopkParams make_topk_params(const kvq_cache* cache, int mode, const uint16_t* q, long long q_bstride, int num_q_heads,
                            int k, int32_t* idx_out, float* score_out, uint8_t* workspace, const TopkPlan& plan) {
  const long long U = units_of(cache);
  TopkParams p{};
  p.c = view_of(cache);
  p.q = q;
  p.q_bstride = q_bstride;
  p.Hq = num_q_heads;
  p.HG = num_q_heads / cache->desc.num_kv_heads;
  p.k = k;
  p.zshift = mode_zero_shift(mode);
  p.smul = mode_scale_mul(mode);
  p.align = topk_align(kernel_mode(mode), cache->desc.head_dim, cache->desc.group_size);
  p.idx_out = idx_out;
  p.score_out = score_out;
  uint8_t* ws = workspace + kStatusBytes + attend_ws_bytes(&cache->desc);
  p.status = reinterpret_cast<int*>(workspace);
  p.counters = reinterpret_cast<unsigned*>(ws);
  const size_t Smax = static_cast<size_t>(topk_splits_max(&cache->desc, k));
  p.cand_score = reinterpret_cast<float*>(ws + align256(U * 4));
  p.cand_idx = reinterpret_cast<int32_t*>(ws + align256(U * 4) + align256(U * Smax * k * 4));
  p.S = plan.S;
  p.chunk = plan.chunk;
  p.spw = plan.spw;
  p.cluster = plan.cluster;
  p.wait_limit = kDefaultWaitLimit;
  return p;
}

}  // namespace

int kvq::device_sm_count() {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  if (cached[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = sms;
  }
  return cached[dev];
}

long long kvq::target_ctas() {
  const int sms = device_sm_count();
  return static_cast<long long>(kCtasPerSmTarget) * (sms > 0 ? sms : 152);
}

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CAPACITY: return "quantized capacity exceeded";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case KVQ_ERR_NOT_INITIALIZED: return "cache not initialized";
    default: return "unknown status";
  }
}

size_t kvq_cache_bytes(const kvq_cache_desc* desc) {
  if (!valid_desc(desc)) return 0;
  return regions(desc).total;
}

kvq_status kvq_cache_init(kvq_cache* cache, const kvq_cache_desc* desc, void* dev_mem, size_t bytes) {
  if (!cache || !valid_desc(desc)) return KVQ_ERR_INVALID_ARG;
  const Regions r = regions(desc);
  if (r.total > 0 && (!dev_mem || (reinterpret_cast<uintptr_t>(dev_mem) & 255u))) return KVQ_ERR_INVALID_ARG;
  if (bytes < r.total) return KVQ_ERR_INVALID_ARG;
  std::memset(cache, 0, sizeof(*cache));
  cache->desc = *desc;
  cache->base = dev_mem;
  cache->bytes = bytes;
  uint64_t off = 0;
  cache->off_k_plane[0] = off; off += r.k_plane;
  cache->off_k_plane[1] = (r.np == 2) ? off : cache->off_k_plane[0];
  if (r.np == 2) off += r.k_plane;
  cache->off_v_plane[0] = off; off += r.v_plane;
  cache->off_v_plane[1] = (r.np == 2) ? off : cache->off_v_plane[0];
  if (r.np == 2) off += r.v_plane;
  cache->off_k_sz = off; off += r.k_sz;
  cache->off_v_sz = off; off += r.v_sz;
  cache->off_res_k = off; off += r.res;
  cache->off_res_v = off; off += r.res;
  cache->quantized_len = 0;
  cache->residual_len = 0;
  cache->residual_start = 0;
  cache->magic = kMagic;
  return KVQ_OK;
}

kvq_status kvq_cache_set_ragged(kvq_cache* cache, kvq_seq_state* seqs, int32_t count) {
  if (!cache || cache->magic != kMagic) return KVQ_ERR_NOT_INITIALIZED;
  if (!valid_desc(&cache->desc) || !seqs || count != cache->desc.batch) return KVQ_ERR_INVALID_ARG;
  if (cache->quantized_len != 0 || cache->residual_len != 0) return KVQ_ERR_INVALID_ARG;
  if (count > kMaxRaggedBatch) return KVQ_ERR_UNSUPPORTED;
  for (int b = 0; b < count; ++b) seqs[b] = kvq_seq_state{0, 0, 0};
  cache->seqs = seqs;
  return KVQ_OK;
}

kvq_status kvq_quantize_append_ragged(kvq_cache* cache, const void* k_new, const void* v_new, int32_t n_max,
                                      const int32_t* n_new, kvq_stream_t stream) {
  if (!cache || cache->magic != kMagic) return KVQ_ERR_NOT_INITIALIZED;
  if (!valid_desc(&cache->desc) || !cache->seqs || !n_new || n_max < 0) return KVQ_ERR_INVALID_ARG;
  const int B = cache->desc.batch, G = cache->desc.group_size;
  int nflush_max = 0, count_max = 0, total = 0;
  SeqAppend plan[kMaxRaggedBatch];
  for (int b = 0; b < B; ++b) {
    if (n_new[b] < 0 || n_new[b] > n_max) return KVQ_ERR_INVALID_ARG;
    const kvq_seq_state& st = cache->seqs[b];
    plan[b] = plan_seq_append(st.quantized_len, st.residual_len, st.residual_start, n_new[b], G);
    if (plan[b].lq + static_cast<long long>(plan[b].nflush) * G > cache->desc.capacity_tokens)
      return KVQ_ERR_CAPACITY;
    nflush_max = std::max(nflush_max, plan[b].nflush);
    if (plan[b].nflush == 0) count_max = std::max(count_max, plan[b].res_count);
    total += n_new[b];
  }
  if (total == 0) return KVQ_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(cache->base);
  if (nflush_max > 0) {
    FlushParams p{};
    p.kplane[0] = base + cache->off_k_plane[0];
    p.kplane[1] = base + cache->off_k_plane[1];
    p.vplane[0] = base + cache->off_v_plane[0];
    p.vplane[1] = base + cache->off_v_plane[1];
    p.ksz = reinterpret_cast<float*>(base + cache->off_k_sz);
    p.vsz = reinterpret_cast<float*>(base + cache->off_v_sz);
    p.res_k = reinterpret_cast<const uint16_t*>(base + cache->off_res_k);
    p.res_v = reinterpret_cast<const uint16_t*>(base + cache->off_res_v);
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.B = B;
    p.Hkv = cache->desc.num_kv_heads;
    p.D = cache->desc.head_dim;
    p.G = G;
    p.fmt = cache->desc.format;
    p.C = cache->desc.capacity_tokens;
    p.n = n_max;
    p.nflush = nflush_max;
    p.res_k_w = reinterpret_cast<uint16_t*>(base + cache->off_res_k);
    p.res_v_w = reinterpret_cast<uint16_t*>(base + cache->off_res_v);
    p.ctr = reinterpret_cast<unsigned*>(base + cache->off_res_v + regions(&cache->desc).res);
    p.ragged = 1;
    for (int b = 0; b < B; ++b) {
      p.seq[b] = plan[b];
      if (plan[b].nflush == 0) p.seq[b].res_count = 0;   // written by the residual copy below
    }
    if (zero_counters_once(cache, p.ctr, s) != KVQ_OK) return KVQ_ERR_CUDA;
    if (launch_flush(p, s) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  if (count_max > 0) {
    ResidualWriteParams w{};
    w.res_k = reinterpret_cast<uint16_t*>(base + cache->off_res_k);
    w.res_v = reinterpret_cast<uint16_t*>(base + cache->off_res_v);
    w.k_new = static_cast<const uint16_t*>(k_new);
    w.v_new = static_cast<const uint16_t*>(v_new);
    w.B = B;
    w.Hkv = cache->desc.num_kv_heads;
    w.D = cache->desc.head_dim;
    w.G = G;
    w.n = n_max;
    w.count = count_max;
    w.ragged = 1;
    for (int b = 0; b < B; ++b) {
      w.seq[b] = plan[b];
      if (plan[b].nflush > 0) w.seq[b].res_count = 0;    // written by the flush launch above
    }
    if (launch_residual_write(w, s) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  long long lq_max = 0;
  int r_max = 0;
  for (int b = 0; b < B; ++b) {
    kvq_seq_state& st = cache->seqs[b];
    const long long T = static_cast<long long>(st.residual_len) + n_new[b];
    st.quantized_len += static_cast<long long>(plan[b].nflush) * G;
    st.residual_len = static_cast<int32_t>(T - static_cast<long long>(plan[b].nflush) * G);
    st.residual_start = static_cast<int32_t>((st.residual_start + static_cast<long long>(plan[b].nflush) * G) % (2 * G));
    lq_max = std::max(lq_max, static_cast<long long>(st.quantized_len));
    r_max = std::max(r_max, st.residual_len);
  }
  cache->quantized_len = lq_max;
  cache->residual_len = r_max;
  return KVQ_OK;
}

kvq_status kvq_quantize_append(kvq_cache* cache, const void* k_new, const void* v_new, int32_t n_new,
                               kvq_stream_t stream) {
  if (!cache || cache->magic != kMagic) return KVQ_ERR_NOT_INITIALIZED;
  if (!valid_desc(&cache->desc)) return KVQ_ERR_INVALID_ARG;
  if (n_new < 0) return KVQ_ERR_INVALID_ARG;
  if (n_new == 0) return KVQ_OK;
  if (cache->seqs) {   // a ragged cache: the same count for every sequence
    int32_t counts[kMaxRaggedBatch];
    for (int b = 0; b < cache->desc.batch; ++b) counts[b] = n_new;
    return kvq_quantize_append_ragged(cache, k_new, v_new, n_new, counts, stream);
  }
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  const int G = cache->desc.group_size;
  const long long r = cache->residual_len;
  const long long T = r + n_new;
  const long long f = (T < 2LL * G) ? 0 : T / G - 1;
  if (cache->quantized_len + f * G > cache->desc.capacity_tokens) return KVQ_ERR_CAPACITY;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(cache->base);
  if (f > 0) {
    FlushParams p{};
    p.kplane[0] = base + cache->off_k_plane[0];
    p.kplane[1] = base + cache->off_k_plane[1];
    p.vplane[0] = base + cache->off_v_plane[0];
    p.vplane[1] = base + cache->off_v_plane[1];
    p.ksz = reinterpret_cast<float*>(base + cache->off_k_sz);
    p.vsz = reinterpret_cast<float*>(base + cache->off_v_sz);
    p.res_k = reinterpret_cast<const uint16_t*>(base + cache->off_res_k);
    p.res_v = reinterpret_cast<const uint16_t*>(base + cache->off_res_v);
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.B = cache->desc.batch;
    p.Hkv = cache->desc.num_kv_heads;
    p.D = cache->desc.head_dim;
    p.G = G;
    p.fmt = cache->desc.format;
    p.C = cache->desc.capacity_tokens;
    p.Lq = cache->quantized_len;
    p.r = static_cast<int>(r);
    p.res_start = cache->residual_start;
    p.n = n_new;
    p.nflush = static_cast<int>(f);
    const long long first_new = std::max(r, f * G);
    p.res_k_w = reinterpret_cast<uint16_t*>(base + cache->off_res_k);
    p.res_v_w = reinterpret_cast<uint16_t*>(base + cache->off_res_v);
    p.first_new = static_cast<int>(first_new);
    p.res_count = static_cast<int>(T - first_new);
    p.ctr = reinterpret_cast<unsigned*>(base + cache->off_res_v + regions(&cache->desc).res);
    // the arrival counters are zero after every flush; zero them before the first
    if (zero_counters_once(cache, p.ctr, s) != KVQ_OK) return KVQ_ERR_CUDA;
    if (launch_flush(p, s) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  const long long first_new = std::max(r, f * G);
  const long long count = T - first_new;
  if (count > 0 && f == 0) {
    ResidualWriteParams w{};
    w.res_k = reinterpret_cast<uint16_t*>(base + cache->off_res_k);
    w.res_v = reinterpret_cast<uint16_t*>(base + cache->off_res_v);
    w.k_new = static_cast<const uint16_t*>(k_new);
    w.v_new = static_cast<const uint16_t*>(v_new);
    w.B = cache->desc.batch;
    w.Hkv = cache->desc.num_kv_heads;
    w.D = cache->desc.head_dim;
    w.G = G;
    w.n = n_new;
    w.r = static_cast<int>(r);
    w.res_start = cache->residual_start;
    w.first_new = static_cast<int>(first_new);
    w.count = static_cast<int>(count);
    if (launch_residual_write(w, s) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  cache->quantized_len += f * G;
  cache->residual_len = static_cast<int32_t>(T - f * G);
  cache->residual_start = static_cast<int32_t>((cache->residual_start + f * G) % (2 * G));
  return KVQ_OK;
}

size_t kvq_workspace_bytes(const kvq_cache* cache, int32_t num_q_heads, int32_t gamma, int32_t top_k) {
  if (!cache_ok(cache)) return 0;
  const int Hkv = cache->desc.num_kv_heads;
  if (num_q_heads < Hkv || num_q_heads % Hkv) return 0;
  if (gamma < 1 || static_cast<long long>(gamma) * (num_q_heads / Hkv) > kMaxRows) return 0;
  if (top_k < 0 || top_k > kMaxTopk) return 0;
  // with a top-k, room for kvq_attend_topk's per-token scores as well
  return kStatusBytes + attend_ws_bytes(&cache->desc) + topk_ws_bytes(&cache->desc, std::max(top_k, 1)) +
         (top_k > 0 ? pre_score_bytes(&cache->desc) : 0);
}

}  // extern "C"

// Every argument check of kvq_attend except the workspace's.  On success sets
// *ws_need to the workspace bytes the call needs.
kvq_status kvq::attend_check(const kvq_cache* cache, int mode, const void* q, int num_q_heads, int gamma,
                             const void* pend_k, const void* pend_v, int n_pend, const int32_t* sel_idx,
                             const void* sel_k, const void* sel_v, int top_k, const void* out, const float* lse,
                             size_t* ws_need) {
  if (!cache || cache->magic != kMagic) return KVQ_ERR_NOT_INITIALIZED;
  if (!valid_desc(&cache->desc)) return KVQ_ERR_INVALID_ARG;
  if (!mode_reads(mode, cache->desc.format)) return KVQ_ERR_UNSUPPORTED;
  const int Hkv = cache->desc.num_kv_heads;
  if (num_q_heads < Hkv || num_q_heads % Hkv || gamma < 1) return KVQ_ERR_INVALID_ARG;
  const int HG = num_q_heads / Hkv;
  if (static_cast<long long>(gamma) * HG > kMaxRows) return KVQ_ERR_UNSUPPORTED;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return KVQ_ERR_INVALID_ARG;
  if (n_pend < 0) return KVQ_ERR_INVALID_ARG;
  if (n_pend > 0 && (n_pend < gamma || !pend_k || !pend_v || !aligned16(pend_k) || !aligned16(pend_v)))
    return KVQ_ERR_INVALID_ARG;
  if (top_k < 0 || top_k > kMaxTopk) return KVQ_ERR_INVALID_ARG;
  if (top_k > 0 && (!sel_idx || !sel_k || !sel_v || !aligned16(sel_idx) || !aligned16(sel_k) ||
                    !aligned16(sel_v)))
    return KVQ_ERR_INVALID_ARG;
  *ws_need = kStatusBytes + attend_ws_bytes(&cache->desc);
  return KVQ_OK;
}

extern "C" {

kvq_status kvq_attend(const kvq_cache* cache, kvq_mode mode, const void* q, int32_t num_q_heads,
                      int32_t gamma, const void* pend_k, const void* pend_v, int32_t n_pend,
                      const int32_t* sel_idx, const void* sel_k, const void* sel_v, int32_t top_k,
                      float sm_scale, void* out, float* lse, void* workspace, size_t ws_bytes,
                      kvq_stream_t stream) {
  size_t need = 0;
  const kvq_status chk = attend_check(cache, mode, q, num_q_heads, gamma, pend_k, pend_v, n_pend, sel_idx, sel_k,
                                      sel_v, top_k, out, lse, &need);
  if (chk != KVQ_OK) return chk;
  if (!workspace || !aligned16(workspace) || ws_bytes < need) return KVQ_ERR_WORKSPACE;
  AttendParams p = make_attend_params(cache, mode, q, num_q_heads, gamma, pend_k, pend_v, n_pend, sel_idx, sel_k,
                                      sel_v, top_k, sm_scale, out, lse, static_cast<uint8_t*>(workspace), false);
  if (p.S_q > attend_splits_max(&cache->desc)) return KVQ_ERR_WORKSPACE;
  if (launch_attend(p, kernel_mode(mode), false, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_attend_topk(const kvq_cache* cache, kvq_mode mode, const void* q, int32_t num_q_heads,
                           int32_t gamma, const void* pend_k, const void* pend_v, int32_t n_pend,
                           const int32_t* sel_idx, const void* sel_k, const void* sel_v, int32_t top_k,
                           float sm_scale, void* out, float* lse, int32_t score_row, int32_t next_k,
                           int32_t* next_idx, float* next_score, void* workspace, size_t ws_bytes,
                           kvq_stream_t stream) {
  size_t need = 0;
  const kvq_status chk = attend_check(cache, mode, q, num_q_heads, gamma, pend_k, pend_v, n_pend, sel_idx, sel_k,
                                      sel_v, top_k, out, lse, &need);
  if (chk != KVQ_OK) return chk;
  if (kernel_mode(mode) == KVQ_MODE_INT8) return KVQ_ERR_UNSUPPORTED;   // no low-bit keys to rank
  if (score_row < 0 || score_row >= gamma) return KVQ_ERR_INVALID_ARG;
  if (next_k < 1 || next_k > kMaxTopk || !next_idx || !aligned16(next_idx)) return KVQ_ERR_INVALID_ARG;
  if (next_score && !aligned16(next_score)) return KVQ_ERR_INVALID_ARG;
  const size_t tk = topk_ws_bytes(&cache->desc, next_k);
  need += tk + pre_score_bytes(&cache->desc);
  if (!workspace || !aligned16(workspace) || ws_bytes < need) return KVQ_ERR_WORKSPACE;
  const long long U = units_of(cache);
  const TopkPlan tp = topk_plan(kernel_mode(mode), cache->desc.head_dim, cache->desc.group_size,
                                cache->quantized_len, U, next_k, true);
  if (static_cast<long long>(tp.S) * next_k > kTopkMaxCand) return KVQ_ERR_UNSUPPORTED;
  if (static_cast<size_t>(tp.S) > static_cast<size_t>(topk_splits_max(&cache->desc, next_k))) return KVQ_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* pre = reinterpret_cast<float*>(ws + kStatusBytes + attend_ws_bytes(&cache->desc) + tk);
  AttendParams p = make_attend_params(cache, mode, q, num_q_heads, gamma, pend_k, pend_v, n_pend, sel_idx, sel_k,
                                      sel_v, top_k, sm_scale, out, lse, ws, true);
  if (p.S_q > attend_splits_max(&cache->desc)) return KVQ_ERR_WORKSPACE;
  p.score_row = score_row;
  p.pre = pre;
  const uint16_t* q_row = static_cast<const uint16_t*>(q) + static_cast<long long>(score_row) * num_q_heads *
                                                               cache->desc.head_dim;
  TopkParams t = make_topk_params(cache, mode, q_row, static_cast<long long>(gamma) * num_q_heads * cache->desc.head_dim,
                                  num_q_heads, next_k, next_idx, next_score, ws, tp);
  t.pre = pre;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_attend(p, kernel_mode(mode), true, s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (launch_topk(t, kernel_mode(mode), true, s) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_attend_plan(const kvq_cache* cache, kvq_mode mode, int32_t num_q_heads, int32_t gamma,
                           int32_t n_pend, int32_t top_k, kvq_attend_plan_info* plan) {
  if (!cache || cache->magic != kMagic) return KVQ_ERR_NOT_INITIALIZED;
  if (!valid_desc(&cache->desc) || !plan) return KVQ_ERR_INVALID_ARG;
  if (!mode_reads(mode, cache->desc.format)) return KVQ_ERR_UNSUPPORTED;
  const int Hkv = cache->desc.num_kv_heads;
  if (num_q_heads < Hkv || num_q_heads % Hkv || gamma < 1 || n_pend < 0 || top_k < 0 || top_k > kMaxTopk)
    return KVQ_ERR_INVALID_ARG;
  if (static_cast<long long>(gamma) * (num_q_heads / Hkv) > kMaxRows) return KVQ_ERR_UNSUPPORTED;
  const AttendPlan pl = plan_attend(cache, mode, gamma * (num_q_heads / Hkv), n_pend, top_k);
  plan->quant_splits = pl.S_q;
  plan->tail_splits = pl.S_t;
  plan->chunk_tokens = pl.chunk;
  plan->cluster = pl.cluster;
  plan->reserved = 0;
  return KVQ_OK;
}

kvq_status kvq_topk(const kvq_cache* cache, kvq_mode mode, const void* q_spec, int32_t num_q_heads,
                    int32_t top_k, int32_t* idx_out, float* score_out, void* workspace, size_t ws_bytes,
                    kvq_stream_t stream) {
  if (!cache || cache->magic != kMagic) return KVQ_ERR_NOT_INITIALIZED;
  if (!valid_desc(&cache->desc)) return KVQ_ERR_INVALID_ARG;
  if (mode == KVQ_MODE_INT8) return KVQ_ERR_UNSUPPORTED;
  if (!mode_reads(mode, cache->desc.format)) return KVQ_ERR_UNSUPPORTED;
  const int Hkv = cache->desc.num_kv_heads;
  if (num_q_heads < Hkv || num_q_heads % Hkv) return KVQ_ERR_INVALID_ARG;
  if (top_k < 1 || top_k > kMaxTopk) return KVQ_ERR_INVALID_ARG;
  if (!q_spec || !idx_out || !aligned16(q_spec) || !aligned16(idx_out)) return KVQ_ERR_INVALID_ARG;
  if (score_out && !aligned16(score_out)) return KVQ_ERR_INVALID_ARG;
  const size_t need = kStatusBytes + attend_ws_bytes(&cache->desc) + topk_ws_bytes(&cache->desc, top_k);
  if (!workspace || !aligned16(workspace) || ws_bytes < need) return KVQ_ERR_WORKSPACE;
  const long long U = units_of(cache);
  const TopkPlan tp = topk_plan(kernel_mode(mode), cache->desc.head_dim, cache->desc.group_size,
                                cache->quantized_len, U, top_k, false);
  if (static_cast<long long>(tp.S) * top_k > kTopkMaxCand) return KVQ_ERR_UNSUPPORTED;
  const size_t Smax = static_cast<size_t>(topk_splits_max(&cache->desc, top_k));
  TopkParams p = make_topk_params(cache, mode, static_cast<const uint16_t*>(q_spec),
                                  static_cast<long long>(num_q_heads) * cache->desc.head_dim, num_q_heads, top_k,
                                  idx_out, score_out, static_cast<uint8_t*>(workspace), tp);
  if (static_cast<size_t>(tp.S) > Smax) return KVQ_ERR_WORKSPACE;
  if (launch_topk(p, kernel_mode(mode), false, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

kvq_status kvq_workspace_status(void* workspace, size_t ws_bytes, kvq_stream_t stream) {
  if (!workspace || ws_bytes < static_cast<size_t>(kStatusBytes)) return KVQ_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (word != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return KVQ_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  return static_cast<kvq_status>(word);
}

kvq_status kvq_selftest_bounded_wait(void* workspace, size_t ws_bytes, int64_t limit_cycles,
                                     kvq_stream_t stream) {
  if (!workspace || !aligned16(workspace) || ws_bytes < static_cast<size_t>(kStatusBytes))
    return KVQ_ERR_WORKSPACE;
  if (limit_cycles < 1 || limit_cycles > (1LL << 31)) return KVQ_ERR_INVALID_ARG;
  if (launch_wait_selftest(static_cast<int*>(workspace), limit_cycles,
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVQ_ERR_CUDA;
  return KVQ_OK;
}

}  // extern "C"
