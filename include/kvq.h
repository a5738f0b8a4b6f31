/*
 * kvq.h: C ABI of the GB300 quantized-KV speculative decode-attention library.
 *
 * The library computes the data-parallel hot path shared by three methods:
 *   - QuantSpec (QuantSpec: Self-Speculative Decoding with Hierarchical Quantized
 *     KV Cache, "Approach"): a hierarchical 4-bit/8-bit KV cache in which the upper
 *     4 bits are the INT4 draft cache and upper+lower 4 bits rebuild the INT8
 *     target cache, plus a double full-precision buffer of 2G recent tokens;
 *   - SpeCache (SpeCache: Speculative Key-Value Caching for Efficient Generation of
 *     LLMs, "Approach"): a 1/2-bit KIVI copy of the KV cache on the GPU, a
 *     speculative token decoded with the output token, and the top-k KV pairs it
 *     predicts, used at 16 bits at the next step;
 *   - MSpecKV (project page, abstract): quantized storage of KV and reconstruction
 *     of only the needed subsets.
 *
 * Entry points: kvq_quantize_append (quantize + append), kvq_attend (fused
 * dequantization + split-K flash-decoding attention with a fused combine) and
 * kvq_topk (per-KV-head top-k under the low-bit keys).
 *
 * Conventions shared by every call:
 *   - Ownership.  The caller owns every buffer: the cache memory handed to
 *     kvq_cache_init, inputs, outputs and the workspace.  The library allocates
 *     no memory.  The only state it keeps is the tuning constants in its code.
 *     A kvq_cache is plain host memory owned by the caller.  It holds device
 *     pointers plus the host-side counters (quantized length, residual fill,
 *     residual start), and kvq_quantize_append updates those counters.
 *   - Asynchrony.  Every call that takes a stream only enqueues work on that
 *     stream (a cudaStream_t passed as void*; NULL = legacy default stream).
 *     None of them synchronizes the device.  Argument errors are returned
 *     before any launch and change nothing.
 *   - Device errors.  Kernels never trap or spin without a bound.  Every wait on
 *     an mbarrier gives up after a bounded time.  A kernel that gives up writes
 *     KVQ_ERR_DEVICE_TIMEOUT into the workspace status word, drains its own
 *     in-flight copies and returns.  kvq_workspace_status reads that word.
 *   - Launch errors are returned as KVQ_ERR_CUDA (from cudaGetLastError).
 *   - Alignment.  Every device pointer must be 16-byte aligned.  The cache memory
 *     must be 256-byte aligned.
 *   - Element types.  bf16 for keys, values and queries (raw 16-bit patterns),
 *     fp32 for scales, zero points, scores and log-sum-exp, int32 for indices.
 *   - Shapes.  head_dim D in {64, 128}.  Group size G in {32, 64, 128} with G
 *     dividing D.  Every sequence of a batch has the same lengths, unless the
 *     cache is ragged (kvq_cache_set_ragged): then each sequence keeps its own
 *     quantized length and residual fill.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* kvq_stream_t; /* a cudaStream_t */

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad shape or count */
  KVQ_ERR_UNSUPPORTED = 2,    /* valid but not built: mode vs format, rows > 8, ... */
  KVQ_ERR_CAPACITY = 3,       /* the append would exceed the quantized capacity */
  KVQ_ERR_WORKSPACE = 4,      /* workspace missing or too small */
  KVQ_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
  KVQ_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up a bounded wait (see above) */
  KVQ_ERR_NOT_INITIALIZED = 7 /* the cache struct was not set up by kvq_cache_init */
} kvq_status;

/* Storage format of the quantized cache. */
typedef enum kvq_format {
  KVQ_FMT_HIER8 = 8, /* hierarchical INT8: upper and lower nibble planes (QuantSpec) */
  KVQ_FMT_INT2 = 2,  /* 2-bit KIVI codes (SpeCache)                                 */
  KVQ_FMT_INT1 = 1   /* 1-bit KIVI codes (SpeCache)                                 */
} kvq_format;

/* Read mode of attention / top-k.  INT8 and INT4 read KVQ_FMT_HIER8: INT8 both
 * nibble planes, INT4 only the upper plane, with scale x16.  So INT4 dequant
 * equals INT8 dequant with the lower nibble zeroed (QuantSpec page, "Approach":
 * the upper 4 bits are the INT4 draft cache).  INT4_MID reads the same upper
 * plane but puts each draft code at the middle of the sixteen 8-bit codes it
 * stands for: its dequant equals INT8 dequant with the lower nibble set to 8,
 * i.e. zero point z + 8 s with the 8-bit scale s (the pages do not say where
 * the draft value lies; this halves the worst-case draft error, 8.5 steps of
 * s against 15.5).  INT2 and INT1 read their own format.  INT1_CENTER reads
 * KVQ_FMT_INT1 with the levels at the centres of the two halves of each
 * group's [min, max]: zero point z + s/4 and scale s/2, with the stored 1-bit
 * scale s = max - min and the same codes (SpeCache page, "Approach", gives
 * 1-bit KIVI a new zero point and scale but no formula; this is the library's
 * reading: for values spread evenly over the range it cuts the mean squared
 * error by four).  Any other pairing returns KVQ_ERR_UNSUPPORTED. */
typedef enum kvq_mode {
  KVQ_MODE_INT8 = 0,
  KVQ_MODE_INT4 = 1,
  KVQ_MODE_INT2 = 2,
  KVQ_MODE_INT1 = 3,
  KVQ_MODE_INT4_MID = 4,
  KVQ_MODE_INT1_CENTER = 5
} kvq_mode;

typedef struct kvq_cache_desc {
  int32_t batch;           /* B  >= 1                                             */
  int32_t num_kv_heads;    /* Hkv >= 1                                            */
  int32_t head_dim;        /* D  in {64, 128}                                     */
  int32_t group_size;      /* G  in {32, 64, 128}, G divides D                    */
  int32_t format;          /* kvq_format                                          */
  int32_t reserved0;       /* must be 0                                           */
  int64_t capacity_tokens; /* C: max quantized tokens per sequence, multiple of G */
} kvq_cache_desc;

/*
 * One layer's cache.  Device layout, all regions inside the caller's memory at
 * 256-byte aligned offsets, with u = b*Hkv + kvh:
 *
 *  key planes    [u][C][D*pb/8] u8, token-major.  Byte j of token row t packs
 *                channels (8/pb)*j + e at bits [pb*e, pb*e+pb).  For HIER8 there
 *                are two planes with pb = 4: upper nibbles (INT4 draft code) and
 *                lower nibbles.  For INT2 and INT1 there is one plane with
 *                pb = 2 or 1.
 *  value planes  [u][C/32][D][32*pb/8] u8, in 32-token slabs.  Slab s, row d
 *                holds the codes of channel d for tokens 32s..32s+31.  Byte j
 *                packs tokens 32s + (8/pb)*j + e at bits [pb*e, pb*e+pb).  Same
 *                planes as the keys.
 *  key scale/zero   [u][C/G][2][D] f32: per (token group, channel), scale row
 *                   then zero-point row.
 *  value scale/zero [u][C][2][D/G] f32: per (token, block of G channels),
 *                   scales then zero points.
 *  residual K, V [u][2G][D] bf16: the double buffer of recent tokens.  The r
 *                live tokens sit in slots (residual_start + i) mod 2G, i in [0, r),
 *                oldest first.  residual_start is 0 or G.  At a flush the older
 *                half is quantized in place, and the other half becomes the
 *                oldest.
 *  flush counters [u] u32: arrival counters of the quantize-append kernel
 *                (zeroed on the stream before the cache's first flush, zero
 *                again after every append).
 *
 * Codes (KIVI-style asymmetric min/max, fp32, round-half-even): scale =
 * (max - min)/(2^b - 1), code = clamp(rint((x - min) * (1/scale)), 0, 2^b - 1),
 * with zero point = min.  A constant group gets scale 0 and codes 0.  Keys are
 * grouped per channel over G tokens, values per token over G channels.
 */
/* Per-sequence state of a ragged cache (see kvq_cache_set_ragged): the same
 * three counters as the uniform ones in kvq_cache, for one sequence. */
typedef struct kvq_seq_state {
  int64_t quantized_len;      /* Lq of this sequence (multiple of G)              */
  int32_t residual_len;       /* r of this sequence, 0 <= r < 2G                   */
  int32_t residual_start;     /* 0 or G                                            */
} kvq_seq_state;

typedef struct kvq_cache {
  kvq_cache_desc desc;
  void* base;                 /* caller's device memory                            */
  uint64_t bytes;             /* its size                                          */
  uint64_t off_k_plane[2];    /* key planes: [0] upper/only, [1] lower (HIER8)     */
  uint64_t off_v_plane[2];    /* value planes, same order                          */
  uint64_t off_k_sz;          /* key scale/zero                                    */
  uint64_t off_v_sz;          /* value scale/zero                                  */
  uint64_t off_res_k;         /* residual keys                                     */
  uint64_t off_res_v;         /* residual values                                   */
  int64_t quantized_len;      /* Lq: quantized tokens per sequence (multiple of G) */
  int32_t residual_len;       /* r: live residual tokens, 0 <= r < 2G              */
  int32_t residual_start;     /* 0 or G                                            */
  uint32_t magic;             /* set by kvq_cache_init                             */
  uint32_t flags;             /* library-owned: bit 0 set once the flush counters
                                 have been zeroed on the device                    */
  kvq_seq_state* seqs;        /* NULL: uniform lengths; else [batch] per-sequence state
                                 (caller-owned host memory, see kvq_cache_set_ragged) */
} kvq_cache;

/* Human-readable name of a status code (static string, never NULL).  The pages
 * have no counterpart: this is part of the library's error reporting. */
const char* kvq_status_string(kvq_status s);

/* Bytes of device memory a cache with this descriptor needs (0 if the descriptor
 * is invalid).  The pages have no counterpart: they give no storage layout, and
 * this one is the library's own (see the layout above). */
size_t kvq_cache_bytes(const kvq_cache_desc* desc);

/* Lay out a cache in caller memory `dev_mem` (>= kvq_cache_bytes, 256-B aligned)
 * and set it empty (Lq = r = 0).  Writes only the host struct: the device
 * memory's contents are ignored until written by kvq_quantize_append.  The
 * pages have no counterpart: it sets up the library's own layout.  Errors:
 * KVQ_ERR_INVALID_ARG for a null struct, an invalid descriptor, null or
 * misaligned memory, or fewer bytes than kvq_cache_bytes. */
kvq_status kvq_cache_init(kvq_cache* cache, const kvq_cache_desc* desc, void* dev_mem,
                          size_t bytes);

/*
 * Make an empty cache ragged: every sequence of the batch keeps its own
 * quantized length, residual fill and residual start, in `seqs`, an array of
 * `count` == batch entries of caller-owned host memory that must outlive the
 * cache's use (SpeCache page, "Key results": batched decoding, 36 sequences at
 * 32K, where real sequences have unequal lengths).  The entries are set to
 * empty.  From then on kvq_quantize_append_ragged appends a different number
 * of tokens to each sequence, kvq_quantize_append appends the same number to
 * all, and kvq_attend, kvq_attend_plan and kvq_topk read each sequence's own
 * lengths: query row i of sequence b sees its quantized tokens [0, Lq_b), its
 * r_b residual tokens and the pending tokens, exactly as a batch of one.  The
 * cache-level quantized_len and residual_len then hold the largest of the
 * sequences' values (for sizing); residual_start is unused.
 * Errors: KVQ_ERR_NOT_INITIALIZED; KVQ_ERR_INVALID_ARG for a null array,
 * count != batch, or a cache that is not empty; KVQ_ERR_UNSUPPORTED for a
 * batch above 64 (the per-sequence lengths travel in the kernels' parameter
 * block).  Writes host memory only.
 */
kvq_status kvq_cache_set_ragged(kvq_cache* cache, kvq_seq_state* seqs, int32_t count);

/*
 * Append n_new tokens of every sequence.  k_new and v_new are bf16
 * [B][Hkv][n_new][D], contiguous, on the device.
 *
 * The double full-precision buffer (QuantSpec page, "Approach") works token by
 * token.  The token goes to residual slot r and r += 1.  When r reaches 2G, the
 * oldest G residual tokens are quantized as token group [Lq, Lq+G), Lq += G and
 * r = G.  After N tokens from empty: Lq = G*(floor(N/G) - 1) once N >= 2G.  A
 * multi-token call gives the same bytes as n single-token calls.  All complete
 * groups are quantized in one launch, which is the bulk path for a prefill.
 * Speculative tokens never enter the cache: pass them to kvq_attend as pending
 * tokens, and append only the accepted ones, so rollback needs no undo.
 *
 * Capacity is checked before anything is enqueued (KVQ_ERR_CAPACITY).  Enqueues
 * at most two kernels.  The host counters are updated at once, so later calls
 * on the same stream see the new state.
 */
kvq_status kvq_quantize_append(kvq_cache* cache, const void* k_new, const void* v_new,
                               int32_t n_new, kvq_stream_t stream);

/*
 * Append to each sequence of a ragged cache its own number of tokens:
 * sequence b appends n_new[b] (0 <= n_new[b] <= n_max) tokens, the first
 * n_new[b] rows of k_new / v_new, bf16 [B][Hkv][n_max][D] (rows past n_new[b]
 * are not read).  n_new is host memory.  Each sequence runs the double-buffer
 * state machine of kvq_quantize_append on its own state (QuantSpec page,
 * "Approach": the 2G full-precision buffer), so sequence b ends with the same
 * bytes as a batch-of-one cache that appended the same tokens.  Capacity is
 * checked for every sequence before anything is enqueued (KVQ_ERR_CAPACITY,
 * nothing changed); KVQ_ERR_INVALID_ARG for a cache that is not ragged, a null
 * n_new, or a count outside [0, n_max].  Enqueues at most two kernels (one
 * flush launch for the sequences that flush, one residual copy for those that
 * do not) and updates the per-sequence host state at once.
 */
kvq_status kvq_quantize_append_ragged(kvq_cache* cache, const void* k_new, const void* v_new,
                                      int32_t n_max, const int32_t* n_new, kvq_stream_t stream);

/* Bytes of workspace that kvq_attend / kvq_topk need for this cache, at any fill
 * up to capacity, on the current device (the split count grows with its SM
 * count; a workspace sized on a device with fewer SMs can be too small, which a
 * call reports as KVQ_ERR_WORKSPACE).  Rows per KV head R = gamma * num_q_heads /
 * num_kv_heads must be <= 8.  top_k <= 1024.  The workspace must be zero-filled
 * once before its first use.  Every call that finishes leaves it reusable.
 * Returns 0 for invalid arguments.  The pages have no counterpart: the
 * workspace holds the split-K partials and the merge's ticket counters of the
 * library's own launch design. */
size_t kvq_workspace_bytes(const kvq_cache* cache, int32_t num_q_heads, int32_t gamma,
                           int32_t top_k);

/*
 * Decode attention of gamma query tokens over the cache (QuantSpec page,
 * "Approach": the draft reads INT4, the target verifies with INT8; SpeCache page,
 * "Approach": attention over the low-bit copy, with the top-k tokens at 16 bits).
 *
 *  q        bf16 [B][gamma][Hq][D].  Query head h reads KV head h / (Hq/Hkv).
 *  pend_k/v bf16 [B][Hkv][n_pend][D]: speculative tokens not yet committed.
 *           Query token i sees pending token p iff p <= n_pend - gamma + i (the
 *           gamma queries are the last gamma pending tokens).  n_pend = 0 means no
 *           pending tokens (pointers may be NULL).  Otherwise n_pend >= gamma.
 *  sel_idx  int32 [B][Hkv][top_k], sel_k/v bf16 [B][Hkv][top_k][D].  An entry
 *           with 0 <= idx < Lq replaces quantized token idx by the given 16-bit
 *           key and value.  Other entries are ignored (-1 pads).  Valid entries
 *           of a (b, kvh) must be distinct.  top_k = 0 means none (NULL allowed).
 *  sm_scale logits are sm_scale * q.k.  A value <= 0 selects 1/sqrt(D).
 *  out      bf16 [B][gamma][Hq][D] (written).
 *  lse      fp32 [B][gamma][Hq] natural-log softmax denominators, or NULL.  A
 *           query that sees no key gets out = 0 and lse = -inf.
 *  Every residual token is visible to every query.  Results do not depend on
 *  how the work is split.
 * Enqueues one kernel.  It splits the quantized context over CTAs and runs one
 * or more CTAs per (b, kvh) for the bf16 tail (kvq_attend_plan reports the
 * split).  When the CTAs of a (b, kvh) number at most 16 and their clusters fit
 * the device as well as plain CTAs would, they run as one thread-block cluster
 * and merge their partials through shared memory; otherwise the partials go to
 * the workspace and whichever CTA of the (b, kvh) finishes last merges them.
 * Setting the environment variable KVQ_ATTEND_CLUSTERS=0 (read on every call)
 * selects the second way for every launch.
 */
kvq_status kvq_attend(const kvq_cache* cache, kvq_mode mode, const void* q, int32_t num_q_heads,
                      int32_t gamma, const void* pend_k, const void* pend_v, int32_t n_pend,
                      const int32_t* sel_idx, const void* sel_k, const void* sel_v, int32_t top_k,
                      float sm_scale, void* out, float* lse, void* workspace, size_t ws_bytes,
                      kvq_stream_t stream);

/*
 * kvq_attend plus the next step's top-k, from one read of the low-bit keys
 * (SpeCache page, "Approach": the speculative token decoded with the output
 * token predicts the next step's top-k KV pairs; "Measured effects": the
 * speculative fetch against output-token-based, non-speculative fetching).
 * The attention pass scores every quantized token with the summed query of
 * query row `score_row` (1: the speculative token of a gamma = 2 SpeCache step;
 * 0: the output token, the non-speculative variant) while it streams the keys,
 * and a selection pass then picks the next_k best per KV head.
 *  All kvq_attend arguments, with kvq_attend's meaning and results (out, lse).
 *  mode        KVQ_MODE_INT4, INT4_MID, INT2, INT1 or INT1_CENTER (INT8 returns
 *              KVQ_ERR_UNSUPPORTED: the hierarchical cache is ranked by its
 *              4-bit draft code).
 *  score_row   0 <= score_row < gamma.
 *  next_k      1..1024; next_idx int32 [B][Hkv][next_k] (device), next_score
 *              fp32, same shape, or NULL.  Identical to kvq_topk(cache, mode,
 *              q[:, score_row], num_q_heads, next_k, ...): same indices, same
 *              score bits, same order and padding.
 *  workspace   at least kvq_workspace_bytes(cache, num_q_heads, gamma, next_k),
 *              which holds the per-token scores between the two passes.
 * Enqueues two kernels.  Errors as kvq_attend and kvq_topk, returned before
 * any launch.
 */
kvq_status kvq_attend_topk(const kvq_cache* cache, kvq_mode mode, const void* q, int32_t num_q_heads,
                           int32_t gamma, const void* pend_k, const void* pend_v, int32_t n_pend,
                           const int32_t* sel_idx, const void* sel_k, const void* sel_v, int32_t top_k,
                           float sm_scale, void* out, float* lse, int32_t score_row, int32_t next_k,
                           int32_t* next_idx, float* next_score, void* workspace, size_t ws_bytes,
                           kvq_stream_t stream);

/*
 * How kvq_attend would split a call with these arguments on the current
 * device.  The paper has no counterpart: this reports the launch plan.
 *  plan->quant_splits  CTAs per (b, kvh) over the quantized context (0 if empty)
 *  plan->tail_splits   CTAs per (b, kvh) for the bf16 tail (0: the quantized
 *                      splits share it out)
 *  plan->chunk_tokens  quantized tokens per split (a multiple of 128)
 *  plan->cluster       1 when each (b, kvh) runs as one thread-block cluster
 * Arguments are checked as kvq_attend checks them; nothing is enqueued.
 */
typedef struct kvq_attend_plan_info {
  int32_t quant_splits;
  int32_t tail_splits;
  int64_t chunk_tokens;
  int32_t cluster;
  int32_t reserved;
} kvq_attend_plan_info;

kvq_status kvq_attend_plan(const kvq_cache* cache, kvq_mode mode, int32_t num_q_heads, int32_t gamma,
                           int32_t n_pend, int32_t top_k, kvq_attend_plan_info* plan);

/*
 * Per KV head, the top_k quantized tokens that score highest under the
 * low-bit keys for the speculative token's query (SpeCache page, "Approach").
 * The query heads sharing a KV head are summed in fp32, in ascending head order.
 * Per key group g the score is exact up to stated roundings:
 *   w_d = fp32(qs_d * s_d)   (s = the mode's key scale: x16 for INT4 and INT4_MID,
 *                            x1/2 for INT1_CENTER; INT4_MID's zero point is
 *                            fp32(zero_d + 8 s_d), INT1_CENTER's fp32(zero_d + s_d/4)
 *                            with the stored scale s_d)
 *   e   = exponent with max_d|w_d| < 2^e, floored at -100
 *   W_d = rint(w_d * 2^(21-e)),  S_t = sum_d W_d * code_{t,d} (exact integer)
 *   p_d = fp32(qs_d * zero_d), f = exponent with max_d|p_d| < 2^f, floored at -80
 *   beta = fp32(sum_d rint(p_d * 2^(40-f))) * 2^(f-40)   (an exact integer sum)
 *   score_t = fp32(fp32(fp32(S_t) * 2^(e-21)) + beta)
 * Tokens are ordered by (score descending, index ascending).  Positions beyond
 * Lq get index -1 and score -inf.
 *  mode     KVQ_MODE_INT4, INT4_MID, INT2, INT1 or INT1_CENTER (INT8 returns
 *           KVQ_ERR_UNSUPPORTED).
 *  q_spec   bf16 [B][Hq][D].
 *  idx_out  int32 [B][Hkv][top_k], in that order.  score_out fp32, same shape,
 *           or NULL.
 *  1 <= top_k <= 1024, and ceil(Lq / 8192) * top_k <= 4096 (each split scores
 *  at most 8192 tokens and the merge holds at most 4096 candidates); a cache
 *  beyond that returns KVQ_ERR_UNSUPPORTED.  Enqueues one kernel.
 */
kvq_status kvq_topk(const kvq_cache* cache, kvq_mode mode, const void* q_spec,
                    int32_t num_q_heads, int32_t top_k, int32_t* idx_out, float* score_out,
                    void* workspace, size_t ws_bytes, kvq_stream_t stream);

/*
 * kvq_attend for callers that cannot allocate device memory.  The paper has no
 * counterpart: this is a deployment variant.  A decode loop that must not
 * allocate after start-up is one such caller: an allocation can synchronize
 * the device or disturb a pre-reserved memory pool.  A host integration with no
 * device allocator of its own is another.
 *
 * Same arguments and results as kvq_attend, minus the workspace.  The workspace
 * is a fixed 16 MiB array compiled into the library, so the call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).  Every GPU
 * that loads the library holds that array until the process exits.
 *  - Limit: the attention workspace kvq_attend would need for this cache
 *    (256 bytes of status word, the ticket counters and the split partials)
 *    must be at most 16 MiB.  Otherwise the call returns KVQ_ERR_WORKSPACE and
 *    enqueues nothing.  Every other argument error returns kvq_attend's status
 *    code, also before anything is enqueued.
 *  - Set-up: the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it.  With CUDA's
 *    lazy module loading, that lookup may load the library's device code and
 *    reserve the array on the device, which can synchronize it.  Make that first
 *    call during start-up, before any stream capture.
 *  - Sharing: every call uses the same array and leaves its last contents there.
 *    Each call clears the ticket counters it needs on `stream` first.  Calls
 *    that overlap on the GPU (other streams, other threads) race on the array:
 *    issue them in order on one stream.
 *  - Device timeouts are recorded in the array's status word, which this entry
 *    point does not report.
 */
kvq_status kvq_attend_static_scratch(const kvq_cache* cache, kvq_mode mode, const void* q,
                                     int32_t num_q_heads, int32_t gamma, const void* pend_k,
                                     const void* pend_v, int32_t n_pend, const int32_t* sel_idx,
                                     const void* sel_k, const void* sel_v, int32_t top_k,
                                     float sm_scale, void* out, float* lse, kvq_stream_t stream);

/*
 * Fetch of the selected tokens' 16-bit K/V from the full-precision store, for
 * kvq_attend's sel_k / sel_v (SpeCache page, "Approach": the full 16-bit
 * cache lives in CPU memory and the top-k pairs the speculative token
 * predicts are fetched for the next step; MSpecKV page, abstract: offloaded
 * KV is reconstructed only in the needed subsets).  The kernel reads pinned
 * host memory directly (over NVLink-C2C on a Grace-Blackwell node).
 *  full_k, full_v  bf16 [B][Hkv][full_tokens][D]: pinned host memory
 *                  (cudaHostAlloc / cudaHostRegister, e.g. a torch pinned
 *                  tensor) or device memory; 16-byte aligned.  The caller
 *                  guarantees that extent.  Pageable host memory returns
 *                  KVQ_ERR_INVALID_ARG before any launch.
 *  sel_idx         int32 [B][Hkv][top_k], device memory (e.g. kvq_topk's
 *                  idx_out).  Entry j of (b, kvh) copies row sel_idx[b][kvh][j]
 *                  of that head; an index outside [0, full_tokens) (the -1
 *                  padding) gives a zero row.
 *  sel_k, sel_v    bf16 [B][Hkv][top_k][D], device memory, 16-byte aligned.
 *  D in {64, 128}; 1 <= top_k <= 1024.  Bit-exact copy.  Enqueues one kernel
 *  on `stream` and returns without waiting.
 */
kvq_status kvq_gather_selected(const void* full_k, const void* full_v, int64_t full_tokens, int32_t batch,
                               int32_t num_kv_heads, int32_t head_dim, const int32_t* sel_idx, int32_t top_k,
                               void* sel_k, void* sel_v, kvq_stream_t stream);

/* Synchronously read (and then clear) the device status word of a workspace:
 * KVQ_OK, or KVQ_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait since the
 * last read.  Synchronizes `stream`. */
kvq_status kvq_workspace_status(void* workspace, size_t ws_bytes, kvq_stream_t stream);

/* Self-test of the bounded-wait path.  Launches one CTA that waits on an
 * mbarrier that nothing ever arrives at, with a limit of `limit_cycles` SM
 * clocks (1..2^31).  On giving up it records KVQ_ERR_DEVICE_TIMEOUT in the
 * workspace status word and returns, so kvq_workspace_status then reports
 * it.  It neither traps nor hangs. */
kvq_status kvq_selftest_bounded_wait(void* workspace, size_t ws_bytes, int64_t limit_cycles,
                                     kvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
