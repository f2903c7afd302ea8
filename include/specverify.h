/*
 * specverify.h -- C ABI of libspecverify.so: the target-model verification step of
 * speculative decoding on one NVIDIA GB300 (sm_103a).
 *
 * Sources (page title, then section):
 *   "Co-Designing AI Models Using Speculative Decoding for Faster LLM Inference"
 *   (summary page), "basic structure": a drafter proposes D tokens, the target verifies
 *   them in parallel and keeps them up to the first mismatch; the acceptance length AL
 *   lies in [1, 1+D]. Same page, guideline 2: with GQA group size G = Hq / Hkv the
 *   verify attention has G * (1 + D) query rows per KV head.
 *   "GPU and LLM, chapter 5": "FlashAttention" and "Online softmax" (the score table is
 *   processed tile by tile in on-chip memory with a running max m and sum l, never
 *   written to HBM); "GQA" (groups of query heads share one K/V head); "Speculative
 *   decoding (2)" (one forward over the k+1 positions; the target's own token replaces
 *   the first rejected draft).
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller, unless stated otherwise.
 *     The library keeps no pointer after a call returns and allocates no device memory:
 *     scratch space is the caller's `workspace`.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream). Host-side checks cover sizes, pointers and alignment only: device arrays
 *     (lengths, tokens) are never read on the host, so no call synchronises.
 *   - Device-side checks (a length beyond its stated maximum, packed sizes beyond the
 *     buffers) make the kernels skip all work and leave outputs untouched; they set a
 *     sticky flag in the workspace that sv_workspace_status() reports.
 *   - A workspace must be zero-filled once before its first use (the flags live in its
 *     first 256 bytes; spec_accept also keeps a completion counter and one key per row
 *     there, which every call leaves at zero) and may be reused by later calls of the
 *     same entry point on the same stream. Two calls that run concurrently must not
 *     share a workspace.
 *   - Return value: SV_OK or an error code; nothing is printed and nothing is thrown.
 *
 * Packed ragged layout (uniform batches are the special case with equal lengths):
 *   for sequence b with cached prefix T_b = seq_lens[b] and draft length D_b = draft_len[b],
 *   W_b = 1 + D_b window rows. Window row 0 is the last accepted token, rows 1..D_b the
 *   drafts. Sequences are stored back to back in batch order:
 *     q, out        [sum_b W_b,         Hq,  d]  rows q_off[b] .. q_off[b] + D_b
 *     k/v cache     [sum_b (T_b + W_b), Hkv, d]  rows kv_off[b] .. kv_off[b] + T_b + D_b
 *   The caller has already written the window's K/V rows at cache positions T_b..T_b+D_b
 *   (the verify forward appends them before attention, as a prefill does).
 *   Window row i attends to cache positions 0..T_b+i inclusive (window-causal mask).
 *   Query head h uses KV head h / G.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SV_API __attribute__((visibility("default")))
#else
#define SV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_NULL = 1,        /* a required pointer is NULL */
  SV_ERR_SHAPE = 2,       /* a size is out of range or inconsistent */
  SV_ERR_DTYPE = 3,       /* unsupported dtype */
  SV_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
  SV_ERR_WORKSPACE = 5,   /* workspace too small */
  SV_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
  SV_ERR_TIMEOUT = 7,     /* a device-side wait gave up (reported by sv_workspace_status) */
  SV_ERR_DEVICE_SHAPE = 8 /* device-side length check failed (sv_workspace_status) */
} sv_status;

typedef enum { SV_BF16 = 0, SV_FP8_E4M3 = 1, SV_FP32 = 2 } sv_dtype;

/* Shape of one spec_verify_attn call. */
typedef struct {
  int32_t batch;          /* B >= 0 (0: nothing to do) */
  int32_t num_q_heads;    /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;   /* Hkv >= 1 */
  int32_t head_dim;       /* d: 64 or 128 */
  int32_t max_draft_len;  /* upper bound on every D_b, 0 <= D_b <= max_draft_len <= 255 */
  int32_t max_seq_len;    /* upper bound on every T_b, <= 2^31 - 1025 */
  int64_t q_rows;         /* rows allocated in q and out, >= sum_b (1 + D_b) */
  int64_t kv_rows;        /* rows allocated in k_cache and v_cache, >= sum_b (T_b+1+D_b),
                             <= 2^31 - 1025 */
  int32_t kv_dtype;       /* SV_BF16, or SV_FP8_E4M3 (OCP E4M3 codes) */
  float softmax_scale;    /* scale on q.k; 0 selects 1/sqrt(head_dim) */
  int32_t sliding_window; /* 0: every earlier key; W >= 1: sliding-window attention over
                             the W most recent positions (see spec_verify_attn) */
} sv_attn_desc;

/* Bytes of workspace spec_verify_attn needs for `desc` on the CURRENT CUDA device
 * (the split-KV partial results depend on its SM count). Returns 0 if desc is invalid. */
SV_API size_t spec_verify_attn_workspace_size(const sv_attn_desc* desc);

/*
 * spec_verify_attn -- GQA verify attention over the cached prefix plus the draft window.
 *
 * For every sequence b, KV head g, query head h in [g*G, (g+1)*G) and window row
 * i in [0, D_b]:
 *   s_j = scale * q[q_off[b]+i, h, :] . K[kv_off[b]+j, g, :],   j = lo .. T_b + i
 *   out[q_off[b]+i, h, :] = sum_j softmax(s)_j * V[kv_off[b]+j, g, :]
 * computed tile by tile with the online-softmax update, so no score table reaches HBM.
 * lo = 0, or with sliding_window = W >= 1, lo = max(0, T_b + i - W + 1): the query at
 * position T_b + i sees the W most recent positions, itself included ("GPU and LLM,
 * chapter 5", "Sliding window: do not keep the distant past"). Key tiles wholly before
 * a unit's window are skipped, so a call reads about min(T_b + 1 + D_b, W + D_b) cache
 * rows per sequence and KV head. Cache rows of positions before T_b - W + 1 are never
 * used and may hold any bits (they may be reclaimed).
 *
 *   q        bf16 [q_rows, Hq, d]
 *   k_cache  bf16 or E4M3 codes [kv_rows, Hkv, d]; v_cache likewise
 *   seq_lens int32 [B] = T_b (prefix length, excluding the window)
 *   draft_len int32 [B] = D_b
 *   kv_scale fp32 [2, Hkv] for SV_FP8_E4M3 (row 0 scales K, row 1 scales V: the real
 *            value of a code c is e4m3(c) * scale); must be NULL for SV_BF16
 *   out      bf16 [q_rows, Hq, d]; only the sum_b W_b packed rows are written
 *   workspace >= spec_verify_attn_workspace_size(desc) bytes, 256-byte aligned
 * q, k_cache, v_cache and out must be 16-byte aligned.
 */
SV_API sv_status spec_verify_attn(const sv_attn_desc* desc, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* seq_lens,
                           const int32_t* draft_len, const float* kv_scale, void* out,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * spec_verify_attn_host_lengths -- spec_verify_attn for callers that also hold the
 * lengths in host memory (an engine's scheduler usually does). The work plan (units,
 * their tiles, each CTA's range) is computed on the host from seq_lens_host and
 * draft_len_host and passed with the attention kernel's launch, so no planning kernel
 * runs on the GPU before the attention kernel (about 6 us per call on the workloads
 * measured). Same arguments, layouts and results as spec_verify_attn, plus:
 *   seq_lens_host, draft_len_host  int32 [B] in HOST memory, equal to seq_lens and
 *                                  draft_len (which are still read on the device)
 * Lengths out of range are reported at once with SV_ERR_SHAPE (host-side check). When
 * the tcgen05 kernel is not used, or the batch is beyond the host plan's capacity (256
 * sequences, 640 units of 128 query rows, 192 CTAs), the call plans on the device
 * exactly like spec_verify_attn.
 */
SV_API sv_status spec_verify_attn_host_lengths(const sv_attn_desc* desc, const void* q,
                                        const void* k_cache, const void* v_cache,
                                        const int32_t* seq_lens, const int32_t* draft_len,
                                        const int32_t* seq_lens_host,
                                        const int32_t* draft_len_host, const float* kv_scale,
                                        void* out, void* workspace, size_t workspace_bytes,
                                        void* stream);

/*
 * spec_verify_attn_paged -- spec_verify_attn over a paged KV cache ("GPU and LLM, chapter 5",
 * "PagedAttention (2): manage with fixed-size pages": the cache is cut into blocks of a
 * fixed number of positions placed anywhere in a pool, and a per-sequence block table
 * records where each block is).
 *
 * The result is that of spec_verify_attn (sliding_window included) with the cache row of
 * position j of sequence b (j = 0 .. T_b + D_b) read from
 *   k_pages[block_table[b * max_blocks_per_seq + j / block_size], j % block_size, g, :]
 * (v_pages likewise). The caller has written the window's K/V (positions T_b .. T_b + D_b)
 * into the pool before the call, as for the packed cache.
 *
 *   k_pages, v_pages  bf16 or E4M3 codes [num_blocks, block_size, Hkv, d], 16-byte aligned
 *   num_blocks        blocks in the pool, >= 1; num_blocks * block_size <= 2^31 - 1025
 *   block_size        positions per block: a power of two in [8, 65536]
 *   block_table       int32 [B, max_blocks_per_seq], row-major, 4-byte aligned; entries
 *                     for logical blocks 0 .. (T_b + D_b) / block_size must name blocks of
 *                     the pool, except, under a sliding window, blocks holding only
 *                     positions before T_b - W + 1, which are never read (they may be
 *                     reclaimed and their entries hold anything); later entries are
 *                     never read
 * desc->kv_rows is ignored. The workspace is that of spec_verify_attn for the same desc.
 * A sequence needing more than max_blocks_per_seq blocks, or a table entry outside
 * [0, num_blocks) that must be read, is reported by sv_workspace_status (SV_ERR_DEVICE_
 * SHAPE); such an entry reads as zeros and no memory outside the pool is touched.
 */
SV_API sv_status spec_verify_attn_paged(const sv_attn_desc* desc, const void* q,
                                 const void* k_pages, const void* v_pages, int64_t num_blocks,
                                 int32_t block_size, const int32_t* block_table,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 const int32_t* draft_len, const float* kv_scale, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace spec_accept needs on the current CUDA device. 0 if invalid. */
SV_API size_t spec_accept_workspace_size(int32_t batch, int32_t max_draft_len, int32_t vocab);

/*
 * spec_accept -- greedy acceptance of the drafts.
 *
 * For every window row r the target's greedy token is amax[r] = the smallest index
 * attaining max(logits[r, :]) (exact comparison; -0.0 ties +0.0; NaN never wins).
 * For sequence b: n_b = the number of leading positions j < D_b with
 * draft_tokens[d_off[b] + j] == amax[q_off[b] + j]; accept_len[b] = n_b + 1 (in
 * [1, 1 + D_b]); next_token[b] = amax[q_off[b] + n_b] (the target's token at the first
 * mismatch, or the bonus token after D_b accepted drafts).
 *
 *   logits       bf16 or fp32 [sum_b (1 + D_b), vocab], row q_off[b] + j is the target's
 *                prediction after window token j of sequence b
 *   draft_tokens int32 [sum_b D_b] packed, d_off[b] = sum_{b'<b} D_b'
 *   draft_len    int32 [B]
 *   accept_len, next_token int32 [B] (outputs)
 *   target_tokens int32 [sum_b (1 + D_b)] (optional output, may be NULL): amax per row
 *   workspace >= spec_accept_workspace_size(batch, max_draft_len, vocab) bytes
 */
SV_API sv_status spec_accept(int32_t batch, int32_t max_draft_len, int32_t vocab,
                      int32_t logits_dtype, const void* logits, const int32_t* draft_tokens,
                      const int32_t* draft_len, int32_t* accept_len, int32_t* next_token,
                      int32_t* target_tokens, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * spec_accept_noalloc -- spec_accept without a workspace argument. It has no counterpart
 * on the pages: it exists for callers that cannot allocate device memory per call, such
 * as inference engines that reserve all device memory once at start-up and pass each
 * operator only its inputs and outputs, leaving nowhere to put per-call scratch.
 *
 * Arguments, results and device-side checks are those of spec_accept. The scratch lives
 * in a device array of SV_ACCEPT_NOALLOC_MAX_WORKSPACE bytes compiled into the library:
 *   - every GPU that loads the library holds that memory until the process exits;
 *   - a shape whose spec_accept_workspace_size() exceeds it is rejected with
 *     SV_ERR_WORKSPACE and nothing is launched (512 KiB covers 43,000 window rows);
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and caches it with the id of the
 *     device's current context; a call in a new context (after cudaDeviceReset, say)
 *     looks it up again. Make the first call in each context before any stream capture;
 *   - all calls share the array and it keeps the last call's contents: two calls that can
 *     run at the same time on the GPU (different streams or host threads) race and may
 *     return wrong tokens;
 *   - device-side length errors leave the outputs untouched and cannot be read back
 *     (there is no workspace to pass to sv_workspace_status): pre-fill accept_len with 0
 *     to detect them.
 * Calls no cudaMalloc, cudaFree or allocating routine.
 */
#define SV_ACCEPT_NOALLOC_MAX_WORKSPACE (512u * 1024u)
SV_API sv_status spec_accept_noalloc(int32_t batch, int32_t max_draft_len, int32_t vocab,
                                     int32_t logits_dtype, const void* logits,
                                     const int32_t* draft_tokens, const int32_t* draft_len,
                                     int32_t* accept_len, int32_t* next_token,
                                     int32_t* target_tokens, void* stream);

/* Bytes of workspace spec_accept_stochastic needs (256: the flag word). 0 if invalid. */
SV_API size_t spec_accept_stochastic_workspace_size(int32_t batch, int32_t max_draft_len,
                                                   int32_t vocab);

/*
 * spec_accept_stochastic -- acceptance for sampled decoding that leaves the distribution
 * of the output that of the target model alone ("GPU and LLM, chapter 5", "Speculative
 * decoding (2)"; the rule of Leviathan, Kalman and Matias, "Fast Inference from
 * Transformers via Speculative Decoding", 2023, which that page cites).
 *
 * For sequence b, with p_j the softmax of target row j and q_j that of draft row j (logits
 * divided by `temperature`), and x_j the drafted tokens:
 *   draft j is kept iff u_accept[j] * q_j(x_j) < p_j(x_j), for j = 0, 1, ... until the
 *   first that is not; with n drafts kept, accept_len[b] = n + 1 and next_token[b] is drawn
 *   from the weights max(0, p_n - q_n) if n < D_b (from p_n if every weight is 0), or from
 *   p_{D_b} if every draft was kept. A draw at u picks the smallest token k whose running
 *   sum of weights, in token order, exceeds u times their total.
 * With x_j drawn from q_j and the u uniform, every emitted token follows the target's
 * distribution. The uniform draws are inputs, so results are reproducible.
 *
 *   target_logits  [sum_b (1 + D_b), vocab] (the target's rows of every window, as for
 *                  spec_accept), bf16 or fp32
 *   draft_logits   [sum_b D_b, vocab], the drafter's logits at every draft position, the
 *                  same dtype; may be NULL when max_draft_len is 0
 *   draft_tokens   int32 [sum_b D_b], each in [0, vocab)
 *   u_accept       fp32 [sum_b D_b], in [0, 1)
 *   u_sample       fp32 [B], in [0, 1)
 *   temperature    > 0 (1: the models' own distributions)
 *   workspace      >= 256 bytes, 256-byte aligned, flag word zero on first use
 * Every row must hold at least one finite logit (rows of NaN give unspecified tokens).
 * A draft length outside [0, max_draft_len] or a draft token outside [0, vocab) sets the
 * workspace flag (sv_workspace_status: SV_ERR_DEVICE_SHAPE) and leaves the outputs of the
 * sequences concerned untouched. vocab <= 2^30. One cluster of 8 CTAs per sequence, each
 * CTA streaming an eighth of every row it reads; rows after the first rejection are not
 * read. Asynchronous.
 */
SV_API sv_status spec_accept_stochastic(int32_t batch, int32_t max_draft_len, int32_t vocab,
                                        int32_t logits_dtype, const void* target_logits,
                                        const void* draft_logits, const int32_t* draft_tokens,
                                        const int32_t* draft_len, const float* u_accept,
                                        const float* u_sample, float temperature,
                                        int32_t* accept_len, int32_t* next_token,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace spec_draft_signals needs on the current CUDA device. 0 if invalid. */
SV_API size_t spec_draft_signals_workspace_size(int32_t rows, int32_t vocab);

/*
 * spec_draft_signals -- the draft signals of "SpecKV: Adaptive Speculative Decoding with
 * Compression-Aware Gamma Selection" (summary, "technical core", item 1), the inputs of
 * its speculation-length controller, for every row of a logits matrix (in that use, the
 * draft model's logits at each drafted position):
 *   confidence[r] = max_j p_j,  entropy[r] = -sum_j p_j ln p_j (nats),
 *   p = softmax(logits[r, :]).
 * The page names the largest probability as one reading of "confidence"; the entropy's
 * base is not given and is taken as e.
 *
 *   logits       bf16 or fp32 [rows, vocab], row-major; every row must hold at least one
 *                finite value (NaN elements are ignored)
 *   confidence, entropy  fp32 [rows] (outputs)
 *   workspace >= spec_draft_signals_workspace_size(rows, vocab) bytes, 256-byte aligned,
 *                zero-filled before its first use (it keeps a completion counter that
 *                every call leaves at zero)
 * One pass over the logits, fp32 arithmetic: a running max, sum of exponentials and
 * exponent-weighted sum per part of a row, merged with the online-softmax rule.
 */
SV_API sv_status spec_draft_signals(int32_t rows, int32_t vocab, int32_t logits_dtype,
                                    const void* logits, float* confidence, float* entropy,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Work plan of one attention call (sv_plan_preview). */
typedef struct {
  int32_t num_units;    /* U: units = (sequence, KV head, row tile of <= 128 query rows) */
  int32_t total_tiles;  /* TT: key tiles of all units, laid end to end on one tile line */
  int32_t tile_keys;    /* KT: cache positions per key tile */
  int32_t num_ctas;     /* C: persistent attention CTAs */
  int32_t unit_ctas;    /* k >= 1: CTA u*k + i takes the i-th of k equal parts of unit u's
                           tiles; 0: CTA c takes a contiguous range of the tile line, ranges
                           balanced with `switch_tiles` charged for each unit started */
  int32_t switch_tiles; /* tiles' worth of time charged for starting a unit */
} sv_plan_info;

/*
 * sv_plan_preview -- the work plan that spec_verify_attn (or the _paged or _host_lengths
 * call) makes for the given lengths, computed on the host; needs no device. For capacity
 * planning, tuning and tests. Units are ordered by sequence, KV head, row tile, except
 * that when every sequence has the same number (> 1) of row tiles they are ordered
 * row-tile-major. A unit's tiles start at the tile holding the first key its rows see
 * (position 0, or under a sliding window of W positions max(0, T_b + i - W + 1) for its
 * first window row i) and end at the tile holding T_b + D_b. The unit-to-CTA policy
 * follows sv_set_unit_ctas, as the call does.
 *
 *   desc          as for the call (q_rows and, for a packed cache, kv_rows are checked)
 *   block_size    0 for a packed cache, else the paged cache's block size (the block
 *                 table itself is not checked)
 *   seq_lens_host, draft_len_host  int32 [B] in host memory
 *   num_sms       SMs of the device the call would run on, 1 .. 192
 *   attn_kernel   1 = mma.sync kernel, 2 = tcgen05 kernel (the kernel sets KT and the
 *                 policy's time model; automatic selection takes 2 for d = 128, and
 *                 for d = 64 with bf16 K/V)
 *   info          out: the counts above
 *   units         out or NULL: int32 [capacity_units][4] = (b, KV head, row tile, first
 *                 cache position of the unit's first tile), in tile-line order
 *   unit_begin    out or NULL: int32 [capacity_units + 1]; unit u holds tiles
 *                 unit_begin[u] .. unit_begin[u + 1] - 1 of the line
 *   cta_begin     out or NULL: int32 [num_ctas + 1][2] = (first tile, its unit) of each
 *                 CTA's range; entry num_ctas is (TT, U). A CTA's range ends where the
 *                 next one's begins.
 * Returns SV_ERR_SHAPE for a length or size out of range (as the calls would report),
 * SV_ERR_WORKSPACE when units or unit_begin is given and U > capacity_units (info is
 * filled), or when the plan is beyond the host plan's capacity (256 sequences, 640
 * units, 192 CTAs).
 */
SV_API sv_status sv_plan_preview(const sv_attn_desc* desc, int32_t block_size,
                                 const int32_t* seq_lens_host, const int32_t* draft_len_host,
                                 int32_t num_sms, int32_t attn_kernel, sv_plan_info* info,
                                 int32_t* units, int32_t* unit_begin, int32_t* cta_begin,
                                 int32_t capacity_units);

/* Synchronises `stream`, then reads the sticky device-side flags of a workspace used by
 * either call: SV_OK, SV_ERR_DEVICE_SHAPE or SV_ERR_TIMEOUT. clear != 0 resets them. */
SV_API sv_status sv_workspace_status(void* workspace, int clear, void* stream);

/* Human-readable name of a status code (static string). */
SV_API const char* sv_status_string(sv_status status);

/* Attention kernel selection, for measurement and tests: 0 = automatic (default),
 * 1 = warp-level mma.sync kernel, 2 = tcgen05 kernel. Returns the previous value, or -1
 * if the value is unknown or the kernel is not built. Process-wide. */
SV_API int sv_set_attn_kernel(int which);

/* How spec_verify_attn spreads its units (sequence, KV head, 128-row tile) over CTAs,
 * for measurement and tests: -1 = by the library's per-tile time model (default), 0 =
 * always one tile line split evenly over the CTAs, k >= 1 = k CTAs per unit, each with
 * an equal share of its tiles, whenever units * k fits the grid (otherwise as 0). Results
 * agree to rounding across modes. Returns the previous value, or -2 if mode is outside
 * [-1, 1024]. Process-wide. */
SV_API int sv_set_unit_ctas(int mode);

/* Row pairs, for measurement and tests. When a KV head serves more than one 128-row tile
 * but at most two (128 < G * (1 + max_draft_len) <= 256), with bf16 K/V, head_dim 128, a
 * packed cache, no sliding window, and batch * num_kv_heads at most the number of SMs,
 * spec_verify_attn (and the host-lengths call) can run one CTA per (sequence, KV head) that
 * holds both row tiles and reads each K/V tile once for both, instead of the unit plan
 * (whose row tiles each stream the keys, the second mostly from L2). 0 = never (default),
 * 1 = whenever it applies. It is one kernel launch: no planning and no combining kernel.
 * It is off by default because it measures slower than the unit plan: with the whole of
 * TMEM taken by two accumulators and two score tiles, Q comes from shared memory and P
 * shares its score tile's columns, so each row tile's score MMA waits for its previous P V.
 * Returns the previous value, or -2 if mode is not 0 or 1. Process-wide. */
SV_API int sv_set_row_pairs(int mode);

/* K/V shared-memory rings of the tcgen05 kernel with bf16 K/V, for measurement and tests.
 * 1 = separate rings of K tiles (four, each free once its score MMA is complete) and V
 * tiles (three, each free once its P V is), filled by two producers, so K loads run
 * further ahead of the score MMAs; 0 = three paired stages of one K and one V tile, free
 * once the tile's P V is complete; -1 (default) = paired stages when a KV head's rows,
 * num_q_heads / num_kv_heads * (1 + max_draft_len), fill more than one 128-row tile but
 * not a whole number of them, or when the CTAs would each stream more than 1024 key tiles
 * (by max_seq_len), split rings otherwise. Results are bit-identical across modes; FP8 K/V
 * is unaffected. Returns the previous value, or -2 if mode is outside [-1, 1].
 * Process-wide. */
SV_API int sv_set_kv_rings(int mode);

/* 1 if spec_verify_attn with this descriptor, cache layout (block_size 0: packed), SM count
 * and kernel (1 = mma.sync, 2 = tcgen05) runs the row-pair kernel under the current
 * setting, 0 if it runs the unit plan that sv_plan_preview describes, -1 if the arguments
 * are invalid. Needs no device. */
SV_API int sv_row_pair_mode(const sv_attn_desc* desc, int32_t block_size, int32_t num_sms,
                            int32_t attn_kernel);

/* Profiling hook: when both are non-NULL, every later spec_verify_attn records `start`
 * just before and `stop` just after its main attention kernel, on the call's stream
 * (cudaEvent_t handles owned by the caller). Pass NULLs to turn it off. Process-wide.
 * The events sit between the call's kernels and so cost them their launch overlap
 * (several microseconds per call): time whole calls with the hook off. */
SV_API void sv_set_profile_events(void* start_event, void* stop_event);

/* Fault injection for tests, on the host: after `after` more kernel launches of the
 * library, the next launch fails without reaching the GPU and the call that makes it
 * returns SV_ERR_CUDA (spec_verify_attn and the paged call launch three kernels in this
 * order: plan, attention, combine; the host-lengths call attention and combine;
 * spec_accept and spec_draft_signals one each). The call's earlier launches have run;
 * its outputs are then unspecified, and its workspace serves the next call as it is. One
 * failure per arming; after < 0 disarms. Returns the launches that were still to go
 * before a pending failure, or -1 if none was pending. Process-wide. */
SV_API int sv_inject_launch_failure(int after);

/* Fault injection for tests, on the device side of the tcgen05 attention kernel's bounded
 * waits: the next verify-attention launch of that kernel gives every barrier wait
 * `limit_cycles` clock cycles instead of about 2 s, and each of its CTAs withholds the K
 * and V loads of the first tile of its range, so the waits for that tile run out. The kernel
 * then sets SV_ERR_TIMEOUT in the workspace (read it with sv_workspace_status); every role
 * of every CTA leaves its loop, the copies and MMAs still in flight are waited for, TMEM
 * is freed, and the kernel returns. The call itself returns SV_OK and its outputs are
 * unspecified; the workspace serves the next call once its flags are cleared. Calls that
 * run the mma.sync kernel leave the arming pending. limit_cycles <= 0 disarms. Returns 1
 * if an arming was pending, else 0. Process-wide. */
SV_API int sv_inject_wait_timeout(int64_t limit_cycles);

/* Library version: major * 10000 + minor * 100 + patch. */
SV_API int sv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
