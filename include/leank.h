/*
 * leank.h -- C ABI of a decode-attention library for a LeanK-pruned KV cache
 * on NVIDIA GB300 (sm_103a).
 *
 * The method (the passages each call follows):
 *   - "KV cache optimisation for LLMs and LeanK pruning" (framerc.cn),
 *     section 2.2 stage 2: a static binary mask beta per (layer, kv head) keeps
 *     a multiple of 32 K channels; section 3.1: heads are grouped by kept count,
 *     the K cache is split into a full-width part for the attention sinks and
 *     the local window and a pruned part K_prun for the middle tokens, and a
 *     fused FlashAttention reads both; section 3.2: a head with no kept channel
 *     drops its middle V as well.
 *   - "FastGen: profile-based adaptive KV compression" (mhpn.cn), section 2.1:
 *     each decode step appends K_t, V_t and then attends with Q_t over the
 *     whole cache; sections 3.1-3.2: per-head policies (local window only,
 *     special tokens only, full); section 5.1: the three integration points
 *     (per-head allocation, policy-aware append, a kernel reading per-head
 *     ranges).
 *
 * Conventions (all calls):
 *   - Every call returns lk_status.  On a non-OK status nothing was enqueued
 *     and lk_last_error() holds a message (per calling thread).
 *   - Device memory (cache buffer, workspace, q/k/v/o/ids) is owned by the
 *     caller and passed as raw device pointers.  The library never calls
 *     cudaMalloc or cudaFree; its handles are host objects.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Hot calls only enqueue work; they never synchronise.
 *   - Tensors are dense row-major: bf16 = 16-bit bfloat16 stored as uint16.
 *   - Errors found on the device (capacity overflow of a special-token head,
 *     an out-of-range token id, a bounded wait that ran out) set a sticky
 *     status word inside the cache; lk_check() reads and clears it.
 */
#ifndef LEANK_H
#define LEANK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lk_status {
  LK_OK = 0,
  LK_ERR_ARG = 1,         /* bad argument (null pointer, range, mask count, ...) */
  LK_ERR_ALIGN = 2,       /* a pointer is not aligned as required */
  LK_ERR_CAPACITY = 3,    /* token capacity or buffer size exceeded */
  LK_ERR_STATE = 4,       /* call not valid in the cache's current state */
  LK_ERR_CUDA = 5,        /* a CUDA runtime call failed (message has the CUDA error) */
  LK_ERR_TIMEOUT = 6,     /* a device-side bounded wait ran out (lk_check) */
  LK_ERR_UNSUPPORTED = 7  /* shape outside what the kernels implement */
} lk_status;

/* Per-(layer, kv head) cache policy (FastGen section 3.1). */
typedef enum lk_policy {
  LK_POLICY_FULL = 0,     /* LeanK layout: sinks + window at full width, middle on kept channels */
  LK_POLICY_LOCAL = 1,    /* last local_only_window tokens only, full width, no sinks */
  LK_POLICY_SPECIAL = 2   /* tokens whose id is special only, full width, in arrival order */
} lk_policy;

/* Model geometry and cache parameters. */
typedef struct lk_plan_desc {
  int32_t num_layers;         /* L >= 1 */
  int32_t num_q_heads;        /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;       /* Hkv >= 1; query head j reads kv head j / (Hq/Hkv) */
  int32_t head_dim;           /* d; must be 128 */
  int32_t sink;               /* S >= 0: attention-sink tokens of FULL heads */
  int32_t local;              /* W >= 1: local window of FULL heads */
  int32_t local_only_window;  /* W_loc >= 1 if any head is LOCAL */
  int32_t vocab;              /* entries of is_special (>= 1 if any head is SPECIAL) */
  int32_t special_capacity;   /* max rows of a SPECIAL head per sequence; 0 = token capacity */
} lk_plan_desc;

typedef struct lk_plan_s* lk_plan;    /* host object owned by the library */
typedef struct lk_cache_s* lk_cache;  /* host object; its device buffer is the caller's */

/* Where one (layer, sequence, kv head) lives inside the cache buffer (byte
 * offsets from the buffer start).  Region A is full width (sinks + window
 * ring, LOCAL ring, or SPECIAL rows); region B holds middle tokens on the
 * kept channels (FULL heads with n_kept > 0).
 *   Contiguous cache (page_rows = 0): middle row m is row m of region B.
 *   Paged cache (page_rows = 128): region B is the page area of the head's
 *   width class, shared by every head of that class; middle row m is row
 *   page_table[m / 128] * 128 + m % 128 of it, page_table being the head's
 *   int32 [max_pages] row at page_table_offset (-1: no page). */
typedef struct lk_region_info {
  int32_t policy;
  int32_t n_kept;             /* kept K channels (FULL), else 0 */
  int32_t rows_a;             /* row capacity of region A */
  int32_t rows_b;             /* rows of region B (paged: of the class's page area) */
  uint64_t k_a_offset;        /* bf16 [rows_a][128] */
  uint64_t v_a_offset;        /* bf16 [rows_a][128] */
  uint64_t k_b_offset;        /* bf16 [rows_b][n_kept], kept channels ascending */
  uint64_t v_b_offset;        /* bf16 [rows_b][128] */
  int32_t page_rows;          /* 0: contiguous region B; else rows per page */
  int32_t max_pages;          /* entries of the head's page-table row */
  uint64_t page_table_offset; /* int32 [max_pages] */
  int32_t kv_format;          /* lk_kv_format of region B */
  int32_t sealed_blocks;      /* INT8 / FP8: complete 128-row blocks (read them with
                                 lk_cache_block); region B's offsets then give
                                 the bf16 tail: middle row m >= 128 * sealed_blocks
                                 is tail row m - 128 * sealed_blocks */
} lk_region_info;

/* Storage format of region B (the middle tokens).
 *   LK_KV_BF16  K_prun and V rows in bf16.
 *   LK_KV_INT8  KIVI-style quantisation applied after pruning and
 *               reorganisation (LeanK 4.2 and 5.2 problem 3; KIVI's
 *               per-channel K / per-token V, pruning white paper 5.2.1):
 *               every complete 128-row block of a head's middle is stored as
 *               INT8 codes with one fp32 scale per kept K channel and one per
 *               V token, scale = max|x| / 127 (fp32), code = x / scale
 *               rounded half to even, clipped to +-127; the last,
 *               incomplete block stays bf16.
 *   LK_KV_FP8   as LK_KV_INT8 with FP8 codes (one of the low-precision
 *               formats of the white paper's 5.2.1): OCP e4m3 (largest
 *               finite value 448), scale = max|x| / 448 (fp32), code = x /
 *               scale rounded to the nearest e4m3 value, ties to the even
 *               code, saturated at +-448; a zero code keeps the sign. */
typedef enum { LK_KV_BF16 = 0, LK_KV_INT8 = 1, LK_KV_FP8 = 2 } lk_kv_format;

/* Cache options for lk_cache_bytes_ex / lk_cache_init_ex. */
typedef struct lk_cache_options {
  int64_t middle_tokens;      /* < 0: contiguous region B; >= 0: paged, pools
                                 sized as in lk_cache_bytes_paged (INT8 / FP8:
                                 sealed blocks are the pages,
                                 floor(middle_tokens/128) per head of a class) */
  int32_t kv_format;          /* lk_kv_format */
  int32_t reserved;           /* 0 */
} lk_cache_options;

/* Build a plan (host only; touches no GPU).
 *   masks      host uint8 [L][Hkv][128], 0/1: the static mask beta (LeanK 2.2).
 *              For FULL heads the kept count must be 0, 32, 64, 96 or 128;
 *              rows of other policies are ignored.
 *   policies   host int32 [L][Hkv] of lk_policy.
 *   is_special host uint8 [vocab] (1 = special id) or NULL if no SPECIAL head.
 * Heads are grouped by (policy, kept count) and each FULL head gets its kept
 * channel list (ascending), used to permute q.  Errors: LK_ERR_ARG,
 * LK_ERR_UNSUPPORTED (head_dim != 128 or Hq/Hkv > 8). */
lk_status lk_build_plan(const lk_plan_desc* desc, const uint8_t* masks, const int32_t* policies,
                        const uint8_t* is_special, lk_plan* out);
void lk_plan_destroy(lk_plan plan);

/* Build the static mask beta on the device from learned channel importances
 * (LeanK 2.2 stage 2):
 *   alpha     device fp32 [L][Hkv][128] importances
 *   eligible  device uint8 [L][Hkv], 1 for heads that take a mask (FULL
 *             policy), or NULL for all; other heads get all ones
 *   prune_pct s in [0, 100]: share of eligible channels pruned; a channel
 *             stays when alpha >= the s-th percentile of the eligible alphas
 *             (linear interpolation, computed in fp32)
 *   align     32, 64 or 128: per-head kept counts become multiples of it
 *   exact     0: counts rounded down; 1: then topped up by +align on the heads
 *             with the largest remainders (ties: lower head index) until the
 *             total is align * floor((1 - s/100) * heads * 128 / align + 1/2)
 *   masks     device uint8 [L][Hkv][128] out; a head keeps its channels of
 *             largest alpha, equal alphas to the lower channel index.
 * L * Hkv <= 8192.  Enqueued on `stream`; copy the masks to the host for
 * lk_build_plan. */
lk_status lk_build_masks(const float* alpha, const uint8_t* eligible, int32_t num_layers, int32_t num_kv_heads,
                         double prune_pct, int32_t align, int32_t exact, uint8_t* masks, void* stream);

/* Host-side query of one head's policy, kept count and kept channels
 * (kept_channels: host int16 [128] or NULL; first n_kept entries valid). */
lk_status lk_plan_head(lk_plan plan, int32_t layer, int32_t kv_head, int32_t* policy,
                       int32_t* n_kept, int16_t* kept_channels);

/* Bytes of the cache buffer for `batch` sequences of up to `capacity_tokens`
 * tokens each (LeanK 3.1 split cache, FastGen 5.1 per-head allocation). */
lk_status lk_cache_bytes(lk_plan plan, int32_t batch, int32_t capacity_tokens, size_t* bytes);

/* Paged variant (continuous batching; paged KV blocks as in the pruning
 * white paper, yyx235 blog, section 3.2 "granularity", with FastGen 5.1's
 * per-head variable allocation): region B of every FULL head with k > 0 is
 * held in 128-row pages of its width class instead of a contiguous
 * capacity-sized run.  Each class gets enough pages for `middle_tokens`
 * middle tokens (positions past the sinks and the window) summed over the
 * batch, plus one partly filled page per sequence; a sequence still holds at
 * most `capacity_tokens` tokens.  Pages are taken by appends and prefills on
 * the device and given back by lk_release_sequence.  Errors as
 * lk_cache_bytes; LK_ERR_ARG for middle_tokens < 0. */
lk_status lk_cache_bytes_paged(lk_plan plan, int32_t batch, int32_t capacity_tokens, int64_t middle_tokens,
                               size_t* bytes);

/* Bytes of the decode workspace (split partials and counters for every
 * layer's entries, staging of lk_step_host) for `batch` sequences. */
lk_status lk_workspace_bytes(lk_plan plan, int32_t batch, size_t* bytes);

/* Bind a cache to a caller-owned device buffer of at least lk_cache_bytes
 * bytes, 256-byte aligned.  Enqueues a zero fill of the buffer and the upload
 * of the plan's tables on `stream`; all layers start empty.  The plan must
 * outlive nothing: the cache copies what it needs.  Needs a CUDA device. */
lk_status lk_cache_init(lk_plan plan, void* dev_buf, size_t bytes, int32_t batch,
                        int32_t capacity_tokens, void* stream, lk_cache* out);
/* lk_cache_bytes / lk_cache_init with explicit options (paging and the
 * storage format of region B).  Errors as lk_cache_bytes; LK_ERR_ARG for a
 * null opt or an unknown kv_format. */
lk_status lk_cache_bytes_ex(lk_plan plan, int32_t batch, int32_t capacity_tokens,
                            const lk_cache_options* opt, size_t* bytes);
lk_status lk_cache_init_ex(lk_plan plan, void* dev_buf, size_t bytes, int32_t batch,
                           int32_t capacity_tokens, const lk_cache_options* opt, void* stream,
                           lk_cache* out);

/* Host copy of sealed block `block` of an INT8 or FP8 cache's (layer, b,
 * kv_head), in logical order: k_codes [128][n_kept] (kept channels
 * ascending), k_scales [n_kept], v_codes [128][128], v_scales [128]; any
 * pointer may be NULL.  Codes are one byte each: INT8 values, or e4m3 bit
 * patterns for FP8.  Synchronises `stream`.  Errors: LK_ERR_STATE (not a
 * quantised cache), LK_ERR_ARG (no such sealed block). */
lk_status lk_cache_block(lk_cache cache, int32_t layer, int32_t b, int32_t kv_head, int32_t block,
                         int8_t* k_codes, float* k_scales, int8_t* v_codes, float* v_scales, void* stream);

/* As lk_cache_init, for a paged cache of lk_cache_bytes_paged bytes. */
lk_status lk_cache_init_paged(lk_plan plan, void* dev_buf, size_t bytes, int32_t batch,
                              int32_t capacity_tokens, int64_t middle_tokens, void* stream, lk_cache* out);
void lk_cache_destroy(lk_cache cache);

/* Zero a caller-owned workspace of at least lk_workspace_bytes bytes
 * (256-byte aligned).  Needed once before the first lk_decode_attn with it,
 * and again after lk_check reported LK_ERR_TIMEOUT. */
lk_status lk_workspace_init(lk_cache cache, void* workspace, size_t ws_bytes, void* stream);

/* Build one empty layer from a dense history of n tokens (prefill, "white
 * paper" 2.3): equal, byte for byte, to n successive lk_append calls.
 *   k, v  device bf16 [B][n][Hkv][128];  ids device int32 [B][n] or NULL.
 * Errors: LK_ERR_STATE if the layer is not empty, LK_ERR_CAPACITY if n
 * exceeds the token capacity. */
lk_status lk_prefill(lk_cache cache, int32_t layer, const void* k, const void* v,
                     const int32_t* ids, int32_t n, void* stream);

/* lk_prefill with a length per sequence: sequence b gets the first lens[b]
 * tokens of its row of the padded inputs.
 *   k, v  device bf16 [B][n_max][Hkv][128];  ids device int32 [B][n_max] or NULL;
 *   lens  host int32 [B], each in [0, n_max].
 * Decode then handles each sequence at its own length (continuous batching). */
lk_status lk_prefill_ragged(lk_cache cache, int32_t layer, const void* k, const void* v,
                            const int32_t* ids, const int32_t* lens, int32_t n_max, void* stream);

/* Prefill one slot b of one layer while the other slots keep their tokens
 * (continuous batching: a new request takes a released slot).
 *   k, v  device bf16 [n][Hkv][128];  ids device int32 [n] or NULL.
 * Sequence b of `layer` must be empty (fresh or released); n = 0 is allowed.
 * The slot becomes active: lk_append writes to it again.  Paged caches take
 * the pages of its middle rows here.  Errors: LK_ERR_STATE (slot not empty),
 * LK_ERR_CAPACITY (n > capacity, or not enough free pages: nothing is
 * launched then). */
lk_status lk_prefill_sequence(lk_cache cache, int32_t layer, int32_t b, const void* k, const void* v,
                              const int32_t* ids, int32_t n, void* stream);

/* Release slot b in every layer: its pages (paged caches) go back to the
 * free stacks, its lengths and special counts become 0, and the slot turns
 * inactive: lk_append skips it (decode gives o = 0 for it) until
 * lk_prefill_sequence fills it again.  Enqueued on `stream`. */
lk_status lk_release_sequence(lk_cache cache, int32_t b, void* stream);

/* Pages of one width class (32, 64, 96 or 128 kept channels) of a paged
 * cache: total and currently free (host mirror, exact at every call
 * boundary).  A contiguous cache reports 0 and 0. */
lk_status lk_cache_pages(lk_cache cache, int32_t width, int64_t* total, int64_t* free_pages);

/* Append one token per sequence to a layer (FastGen 2.1, 3.2 stage 2).
 *   k, v  device bf16 [B][Hkv][128];  ids device int32 [B] or NULL.
 * FULL heads: token n < S goes to sink row n; later tokens go to window ring
 * row S + (n-S) mod W, and once the window is full the token n-W it replaces
 * first moves to the middle (K gathered to the kept channels into K_prun row
 * n-W-S, V copied; dropped when n_kept = 0).  LOCAL: ring row n mod W_loc.
 * SPECIAL: appended (row = count) only if is_special[id].  Bit-exact copies.
 * Released slots (lk_release_sequence) are skipped.  Paged caches take a
 * page from the class's free stack when a middle row starts a new page.
 * Errors: LK_ERR_CAPACITY when an active sequence of the layer already holds
 * capacity_tokens, or a paged cache has too few free pages (nothing is
 * launched then). */
lk_status lk_append(lk_cache cache, int32_t layer, const void* k, const void* v,
                    const int32_t* ids, void* stream);

/* Decode attention of one layer (LeanK 3.1 fused FlashAttention over the
 * split cache; FastGen 3.2 per-policy ranges).
 *   q  device bf16 [B][Hq][128];  o  device fp32 [B][Hq][128].
 * For query head j of sequence b (kv head h = j / G): scores q.k / sqrt(128)
 * over sinks + window at all channels and over the middle tokens at the kept
 * channels (q gathered to the kept channel list), one softmax over both,
 * o = sum p V.  Split over tokens across CTAs; partials are merged inside the
 * same launch.  A head with no resident token gives o = 0.
 * workspace: >= lk_workspace_bytes bytes, zeroed once by lk_workspace_init;
 * calls sharing one workspace must not overlap on the GPU. */
lk_status lk_decode_attn(lk_cache cache, int32_t layer, const void* q, float* o,
                         void* workspace, size_t ws_bytes, void* stream);

/* lk_decode_attn without a caller workspace.  The pages have no counterpart:
 * this is a library convenience.  Some callers cannot call cudaMalloc at all
 * -- a plugin running inside a host runtime that owns the device allocator
 * and its memory accounting, or a latency-critical loop where an allocation
 * would synchronise the device -- and so cannot provide the split workspace.
 * This entry point keeps the split counters and partials in a fixed 8 MiB
 * device array built into the library (a file-scope __device__ array that
 * every GPU loading the library holds until the process exits); it
 * allocates nothing.
 *   q, o  as for lk_decode_attn.
 * Limit: the split scratch of the cache (about (256 + B*Hkv) * G * 520
 * bytes) must fit in 8 MiB, else LK_ERR_CAPACITY and nothing is enqueued.
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress, which allocates nothing); on the first call on a
 * device that lookup may load the library's device code into the context,
 * so make that first call before any stream capture.  Each call clears the
 * split counters on `stream` before its launch; the partials need no
 * clearing (each is written before it is read).  All calls share the one
 * array and it keeps the last call's contents: calls that overlap on the GPU
 * (other streams, other threads) race and give wrong results. */
lk_status lk_decode_attn_static(lk_cache cache, int32_t layer, const void* q, float* o, void* stream);

/* lk_append over layers layer0 .. layer0+nlayers-1 in one launch:
 *   k, v  device bf16 [nlayers][B][Hkv][128];  ids device int32 [B] or NULL
 *   (the same token enters every layer). */
lk_status lk_append_layers(lk_cache cache, int32_t layer0, int32_t nlayers, const void* k, const void* v,
                           const int32_t* ids, void* stream);

/* lk_decode_attn over layers layer0 .. layer0+nlayers-1 in one launch (the
 * work of all layers is split across the CTAs together):
 *   q  device bf16 [nlayers][B][Hq][128];  o  device fp32 [nlayers][B][Hq][128].
 * Useful when every layer's query is known up front (benchmarks, drafts). */
lk_status lk_decode_attn_layers(lk_cache cache, int32_t layer0, int32_t nlayers, const void* q, float* o,
                                void* workspace, size_t ws_bytes, void* stream);

/* One decode step of a layer: the append of the new token followed by
 * attention with the new query (FastGen 2.1: append K_t, V_t, then attend
 * with Q_t), in one launch.  Same arguments, results and errors as
 *   lk_append(cache, layer, k, v, ids, stream);
 *   lk_decode_attn(cache, layer, q, o, workspace, ws_bytes, stream);
 * and the cache is left as they leave it (byte for byte, except that a
 * paged cache may hand out its free pages in another order).  With a bf16
 * middle one kernel does both: the CTA that combines a head's split
 * partials adds the new token (and the token leaving a full window for the
 * middle) to the softmax from the inputs, then writes them into the cache;
 * the window slot being replaced is left out of the scores.  INT8 / FP8 caches
 * (where an append may seal a block, changing the values decode reads) run
 * the two launches.  Nothing is launched on an error. */
lk_status lk_step(lk_cache cache, int32_t layer, const void* q, const void* k, const void* v,
                  const int32_t* ids, float* o, void* workspace, size_t ws_bytes, void* stream);

/* lk_step over layers layer0 .. layer0+nlayers-1 in one launch: q, o as for
 * lk_decode_attn_layers, k, v, ids as for lk_append_layers. */
lk_status lk_step_layers(lk_cache cache, int32_t layer0, int32_t nlayers, const void* q, const void* k,
                         const void* v, const int32_t* ids, float* o, void* workspace, size_t ws_bytes,
                         void* stream);

/* One decode step end to end from host memory: q [B][Hq][128] bf16, k, v
 * [B][Hkv][128] bf16 and ids [B] int32 (NULL allowed) in, o [B][Hq][128]
 * fp32 out.  When every buffer is page-locked and mapped into the device's
 * address space (cudaHostAlloc / cudaMallocHost, cudaHostRegister with
 * mapping; torch's pin_memory), the append and decode kernels read the
 * inputs from host memory and write o there directly over the host link
 * (NVLink-C2C on Grace) -- no staging copies.  Otherwise the inputs are
 * copied into the workspace, lk_step runs, and o is copied back (pinned
 * buffers keep those copies asynchronous).  Read o only after synchronising
 * `stream`. */
lk_status lk_step_host(lk_cache cache, int32_t layer, const void* q_host, const void* k_host,
                       const void* v_host, const int32_t* ids_host, float* o_host,
                       void* workspace, size_t ws_bytes, void* stream);

/* lk_step_host with the step's inputs in one host block: host_in = q bf16
 * [B][Hq][128] | k bf16 [B][Hkv][128] | v bf16 [B][Hkv][128] | ids int32 [B]
 * (present iff has_ids != 0), back to back.  Read in place when the block
 * and o are mapped page-locked memory, else moved by a single copy each
 * way. */
lk_status lk_step_host_packed(lk_cache cache, int32_t layer, const void* host_in, int32_t has_ids,
                              float* o_host, void* workspace, size_t ws_bytes, void* stream);

/* A step of layers layer0 .. layer0+nlayers-1 from host memory, as
 * lk_append_layers + lk_decode_attn_layers: host_in = q bf16
 * [nlayers][B][Hq][128] | k bf16 [nlayers][B][Hkv][128] | v (as k) | ids
 * int32 [B] (present iff has_ids != 0; the same token for every layer),
 * back to back; o_host fp32 [nlayers][B][Hq][128] out.  Both must be
 * page-locked and mapped into the device's address space (the kernels read
 * and write them in place over the host link); otherwise LK_ERR_ARG and
 * nothing is launched.  Two launches whatever the step mode (the fused
 * kernel stages the new token with bulk copies, which are kept away from
 * host memory).  Errors as for lk_append_layers and lk_decode_attn_layers.
 * Read o only after synchronising `stream`. */
lk_status lk_step_layers_host_packed(lk_cache cache, int32_t layer0, int32_t nlayers, const void* host_in,
                                     int32_t has_ids, float* o_host, void* workspace, size_t ws_bytes,
                                     void* stream);

/* Host-tracked token count of a layer: the longest sequence's length. */
lk_status lk_cache_length(lk_cache cache, int32_t layer, int32_t* n);

/* Host-tracked token count of every sequence of a layer (lens: host int32 [B]). */
lk_status lk_cache_lengths(lk_cache cache, int32_t layer, int32_t* lens);

/* Location of one (layer, sequence, kv head) in the cache buffer. */
lk_status lk_cache_region(lk_cache cache, int32_t layer, int32_t b, int32_t kv_head,
                          lk_region_info* out);

/* K+V bytes one lk_decode_attn of `layer` reads from the resident cache
 * (synchronises `stream` to read the special-token counts). */
lk_status lk_resident_bytes(lk_cache cache, int32_t layer, void* stream, uint64_t* bytes);

/* How lk_step / lk_step_layers run a step on a bf16 middle:
 *   LK_STEP_AUTO   the library's choice (default): one fused launch when
 *                  the decode's CTAs each stream at least 256 KB and meet
 *                  at most 32 (layer, sequence, kv head) entries (e.g. a
 *                  32K-token layer: 26.6 -> 25.1 us per step), else the
 *                  append and decode launches (a 0.24 MB layer, or a
 *                  32-layer, 64-sequence step, are faster that way);
 *   LK_STEP_FUSED  always one launch;   LK_STEP_SPLIT  always two.
 * Results and cache contents do not depend on the mode.  INT8 / FP8 middles
 * always run two launches. */
typedef enum { LK_STEP_AUTO = 0, LK_STEP_FUSED = 1, LK_STEP_SPLIT = 2 } lk_step_mode;
lk_status lk_set_step_mode(lk_cache cache, int32_t mode);

/* Whether lk_step_layers(cache, layer0, nlayers, ...) would run as one fused
 * launch now (at the host's current lengths): *fused = 1 or 0. */
lk_status lk_step_is_fused(lk_cache cache, int32_t layer0, int32_t nlayers, int32_t* fused);

/* Override the number of CTAs of lk_decode_attn (0 = the library's choice:
 * one per SM, or 27/32 of the SMs for a bf16 launch over at most 64
 * (sequence, kv head) entries, where fewer, longer streams reach a higher
 * HBM rate); for tuning and split-invariance tests.  Must be <= 256. */
lk_status lk_set_decode_ctas(lk_cache cache, int32_t ctas);

/* Bound of the decode kernel's waits on its stage ring and on its warps'
 * segment barriers, in ns (default 1 s; at most 10 s).  A wait that runs out
 * records LK_ERR_TIMEOUT for lk_check and the launch's outputs are garbage;
 * after it, call lk_workspace_init before the next decode.  0 makes every
 * wait that is not already complete run out at once: a way to exercise that
 * failure path without a fault.  The kernel's final wait for its own copies
 * to land keeps its 1 s bound whatever this is.  Errors: LK_ERR_ARG. */
lk_status lk_set_wait_limit(lk_cache cache, uint64_t ns);

/* Synchronise `stream`, read the device status word and, when a bit is set,
 * clear it on `stream` and synchronise again (the clear has landed when the
 * call returns).  Returns
 * LK_ERR_TIMEOUT, LK_ERR_CAPACITY or LK_ERR_ARG (bad token id) for a set
 * bit, LK_ERR_CUDA for a pending CUDA error, else LK_OK. */
lk_status lk_check(lk_cache cache, void* stream);

/* Message of the last non-OK status on the calling thread ("" if none). */
const char* lk_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* LEANK_H */
