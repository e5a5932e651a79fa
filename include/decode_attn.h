/*
 * decode_attn.h -- C ABI of the fused decode-step attention library for GB300
 * (sm_103a): KV append + grouped-query attention over a paged KV cache or a
 * sliding-window ring buffer + per-head attention-sink logits.
 *
 * The operation (SimpleLLM README, changes table):
 *   row "one decode-attention kernel for sinks, sliding window, GQA and the KV
 *        append (replaces four ops)"           -> decode_attn_paged / _ring
 *   row "paged KV cache for full-attention layers" -> the paged layout
 *   row "ring buffer for sliding-window layers"    -> the ring layout
 *   row "CUDA graphs for any set of active slots"  -> every call is
 *        capturable: no host read of seq_lens, no allocation once reserved.
 * The pages print no formula; the definition used is, for every active
 * sequence b (L = seq_lens[b] > 0, the length AFTER this step's append; the
 * new token has position p = L - 1), query head h and KV head g = h / (Hq/Hkv):
 *     J   = { j : lo <= j < L },  lo = max(0, L - W) if a window W applies, else 0
 *     s_j = scale * <q[b,h,:], k_j[g,:]>
 *     out[b,h,:] = sum_j e^{s_j} v_j[g,:] / (e^{sink[h]} + sum_j e^{s_j})
 * and out[b] = 0 when L == 0 (inactive slot). The sink is a raw logit (not
 * multiplied by scale) and carries no value vector.
 *
 * Conventions for every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *     16-byte aligned. The library keeps none of them after the call returns.
 *   - bf16 tensors: q, k_new, v_new, k_cache, v_cache, out. int32: block_table,
 *     seq_lens. fp32: sinks.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream). A return of 0 means "validated and
 *     launched"; faults found by the kernel itself (a bad length or page id)
 *     are recorded in a device status word, see decode_attn_device_status().
 *   - Return value: 0 on success, else a negative DA_ERR_* code; nothing is
 *     launched when a code is returned.
 *   - Supported now: head_dim 64, page_size 16, query heads per KV head
 *     (G = Hq/Hkv) in {1, 2, 4, 8, 16}, batch <= 1024, Hq <= 1024, batch*Hkv <= 65536,
 *     ring capacity >= 16, a GPU with at most 160 SMs. Anything else returns
 *     DA_ERR_UNSUPPORTED.
 *   - The attention entry points use a library-owned workspace per device
 *     (split partials and arrival counters). It is allocated on first use or
 *     by decode_attn_reserve(); during stream capture a call that would need
 *     a larger workspace returns DA_ERR_WORKSPACE instead of allocating.
 *     Calls that run concurrently on different streams of one device share
 *     this workspace and must not overlap, unless each of those streams has a
 *     workspace of its own (decode_attn_stream_reserve).
 */
#ifndef DECODE_ATTN_H
#define DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DA_API __attribute__((visibility("default")))
#else
#define DA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define DA_OK 0
#define DA_ERR_INVALID_ARG (-1) /* null pointer, misalignment, Hq % Hkv != 0, bad size */
#define DA_ERR_UNSUPPORTED (-2) /* a shape outside the supported set above */
#define DA_ERR_WORKSPACE (-3)   /* workspace too small while the stream is capturing */
#define DA_ERR_CUDA (-4)        /* a CUDA runtime call or launch failed */
#define DA_ERR_SCRATCH_LIMIT (-5) /* decode_attn_paged_noalloc: shape beyond its fixed scratch */

/* Bits of the device status word (decode_attn_device_status). */
#define DA_STATUS_BAD_SEQ_LEN 1u /* seq_lens[b] < 0, or beyond max_seq_len / the block table row;
                                    the slot is treated as inactive (output 0, no append) */
#define DA_STATUS_BAD_PAGE 2u    /* a block-table entry outside [0, num_pages); that tile reads
                                    zeros and the append into it is skipped */
#define DA_STATUS_TIMEOUT 4u     /* a bounded wait on a tile copy expired; output is garbage */
#define DA_STATUS_BAD_POSITION 8u /* a position L - 1 beyond the rotary tables; row 0 was used */

typedef struct {
    int batch;        /* B: number of sequence slots */
    int num_q_heads;  /* Hq */
    int num_kv_heads; /* Hkv; Hq % Hkv == 0 */
    int head_dim;     /* D (64) */
} da_shape;

/*
 * decode_attn_paged -- one decode step of attention for a full-attention (or
 * windowed) layer whose KV cache is paged. Fuses the KV append: the new
 * token's k_new/v_new are written into the cache AND used for this step.
 *
 *   q          [B, Hq, D]                    query of the new token
 *   k_new,v_new[B, Hkv, D]                   its key / value; both NULL = no append
 *                                            (token p is then read from the cache)
 *   k_cache,   [num_pages, Hkv, page_size, D] paged pool; token j of sequence b sits in
 *   v_cache                                   page block_table[b][j / 16], slot j % 16.
 *                                            Written only at token p's cell.
 *   block_table[B, max_pages_per_seq]        physical page per logical page
 *   seq_lens   [B]                           post-append lengths, 0 = inactive slot
 *   sinks      [Hq] or NULL                  sink logits (NULL = no sink)
 *   window     0 = full attention, W > 0 = attend to the last W positions (incl. p)
 *   scale      multiplier of q.k (1/sqrt(D) for gpt-oss)
 *   out        [B, Hq, D]                    written for every slot (0 for inactive)
 *   max_seq_len upper bound of seq_lens (<= max_pages_per_seq * page_size)
 * Distinct active sequences must not share the page that receives their append.
 */
DA_API int decode_attn_paged(const void *q, const void *k_new, const void *v_new,
                      void *k_cache, void *v_cache,
                      const int32_t *block_table, const int32_t *seq_lens, const float *sinks,
                      int window, float scale, void *out,
                      da_shape s, int page_size, int max_pages_per_seq, int num_pages,
                      int max_seq_len, void *stream);

/*
 * decode_attn_ring -- one decode step for a sliding-window layer whose KV
 * lives in a per-sequence ring of `window` cells: k_cache/v_cache are
 * [B, Hkv, window, D] and token j of sequence b sits in cell j % window.
 * Attends to the last min(L, window) tokens; the append overwrites cell
 * p % window (which held token p - window, now outside the window).
 * Other arguments as in decode_attn_paged.
 */
DA_API int decode_attn_ring(const void *q, const void *k_new, const void *v_new,
                     void *k_cache, void *v_cache,
                     const int32_t *seq_lens, const float *sinks,
                     int window, float scale, void *out, da_shape s, void *stream);

/*
 * decode_attn_paged_rope / decode_attn_ring_rope -- the same steps with the rotary
 * position embedding fused in front of the append (SimpleLLM README, changes table,
 * row "RoPE as one fused kernel at every batch size"). The query and the new key are
 * rotated to position p = L - 1 before the new key is stored and before the scores:
 * for i < D/2 the pair (x_i, x_{i+D/2}) becomes
 *     (x_i c - x_{i+D/2} s,  x_{i+D/2} c + x_i s),   c = rope_cos[p][i], s = rope_sin[p][i]
 * (the rotate-half form of gpt-oss). v is not rotated; cached keys are expected to be
 * stored rotated already.
 *   rope_cos, rope_sin  [max_position, D/2] fp32 device tables, 16-byte aligned; any
 *                       frequency scaling (e.g. YaRN) is the caller's, folded into them
 *   max_position        rows of the tables; a position beyond them sets
 *                       DA_STATUS_BAD_POSITION and uses row 0
 * The new key is rotated in fp32 (each product, sum and difference rounded separately)
 * and stored rounded to bf16, nearest even; the query is rounded to bf16 for the scores.
 * Other arguments as in decode_attn_paged / decode_attn_ring.
 */
DA_API int decode_attn_paged_rope(const void *q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache,
                                  const int32_t *block_table, const int32_t *seq_lens,
                                  const float *sinks, const float *rope_cos, const float *rope_sin,
                                  int max_position, int window, float scale, void *out,
                                  da_shape s, int page_size, int max_pages_per_seq, int num_pages,
                                  int max_seq_len, void *stream);
DA_API int decode_attn_ring_rope(const void *q, const void *k_new, const void *v_new,
                                 void *k_cache, void *v_cache, const int32_t *seq_lens,
                                 const float *sinks, const float *rope_cos, const float *rope_sin,
                                 int max_position, int window, float scale, void *out, da_shape s,
                                 void *stream);

/*
 * decode_attn_paged_fp8 / decode_attn_ring_fp8 -- the same decode step over an fp8 KV
 * cache (17/32 of the bytes of bf16 per cached token). The pages only name quantisation; the
 * format here: every cached K or V row of one token and KV head is 64 OCP e4m3 codes
 * (FN variant: no infinities, largest finite 448) and one fp32 scale; its value is
 * e4m3(code) * scale. The cache is an array of 2176-byte blocks, one per 16 tokens of one
 * KV head, each holding (byte offsets):
 *      0  K codes [16][64]      (row t = token t of the block)
 *   1024  V codes [64][16]      (transposed: row d holds the 16 tokens' element d)
 *   2048  K scales [16] fp32
 *   2112  V scales [16] fp32
 *   paged: kv_cache [num_pages, Hkv, 2176] bytes; block (page, g) holds the page's tokens.
 *   ring:  kv_cache [B, Hkv, W / 16, 2176] bytes; cell c = p % W of (b, g) is token c % 16
 *          of block c / 16; W % 16 == 0.
 * One block is one contiguous copy. kv_cache must be 16-byte aligned; it is read, and the
 * new token's bytes written, in place.
 * The new token is quantised when it is appended: scale = max_d |x_d| / 448 in fp32 (1 when
 * the row is all zero), code_d = the e4m3 value nearest to x_d / scale (fp32 division),
 * ties to even, saturating at +-448; its K row, V column and both scales are written.
 * Scores and the PV product run in fp16 on tensor cores: |q| must stay below 65504.
 * Other arguments, the status and the error behaviour as in decode_attn_paged / _ring.
 */
DA_API int decode_attn_paged_fp8(const void *q, const void *k_new, const void *v_new,
                                 void *kv_cache, const int32_t *block_table,
                                 const int32_t *seq_lens, const float *sinks, int window,
                                 float scale, void *out, da_shape s, int page_size,
                                 int max_pages_per_seq, int num_pages, int max_seq_len,
                                 void *stream);
DA_API int decode_attn_ring_fp8(const void *q, const void *k_new, const void *v_new,
                                void *kv_cache, const int32_t *seq_lens, const float *sinks,
                                int window, float scale, void *out, da_shape s, void *stream);

/*
 * decode_attn_paged_fp8_rope / decode_attn_ring_fp8_rope -- the fp8 steps with the rotary
 * embedding fused in (SimpleLLM README, changes table, rows "RoPE as one fused kernel at
 * every batch size" and "one decode-attention kernel for sinks, sliding window, GQA and the
 * KV append"): q and the new key are rotated to position p = L - 1 exactly as in
 * decode_attn_paged_rope (the new key in fp32, rounded to bf16 nearest even), and the
 * rotated key is then quantised and appended as in decode_attn_paged_fp8. The rotated
 * query is rounded to bf16, then converted to fp16 for the products. rope_cos, rope_sin and
 * max_position as in decode_attn_paged_rope; the other arguments as in the fp8 calls.
 */
DA_API int decode_attn_paged_fp8_rope(const void *q, const void *k_new, const void *v_new,
                                      void *kv_cache, const int32_t *block_table,
                                      const int32_t *seq_lens, const float *sinks,
                                      const float *rope_cos, const float *rope_sin, int max_position,
                                      int window, float scale, void *out, da_shape s, int page_size,
                                      int max_pages_per_seq, int num_pages, int max_seq_len,
                                      void *stream);
DA_API int decode_attn_ring_fp8_rope(const void *q, const void *k_new, const void *v_new,
                                     void *kv_cache, const int32_t *seq_lens, const float *sinks,
                                     const float *rope_cos, const float *rope_sin, int max_position,
                                     int window, float scale, void *out, da_shape s, void *stream);

/*
 * decode_attn_paged_multi / decode_attn_ring_multi -- several query tokens per sequence in
 * one call: speculative verification (draft tokens checked in one step) and chunked
 * prefill appending a run of tokens into pages (the teaching repo's chapters "Speculative
 * Decoding" and "Chunked Prefill", table "The files" on the page "Run it locally", name
 * both; the plain causal reading is used).
 *   q_tokens = T; n_b = q_lens[b] (T when q_lens == NULL), 0 <= n_b <= T, n_b <= seq_lens[b];
 *   seq_lens[b] = L counts the cached tokens plus the n_b new ones (0 = inactive slot).
 *   New token t < n_b sits at position p = L - n_b + t. Query row (t, h) attends the
 *   positions lo..p (causal), lo = max(0, p - W + 1) under a window (paged: window > 0;
 *   ring: always, W = its capacity), else 0; GQA, sinks and scale as in decode_attn_paged.
 *   Positions >= L - n_b are the new tokens, read from k_new / v_new; the others come from
 *   the cache, which holds the history before the call. Afterwards the n_b new tokens are
 *   written into their cells (paged: their pages; ring: cell p % W, the last W of them).
 *   Rows t >= n_b and inactive slots are written as zero.
 *   q, out        [B, T, Hq, 64] bf16 (device)
 *   k_new, v_new  [B, T, Hkv, 64] bf16 (device, required), rows t >= n_b ignored
 *   q_lens        [B] int32 (device) or NULL
 *   caches, block_table, sinks, page_size, max_pages_per_seq, num_pages, max_seq_len:
 *                 as in decode_attn_paged / decode_attn_ring (the ring's W >= 16).
 * Two kernels on `stream`: the attention, then the append (the ring's early query tokens
 * still read the cells the later new tokens overwrite); paged calls of up to four tokens
 * with T * G <= 32 run one kernel with the append fused (a paged cell of a new token is
 * read only through the tile its own kernel pass patches); calls with many key splits add a
 * kernel that folds the splits' partials. Split partials and counters live
 * in a second library workspace (decode_attn_multi_workspace_bytes / _reserve); it is
 * allocated on first use outside graph capture, else DA_ERR_WORKSPACE. T <= 4096.
 * Bad lengths (n_b > T, n_b > L, L beyond the block table) set DA_STATUS_BAD_SEQ_LEN and
 * the slot is treated as inactive.
 */
DA_API int decode_attn_paged_multi(const void *q, const void *k_new, const void *v_new,
                                   void *k_cache, void *v_cache, const int32_t *block_table,
                                   const int32_t *seq_lens, const int32_t *q_lens,
                                   const float *sinks, int window, float scale, void *out,
                                   da_shape s, int q_tokens, int page_size, int max_pages_per_seq,
                                   int num_pages, int max_seq_len, void *stream);
DA_API int decode_attn_ring_multi(const void *q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, const int32_t *seq_lens,
                                  const int32_t *q_lens, const float *sinks, int window,
                                  float scale, void *out, da_shape s, int q_tokens, void *stream);
/*
 * decode_attn_paged_multi_rope / decode_attn_ring_multi_rope -- the several-token steps
 * above with the rotary embedding of decode_attn_paged_rope (the SimpleLLM README's changes
 * table, row "RoPE as one fused kernel at every batch size", applied at each new token's
 * own position): query row (t, h) and new key (t, g) of every new token t < n are rotated to
 * position p = L - n + t before the append and the scores (rotate-half pairs, each product
 * and the sum or difference in fp32, rounded to bf16 nearest even). Cached keys are expected
 * to be stored rotated already; v is not rotated. Rows t >= n are used as given.
 *   rope_cos, rope_sin, max_position: as in decode_attn_paged_rope (a position at or beyond
 *     max_position sets DA_STATUS_BAD_POSITION and uses row 0).
 *   The rotated q and k_new are written to the multi-token workspace (its size from
 *     decode_attn_multi_workspace_bytes covers them) by a kernel launched ahead of the
 *     attention, so the call makes one launch more than decode_attn_multi_launches says.
 *     q and k_new themselves are not modified.
 *   The other arguments, the results and the errors as in decode_attn_paged_multi /
 *   decode_attn_ring_multi; null tables return DA_ERR_INVALID_ARG.
 */
DA_API int decode_attn_paged_multi_rope(const void *q, const void *k_new, const void *v_new,
                                        void *k_cache, void *v_cache, const int32_t *block_table,
                                        const int32_t *seq_lens, const int32_t *q_lens,
                                        const float *sinks, const float *rope_cos,
                                        const float *rope_sin, int max_position, int window,
                                        float scale, void *out, da_shape s, int q_tokens,
                                        int page_size, int max_pages_per_seq, int num_pages,
                                        int max_seq_len, void *stream);
DA_API int decode_attn_ring_multi_rope(const void *q, const void *k_new, const void *v_new,
                                       void *k_cache, void *v_cache, const int32_t *seq_lens,
                                       const int32_t *q_lens, const float *sinks,
                                       const float *rope_cos, const float *rope_sin,
                                       int max_position, int window, float scale, void *out,
                                       da_shape s, int q_tokens, void *stream);
/* Bytes of the multi-token workspace for a shape, T, the ring capacity (0 for paged calls)
 * and the longest sequence (with room for the rotated q and k_new of the _rope forms);
 * decode_attn_multi_reserve allocates it (call before capture). */
DA_API size_t decode_attn_multi_workspace_bytes(da_shape s, int q_tokens, int ring_window,
                                                int max_seq_len);
DA_API int decode_attn_multi_reserve(size_t bytes);
/* Kernel launches one such call makes, for the same arguments as
 * decode_attn_multi_workspace_bytes: 1 when the append is fused into the attention kernel;
 * else the attention and the append, plus a kernel that folds the key splits' partials when
 * a sequence's keys are cut into many splits. 0 for invalid arguments or without a device. */
DA_API int decode_attn_multi_launches(da_shape s, int q_tokens, int ring_window, int max_seq_len);

/*
 * kv_append -- the append alone: bit-copies k_new/v_new [B, Hkv, D] of every
 * active sequence into the cell of position p = seq_lens[b] - 1.
 * block_table != NULL: paged cache (page_size, max_pages_per_seq, num_pages as
 * above; window ignored). block_table == NULL: ring cache [B, Hkv, window, D].
 */
DA_API int kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
              const int32_t *block_table, const int32_t *seq_lens,
              int window, da_shape s, int page_size, int max_pages_per_seq,
              int num_pages, void *stream);

/*
 * decode_attn_paged_noalloc -- decode_attn_paged for callers that cannot allocate
 * device memory when they call it (a serving runtime that owns every byte of the GPU
 * through its own pool, a plugin host that forbids cudaMalloc, or code that must not
 * risk the device-wide synchronisation cudaMalloc/cudaFree can cause). Same arguments,
 * layouts and results as decode_attn_paged. The pages describe nothing like it: it is
 * an interface choice of this library, not part of the method.
 *
 * Instead of the library workspace it uses one fixed array compiled into the library
 * (1.3 MiB of device memory on every GPU that loads the library, held until the
 * process exits). It never calls cudaMalloc, cudaFree or any allocating routine.
 *   - Limits: batch * num_kv_heads <= 4096 and a GPU with at most 160 SMs; beyond
 *     that it returns DA_ERR_SCRATCH_LIMIT and launches nothing.
 *   - The first call on a device looks up the array's device address (with that device
 *     current); make that first call before any stream capture. A first call made while
 *     `stream` is capturing returns DA_ERR_WORKSPACE and launches nothing.
 *   - Every call on a device shares the one array (it clears the arrival counters it
 *     needs at the start of each call), so calls that overlap on the GPU, e.g. on two
 *     streams at once, race and give wrong results. Serialise them.
 */
DA_API int decode_attn_paged_noalloc(const void *q, const void *k_new, const void *v_new,
                                     void *k_cache, void *v_cache,
                                     const int32_t *block_table, const int32_t *seq_lens,
                                     const float *sinks, int window, float scale, void *out,
                                     da_shape s, int page_size, int max_pages_per_seq,
                                     int num_pages, int max_seq_len, void *stream);

/* Workspace the attention calls need on the current device for this shape. */
DA_API size_t decode_attn_workspace_bytes(da_shape s, int max_seq_len);

/* Make sure the current device's workspace holds at least `bytes` (allocates
 * and zeroes synchronously). Call before capturing a CUDA graph. */
DA_API int decode_attn_reserve(size_t bytes);

/*
 * decode_attn_stream_reserve -- give the attention calls issued on `stream` (a cudaStream_t
 * of the current device, as void*) workspaces of their own, so that they may run at the
 * same time as calls on other streams (two layers or two micro-batches in flight at once).
 * The pages describe one stream of kernels; this is an interface choice of the library.
 *   - `bytes` and `multi_bytes`: sizes to hold at least now, for one-token calls
 *     (decode_attn_workspace_bytes) and several-token calls
 *     (decode_attn_multi_workspace_bytes); 0 allocates nothing yet. The first call on the
 *     stream outside a capture grows a workspace that is too small, as for the device's.
 *   - Both are owned by the library, allocated and zeroed synchronously, and held until
 *     decode_attn_stream_release(stream). Calls on streams without a reservation keep
 *     using the device's workspace. Calls on one stream still run in order, so they
 *     share its workspaces safely.
 *   - Returns DA_ERR_WORKSPACE while `stream` is capturing, DA_ERR_INVALID_ARG if the
 *     stream already has workspaces on another device, DA_ERR_CUDA if allocation fails.
 */
DA_API int decode_attn_stream_reserve(void *stream, size_t bytes, size_t multi_bytes);

/*
 * decode_attn_stream_release -- synchronise `stream` and free the workspaces that
 * decode_attn_stream_reserve gave it; later calls on it use the device's workspace again.
 * A graph captured on the stream keeps the freed addresses: do not launch it afterwards.
 * Release before destroying the stream (a new stream may get the same handle). The
 * library's lock is held while the stream synchronises, so attention calls made meanwhile
 * from other host threads wait for it: release between steps, not inside one. Returns
 * DA_OK also when the stream has none, DA_ERR_WORKSPACE while it is capturing.
 */
DA_API int decode_attn_stream_release(void *stream);

/*
 * decode_attn_test_expire_wait -- a testing aid for the bounded-wait failure path. It arms a
 * one-shot: in the next one-token attention call (decode_attn_paged / _ring and their
 * _rope / _fp8 forms), the first worker gives up at its first tile wait from its tile
 * `tile` on (0-based, counted over that worker's share of the tiles), after that tile has
 * landed, exactly as if the bounded wait had expired (a worker takes its tiles two at a
 * time, one wait per pass; if its share has no wait at or after `tile`, nothing happens).
 * The call then records DA_STATUS_TIMEOUT, its output is garbage, no copy is left in
 * flight, and the library's arrival counters are back at zero for the next call. tile < 0
 * disarms. No GPU fault, trap or hang is involved. Returns DA_OK.
 */
DA_API int decode_attn_test_expire_wait(int tile);

/*
 * decode_attn_set_early_inputs -- what the attention kernels read before they wait for the
 * kernel launched just before them in the stream (process-wide). Every attention kernel is
 * launched as a programmatic dependent of that kernel: it may start while it is still
 * running and waits for it before reading anything the level below does not name.
 *   level 0 (the default): nothing is read before the wait.
 *   level 1: seq_lens, q_lens, block_table and sinks are read, the split of the keys is
 *            worked out and the block-table entries of the first tiles are loaded before the
 *            wait. Valid when those four were written before the previous kernel started
 *            (by host copies or by earlier kernels), not by that kernel.
 *   level 2: as level 1, and each worker whose share of the keys is longer than its
 *            pipeline also starts L2 prefetches of its first cache tiles before the wait.
 *            A prefetch only warms the GPU-wide L2, where a later write by the previous
 *            kernel still lands, so the cache is read for the attention after the wait as at
 *            the other levels: the conditions are those of level 1. The call's own append
 *            is applied after the wait, as at every level.
 * q, k_new, v_new, the cache and the rotary tables are always read, and the output and the
 * cache always written, after the wait. An engine that uploads a step's lengths and tables
 * before the step and then runs its layers, each attention call preceded by a projection or
 * another layer's attention, meets these conditions; so does a captured step replayed after
 * the uploads. If the previous kernel was itself launched as a programmatic dependent and
 * lets its dependents start before it has waited for its own predecessor, that predecessor
 * must meet the same conditions (this library's kernels let the next kernel start only
 * after their own wait).
 * Returns the previous level, or DA_ERR_INVALID_ARG for a level outside 0..2 (unchanged).
 */
DA_API int decode_attn_set_early_inputs(int level);

/* Wait for `stream`, then return the device status word (DA_STATUS_* bits, 0
 * if clean) of the current device and clear it; negative DA_ERR_CUDA on
 * failure. */
DA_API int decode_attn_device_status(void *stream);

/* Text for a return code; for DA_ERR_CUDA it includes the last CUDA error of
 * the calling thread. The pointer stays valid until the thread's next call. */
DA_API const char *decode_attn_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H */
