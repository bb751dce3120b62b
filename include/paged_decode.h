/*
 * paged_decode.h -- C ABI of the GB300 (sm_103a) paged GQA decode library:
 * ReshapeAndCache, dense GQA paged decode attention with split-KV, and Quest
 * sparse paged attention (per-block min/max key metadata, block scoring,
 * top-K selection, attention over the selected blocks).
 *
 * Sources (web pages, by title and section):
 *   [P1] "Ascend Kernel-to-Serving Pipeline": sections "ReshapeAndCache",
 *        "GQA Paged Attention", "Quest Sparse Attention", "Sparse precision".
 *   [P2] "18 e2e inference serving" (TileLang tutorial): 2.4 (decode
 *        attention is memory-bound), 2.6 (paged KV layout, block table),
 *        4.1 (split-KV partial outputs combined with l_s weights), 6.1 (run on
 *        the framework's current stream).
 *   The Quest scoring rule (per-block elementwise min/max of K; score =
 *   sum over the GQA group of sum_d max(q_d*min_d, q_d*max_d); top-K with ties
 *   to the lower block index) is part of the method's statement; the pages
 *   only say "score logical blocks cheaply, keep the top-K" ([P1] "Quest").
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers owned by the caller; the library never
 *     allocates device memory. Scratch space comes from a caller-provided
 *     workspace whose size a *_workspace_size() function returns.
 *   - bf16 tensors are passed as pa_bf16 (the raw 16-bit pattern).
 *   - Layouts are contiguous, row-major:
 *       query / out      [B][Hq][D]
 *       key / value      [T][Hkv][D]         (this step's new tokens)
 *       key_cache,
 *       value_cache      [NB][BS][Hkv][D]    (one layer, [P2] 2.6)
 *       kmin / kmax      [NB][Hkv][D]        (Quest metadata per physical block)
 *       block_tables     [B][MBS] int32      (logical -> physical block)
 *       context_lens     [B] int32           (valid tokens, including this step's)
 *       slot_mapping     [T] int64           (flat slot = block * BS + offset)
 *       selected         [B][Hkv][topk] int32 (logical blocks, ascending, -1 padded)
 *   - Query head h reads KV head h / (Hq / Hkv) ([P1] "GQA Paged Attention":
 *     Hq is an integer multiple of Hkv).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every call
 *     is asynchronous on that stream and returns a pa_status. Argument errors
 *     are detected on the host before anything is launched.
 *   - Kernels launch with programmatic stream serialization: a kernel may
 *     start while the previous kernel in the stream finishes, and waits for
 *     it before reading anything that kernel may write. The exceptions are
 *     context_lens (read before that wait by every decode and selection
 *     call, and cu_seqlens_q by pa_decode_multi) and block_tables (read
 *     before it by the bf16 dense decode and by the selection's score
 *     kernel). No kernel of this library writes them. A caller kernel that
 *     writes them and lets dependent launches start early must not run just
 *     before such a call. A kernel that never triggers early starts its
 *     dependents only when it completes, so the usual case is safe.
 *   - Supported shapes: head_dim D in {64, 128}; block_size BS = 16;
 *     group size Hq / Hkv in 1..8; B <= 4096.
 *   - Device data is never trusted to the point of a fault: negative or
 *     out-of-pool slots are skipped, context_lens are clamped to
 *     [0, MBS * BS], block-table entries outside [0, NB) make that block read
 *     as empty (no tokens). pa_check_metadata() reports such entries.
 *   - The library keeps no state between calls except per-device launch
 *     parameters computed on first use.
 */
#ifndef PAGED_DECODE_H
#define PAGED_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points are the only symbols the shared library exports. */
#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef uint16_t pa_bf16; /* bfloat16 bit pattern */
typedef uint8_t pa_e4m3;  /* 8-bit float, E4M3 variant (see the 8-bit cache section) */

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, Hq % Hkv != 0 ... */
    PA_ERR_UNSUPPORTED = -2, /* shape outside the supported set listed above */
    PA_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required */
    PA_ERR_CUDA = -4,        /* a CUDA runtime/driver call or launch failed */
    PA_ERR_DEVICE = -5       /* a kernel recorded a device-side failure (timeout) */
} pa_status;

/* Human-readable name of a pa_status value (static storage). */
PA_API const char *pa_status_string(int status);

/* The CUDA error code of the last PA_ERR_CUDA returned on this thread. */
PA_API int pa_last_cuda_error(void);

/* ReshapeAndCache ([P1] "ReshapeAndCache"): for every token t < num_tokens
 * with slot = slot_mapping[t] >= 0, copies key[t] and value[t] (all KV heads)
 * to key_cache / value_cache at block slot / block_size, offset
 * slot % block_size. Negative slots are skipped; slots >= num_blocks *
 * block_size are skipped as well. Slots must be distinct (two tokens writing
 * one slot race). num_tokens == 0 is a no-op. */
PA_API int pa_reshape_and_cache(const pa_bf16 *key, const pa_bf16 *value,
                         pa_bf16 *key_cache, pa_bf16 *value_cache,
                         const int64_t *slot_mapping, int64_t num_tokens,
                         int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, void *stream);

/* Bytes of workspace pa_decode / quest_sparse_decode need on the CURRENT
 * device for this batch and head shape (0 on invalid arguments). The
 * workspace holds split-KV partial outputs, their log-sum-exp, per-sequence
 * arrival counters and a status word. It must be ZERO-FILLED before its first
 * use; every successful call leaves it zeroed again, so one buffer can serve
 * any number of sequential calls on one stream. Calls that overlap in time
 * must use different workspaces. */
PA_API size_t pa_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim);

/* Dense GQA paged decode attention ([P1] "GQA Paged Attention"; split-KV and
 * combine per [P2] 4.1). One query token per sequence:
 *   out[b][h] = softmax_t(scale * query[b][h] . K[b][t]) . V[b][t]
 * over t < context_lens[b], with K/V[b][t] at key/value_cache
 * [block_tables[b][t / BS]][t % BS][h / G]. The score vector is never
 * materialised (online softmax, fp32 accumulation); the KV range of the batch
 * is split evenly over the GPU's warps and partial results are merged with
 * log-sum-exp weights. out is bf16 (round to nearest even); a sequence with
 * context_lens[b] == 0 gets a zero output. */
PA_API int pa_decode(pa_bf16 *out, const pa_bf16 *query,
              const pa_bf16 *key_cache, const pa_bf16 *value_cache,
              const int32_t *block_tables, int max_blocks_per_seq,
              const int32_t *context_lens, int batch, int num_q_heads,
              int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
              float scale, void *workspace, size_t workspace_bytes, void *stream);

/* pa_decode on at most max_ctas CTAs (max_ctas 0, or at least one per SM:
 * one CTA per SM, as pa_decode; max_ctas < 0 is PA_ERR_INVALID_ARG). For a
 * step that runs other work on its own stream beside the dense decode: a
 * decode CTA takes a whole SM's shared memory, and its persistent grid cuts
 * the batch's KV blocks into max_ctas equal ranges, so the SMs beyond
 * max_ctas stay free for the other stream. The split-KV pieces, and so the
 * rounding of the result, depend on max_ctas; for a given max_ctas the result
 * is deterministic. Workspace: as pa_decode. */
PA_API int pa_decode_budget(pa_bf16 *out, const pa_bf16 *query,
                     const pa_bf16 *key_cache, const pa_bf16 *value_cache,
                     const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *context_lens, int batch, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                     float scale, int max_ctas, void *workspace, size_t workspace_bytes,
                     void *stream);

/* Size of the fixed scratch buffer behind pa_decode_no_alloc (8 MiB). */
#define PA_NO_ALLOC_SCRATCH_BYTES (8u << 20)

/* pa_decode for callers that may not allocate device memory at all (no
 * counterpart on the pages; an addition of this library). Examples: a plugin
 * inside a serving engine that is handed only its input and output tensors
 * while the engine keeps the rest of HBM for its KV-cache pool, or a
 * latency-critical loop where cudaMalloc/cudaFree are not allowed because
 * they can synchronise the device. Same arguments and result as pa_decode,
 * without a workspace: the scratch is a PA_NO_ALLOC_SCRATCH_BYTES buffer
 * compiled into the library, present on every GPU that loads it until the
 * process exits. The call allocates nothing. Its first call on a device
 * looks up that buffer's device address (make that first call before any
 * stream capture). Every call clears the buffer's status word and counters on
 * `stream` and then runs pa_decode's kernel; all calls share the one buffer,
 * so calls that overlap on the GPU race. Returns PA_ERR_WORKSPACE when the
 * batch and head shape need more scratch than the buffer holds (about
 * B * Hkv + number_of_SMs partial slots of (8 * head_dim + 8) floats).
 * A kernel that gave up on a bounded wait (the output is then undefined) is
 * reported by pa_decode_no_alloc_status, which must be read before the next
 * pa_decode_no_alloc call on that device clears the status word. */
PA_API int pa_decode_no_alloc(pa_bf16 *out, const pa_bf16 *query,
                              const pa_bf16 *key_cache, const pa_bf16 *value_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int batch, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                              float scale, void *stream);

/* Device-side status of the last pa_decode_no_alloc call on the current
 * device: waits for `stream`, then reads the fixed buffer's status word.
 * PA_OK, PA_ERR_DEVICE if that call's kernel gave up on a bounded wait, or
 * PA_ERR_INVALID_ARG if pa_decode_no_alloc has not run on this device yet.
 * Allocates nothing. */
PA_API int pa_decode_no_alloc_status(void *stream);

/* Quest metadata update for the tokens of one ReshapeAndCache call. For each
 * physical block touched by a valid slot: if one of the call's tokens lands
 * at offset 0 (the block starts fresh) the block's kmin/kmax become the
 * elementwise min/max over the call's tokens in that block; otherwise they
 * become min/max of the old values and those tokens. min/max follow IEEE
 * totalOrder (-0 < +0), so the result is independent of token order.
 * Slots must be the ones passed to pa_reshape_and_cache (same skip rules). */
PA_API int quest_update_meta(pa_bf16 *kmin, pa_bf16 *kmax, const pa_bf16 *key,
                      const int64_t *slot_mapping, int64_t num_tokens,
                      int num_kv_heads, int head_dim, int block_size,
                      int64_t num_blocks, void *stream);

/* The write path in one launch: pa_reshape_and_cache followed by
 * quest_update_meta on the same tokens, with identical results (the fused
 * KV-update step of "Day-0 porting of a sparse-attention model", section on
 * the prefill/decode pipeline, where the cache update is folded into one
 * kernel launch). Same argument rules as the two calls it replaces. */
PA_API int quest_reshape_and_cache(const pa_bf16 *key, const pa_bf16 *value,
                                   pa_bf16 *key_cache, pa_bf16 *value_cache,
                                   pa_bf16 *kmin, pa_bf16 *kmax,
                                   const int64_t *slot_mapping, int64_t num_tokens,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int64_t num_blocks, void *stream);

/* Quest metadata from scratch: for every sequence b and logical block
 * j < ceil(context_lens[b] / BS), kmin/kmax of physical block
 * block_tables[b][j] = elementwise min/max of K over the block's valid tokens
 * (positions < context_lens[b]). Blocks no sequence uses are left as they are. */
PA_API int quest_rebuild_meta(pa_bf16 *kmin, pa_bf16 *kmax, const pa_bf16 *key_cache,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, int batch, int num_kv_heads,
                       int head_dim, int block_size, int64_t num_blocks, void *stream);

/* Bytes of workspace quest_select_topk needs (0 on invalid arguments). The
 * first batch * num_kv_heads * max_blocks_per_seq floats of the workspace hold
 * the block scores [B][Hkv][MBS] after the call (entries for blocks past a
 * sequence's context are not written). No zero-fill needed. */
PA_API size_t quest_select_workspace_size(int batch, int num_kv_heads, int max_blocks_per_seq);

/* Quest block selection ([P1] "Quest Sparse Attention"). For each sequence b
 * and KV head g, every logical block j < ceil(context_lens[b] / BS) gets the
 * score  sum_{h in group g} sum_d max(q[b,h,d]*kmin[p,g,d], q[b,h,d]*kmax[p,g,d])
 * with p = block_tables[b][j] (an upper bound of the group's summed logits on
 * that block). The score is computed in fp32 in one fixed order:
 *   P_d = sum_h max(q,0), N_d = sum_h min(q,0) (h ascending, from +0);
 *   t_d = fl(fl(P_d*kmax_d) + fl(N_d*kmin_d));
 *   D split into 32 chunks of D/32 consecutive d, each summed left to right;
 *   the 32 chunk sums combined by a xor-butterfly (offsets 16, 8, 4, 2, 1).
 * The topk highest-scoring blocks are selected (ties: the lower block index;
 * scores compared in IEEE totalOrder) and written ascending to
 * selected[b][g][0..), the rest of the row padded with -1. If a sequence has
 * no more than topk blocks, all of them are selected. */
PA_API int quest_select_topk(int32_t *selected, const pa_bf16 *query,
                      const pa_bf16 *kmin, const pa_bf16 *kmax,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int batch, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                      int topk, void *workspace, size_t workspace_bytes, void *stream);

/* Quest sparse paged attention ([P1] "Quest Sparse Attention", "Sparse
 * precision"): exact attention, as pa_decode, over only the tokens of the
 * logical blocks listed in selected[b][h / G][0..topk) (entries < 0 or past
 * the sequence's blocks are ignored; entries must be distinct), tokens at
 * positions >= context_lens[b] masked. Uses the same workspace as pa_decode
 * (size from pa_decode_workspace_size, same zero-fill rule). */
PA_API int quest_sparse_decode(pa_bf16 *out, const pa_bf16 *query,
                        const pa_bf16 *key_cache, const pa_bf16 *value_cache,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, const int32_t *selected, int topk,
                        int batch, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int64_t num_blocks, float scale,
                        void *workspace, size_t workspace_bytes, void *stream);

/* quest_sparse_decode with a cap on the CTAs it launches (max_ctas 0: the
 * default of quest_sparse_decode, half the SMs when the batch's (sequence,
 * KV head) segments fit in them, else one CTA per SM; max_ctas < 0 is
 * PA_ERR_INVALID_ARG). For a
 * step that runs the sparse decode on its own stream beside a dense
 * pa_decode: each sparse CTA needs a whole SM's shared memory, so they start
 * as the dense call's CTAs finish, and a smaller grid lets the sparse call
 * complete without waiting for the last of them. The split-KV pieces, and so
 * the rounding of the result, depend on max_ctas; for a given max_ctas the
 * result is deterministic. */
PA_API int quest_sparse_decode_budget(pa_bf16 *out, const pa_bf16 *query,
                               const pa_bf16 *key_cache, const pa_bf16 *value_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, const int32_t *selected, int topk,
                               int batch, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int64_t num_blocks, float scale, int max_ctas,
                               void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace quest_decode / quest_decode_fp8 need (0 for an invalid
 * or unsupported shape): the pa_decode workspace, then the block scores. */
PA_API size_t quest_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                          int max_blocks_per_seq);

/* The Quest path after the write ([P1] "Quest Sparse Attention": score the
 * blocks, keep the top-K, attend over those only) in two launches:
 * quest_select_topk's block scores, then one sparse-decode launch whose CTAs
 * each select the top-K blocks of their own (sequence, KV head) segments
 * from those scores and attend over them. Results: `selected` [B][Hkv][topk]
 * exactly as quest_select_topk writes it, and `out` as quest_sparse_decode
 * on that selection (with the same max_ctas, bit for bit). It saves the
 * top-K launch and the selection's round trip through global memory. For a
 * large selection (batch * num_kv_heads * topk at least 96 items per SM),
 * where every sparse CTA would hold several whole segments and select for
 * each in turn, it runs quest_select_topk and quest_sparse_decode_budget
 * instead (three launches, the same results).
 * max_ctas: as quest_sparse_decode_budget (0: the default). Workspace:
 * quest_decode_workspace_size bytes, zero-filled once, as pa_decode's (the
 * scores follow the decode part). Errors as quest_select_topk and
 * quest_sparse_decode. */
PA_API int quest_decode(pa_bf16 *out, int32_t *selected, const pa_bf16 *query,
                 const pa_bf16 *kmin, const pa_bf16 *kmax,
                 const pa_bf16 *key_cache, const pa_bf16 *value_cache,
                 const int32_t *block_tables, int max_blocks_per_seq,
                 const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
                 int head_dim, int block_size, int64_t num_blocks, int topk, float scale,
                 int max_ctas, void *workspace, size_t workspace_bytes, void *stream);

/* Reads the status word a pa_decode / quest_sparse_decode workspace carries
 * (synchronises `stream`): PA_OK, or PA_ERR_DEVICE if a kernel gave up on a
 * wait (its output is then undefined and the workspace must be zero-filled
 * again before reuse). */
PA_API int pa_workspace_status(const void *workspace, void *stream);

/* Input checker (not on the hot path). Counts, on the device, into
 * counts[0..3] (device int32, overwritten):
 *   [0] slots >= num_blocks * block_size,
 *   [1] context_lens outside [0, max_blocks_per_seq * block_size],
 *   [2] block-table entries j < ceil(ctx/BS) outside [0, num_blocks),
 *   [3] valid slots that repeat an earlier token's slot.
 * Any pointer may be NULL (with its count 0) to skip that check. */
PA_API int pa_check_metadata(int32_t *counts, const int64_t *slot_mapping, int64_t num_tokens,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int batch, int block_size,
                      int64_t num_blocks, void *stream);

/* Multi-token query rows ([P2] 2.7 "continuous batching and varlen": a
 * chunked-prefill chunk or speculative tokens mixed into a decode batch;
 * [P2] 3.3: flat query rows with cu_seqlens_q, causal mask aligned on the
 * right). Sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
 * of query / out [total_q][Hq][D]: its q_len = cu[b+1] - cu[b] newest tokens,
 * at positions context_lens[b] - q_len .. context_lens[b] - 1 (context_lens
 * includes them, and ReshapeAndCache has written their K/V). Row i of
 * sequence b attends, as pa_decode, to the positions
 *     t < context_lens[b] - q_len + i + 1
 * (itself and everything before it); a row whose limit is <= 0 gets a zero
 * output. cu_seqlens_q is [batch + 1] int32 on the device, 0 = cu[0] <= ... <=
 * cu[batch] = total_q (not checked on the host; a malformed array gives
 * undefined rows, never a fault). block_tables and context_lens are per
 * sequence. Up to 4 query rows of a sequence share one pass over its KV.
 * Workspace: pa_decode_multi_workspace_size(total_q, ...) bytes, zero-filled
 * once like pa_decode's. Supported: batch, total_q <= 2048; other limits as
 * pa_decode. */
PA_API size_t pa_decode_multi_workspace_size(int total_q, int num_q_heads, int num_kv_heads, int head_dim);

PA_API int pa_decode_multi(pa_bf16 *out, const pa_bf16 *query,
                    const pa_bf16 *key_cache, const pa_bf16 *value_cache,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *cu_seqlens_q, const int32_t *context_lens,
                    int batch, int total_q, int num_q_heads, int num_kv_heads,
                    int head_dim, int block_size, int64_t num_blocks, float scale,
                    void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------- the step's write folded into decode ----
 * A decode step writes each sequence's new token into the cache ([P1]
 * "ReshapeAndCache", and the Quest metadata update) and then attends over
 * the cache including it. These two calls fold that write into the step's
 * first launch, for the decode case: one new token per sequence, at its
 * position ctx_b - 1.
 *
 * key, value: [batch][Hkv][D] bf16, the new token of each sequence;
 * slot_mapping: [batch] int64. Token b is written at slot_mapping[b] when
 * that is the slot of position ctx_b - 1 of sequence b, i.e.
 *     block_tables[b][(ctx_b - 1) / BS] * BS + (ctx_b - 1) % BS
 * with that table entry inside the pool. Any other slot (negative, past the
 * pool, or another position) is not written. pa_reshape_and_cache writes any
 * in-pool slot instead. The slots of one call must be distinct, and no other
 * kernel may touch the written blocks while the call runs. With those slots,
 * the results are byte for byte those of the separate calls (the write, then
 * pa_decode or quest_decode): caches, metadata, selection and outputs.
 * bf16 cache only; 16-byte aligned key and value. Workspaces and errors as
 * pa_decode / quest_decode. */

/* ReshapeAndCache of the step's tokens, then pa_decode, in one launch: the
 * CTA that reads a sequence's last block writes the new token's slice of
 * its KV head into it first. kmin / kmax: both null, or the Quest metadata,
 * updated as quest_update_meta does (reset when the token lands at offset 0
 * of its block, else merged). */
PA_API int pa_reshape_and_decode(pa_bf16 *out, const pa_bf16 *query, const pa_bf16 *key,
                                 const pa_bf16 *value, const int64_t *slot_mapping,
                                 pa_bf16 *key_cache, pa_bf16 *value_cache, pa_bf16 *kmin,
                                 pa_bf16 *kmax, const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *context_lens, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                 float scale, void *workspace, size_t workspace_bytes, void *stream);

/* quest_reshape_and_cache of the step's tokens, then quest_decode, in two
 * launches: the score launch's warp that scores a sequence's last block
 * writes the new token's slice of its KV head and updates the block's
 * metadata before scoring it; then the fused top-K and sparse decode. */
PA_API int quest_reshape_and_decode(pa_bf16 *out, int32_t *selected, const pa_bf16 *query,
                                    const pa_bf16 *key, const pa_bf16 *value,
                                    const int64_t *slot_mapping, pa_bf16 *kmin, pa_bf16 *kmax,
                                    pa_bf16 *key_cache, pa_bf16 *value_cache,
                                    const int32_t *block_tables, int max_blocks_per_seq,
                                    const int32_t *context_lens, int batch, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int64_t num_blocks, int topk, float scale, int max_ctas,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------- 8-bit KV cache ----
 * The same path over a KV cache stored in 8 bits per element, which halves
 * the bytes decode attention reads ([P2] 2.5 and 3.1: long-context serving is
 * bound by KV bandwidth, and KV quantisation is the lever the tutorial names).
 *
 * Format: the E4M3 variant of the OCP 8-bit float ("fn": sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits, no infinities, largest finite 448,
 * 0x7F / 0xFF NaN). Element d of KV head h of a token is stored as
 *     code = e4m3(fl32(x / scale[h])),
 * rounded to nearest with ties to the even mantissa, magnitudes beyond 448
 * (and infinities) saturated to +-448, NaN stored as 0x7F; it stands for
 * decode(code) * scale[h]. k_scale and v_scale are [Hkv] fp32 device arrays,
 * positive and finite, fixed by the caller for the cache's lifetime (a
 * calibration outside this library). Quest metadata of an 8-bit cache are
 * E4M3 codes too: the elementwise min / max of the stored K codes (numeric
 * order, -0 < +0), [NB][Hkv][D] bytes.
 *
 * Layouts: key_cache [NB][BS][Hkv][D] bytes (as the bf16 cache) and kmin /
 * kmax [NB][Hkv][D] bytes; value_cache [NB][Hkv][D][BS] bytes: per block and
 * KV head a dim-by-token matrix whose 16-byte row of dim d holds the block's
 * tokens in the order 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15 (token o at byte
 * 4*((o%8)/2) + 2*(o/8) + o%2), the order the attention kernel's fragment
 * loads take it in. Supported: head_dim 128, block_size 16; 16-byte aligned
 * pointers. Queries stay bf16; the
 * attention converts them to f16 (values outside the f16 range, about
 * 6.1e-5 .. 65504 in magnitude, are rounded or overflow there), multiplies
 * exactly decoded K / V codes in f16 with fp32 accumulation, and applies the
 * scales in fp32. The decode workspace is the one pa_decode uses. */

/* ReshapeAndCache into an 8-bit cache: the slot arithmetic of
 * pa_reshape_and_cache ([P1] "ReshapeAndCache"), each element quantised as
 * above with its KV head's scale. */
PA_API int pa_reshape_and_cache_fp8(const pa_bf16 *key, const pa_bf16 *value,
                             pa_e4m3 *key_cache, pa_e4m3 *value_cache,
                             const int64_t *slot_mapping, int64_t num_tokens,
                             const float *k_scale, const float *v_scale, int num_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks, void *stream);

/* Metadata update of an 8-bit cache for this call's tokens: the rule of
 * quest_update_meta on the tokens' codes (the codes pa_reshape_and_cache_fp8
 * stores). */
PA_API int quest_update_meta_fp8(pa_e4m3 *kmin, pa_e4m3 *kmax, const pa_bf16 *key,
                          const int64_t *slot_mapping, int64_t num_tokens,
                          const float *k_scale, int num_kv_heads, int head_dim,
                          int block_size, int64_t num_blocks, void *stream);

/* pa_reshape_and_cache_fp8 followed by quest_update_meta_fp8, one launch. */
PA_API int quest_reshape_and_cache_fp8(const pa_bf16 *key, const pa_bf16 *value,
                                pa_e4m3 *key_cache, pa_e4m3 *value_cache,
                                pa_e4m3 *kmin, pa_e4m3 *kmax,
                                const int64_t *slot_mapping, int64_t num_tokens,
                                const float *k_scale, const float *v_scale, int num_kv_heads,
                                int head_dim, int block_size, int64_t num_blocks, void *stream);

/* Metadata of every block the sequences use, recomputed from an 8-bit cache
 * (as quest_rebuild_meta). */
PA_API int quest_rebuild_meta_fp8(pa_e4m3 *kmin, pa_e4m3 *kmax, const pa_e4m3 *key_cache,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int batch, int num_kv_heads,
                           int head_dim, int block_size, int64_t num_blocks, void *stream);

/* Quest selection on 8-bit metadata: the score of quest_select_topk with
 * kmin_d / kmax_d the decoded codes (exact in fp32), same evaluation order,
 * same top-K rule and workspace. The cache's K scale is left out: it
 * multiplies every score of a (sequence, KV head) row by one positive factor
 * and cannot change that row's selection. */
PA_API int quest_select_topk_fp8(int32_t *selected, const pa_bf16 *query,
                          const pa_e4m3 *kmin, const pa_e4m3 *kmax,
                          const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *context_lens, int batch, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                          int topk, void *workspace, size_t workspace_bytes, void *stream);

/* Dense GQA paged decode attention ([P1] "GQA Paged Attention", split-KV per
 * [P2] 4.1) over an 8-bit cache: pa_decode with K and V read as
 * decode(code) * scale[kvh]. Same workspace and status rules as pa_decode. */
PA_API int pa_decode_fp8(pa_bf16 *out, const pa_bf16 *query,
                  const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                  const float *k_scale, const float *v_scale,
                  const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
                  int head_dim, int block_size, int64_t num_blocks, float scale,
                  void *workspace, size_t workspace_bytes, void *stream);

/* pa_decode_fp8 on at most max_ctas CTAs (as pa_decode_budget). */
PA_API int pa_decode_fp8_budget(pa_bf16 *out, const pa_bf16 *query,
                         const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                         const float *k_scale, const float *v_scale,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, float scale, int max_ctas,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Quest sparse attention ([P1] "Quest Sparse Attention") over an 8-bit
 * cache: quest_sparse_decode with K and V decoded as in pa_decode_fp8. */
PA_API int quest_sparse_decode_fp8(pa_bf16 *out, const pa_bf16 *query,
                            const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *selected, int topk,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, float scale,
                            void *workspace, size_t workspace_bytes, void *stream);

/* quest_sparse_decode_fp8 with a cap on the CTAs it launches, as
 * quest_sparse_decode_budget. */
PA_API int quest_sparse_decode_fp8_budget(pa_bf16 *out, const pa_bf16 *query,
                                   const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                                   const float *k_scale, const float *v_scale,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, const int32_t *selected, int topk,
                                   int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int64_t num_blocks, float scale, int max_ctas,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* quest_decode over an 8-bit cache: quest_select_topk_fp8's scores, then the
 * fused selection and quest_sparse_decode_fp8. */
PA_API int quest_decode_fp8(pa_bf16 *out, int32_t *selected, const pa_bf16 *query,
                     const pa_e4m3 *kmin, const pa_e4m3 *kmax,
                     const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                     const float *k_scale, const float *v_scale,
                     const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int64_t num_blocks, int topk, float scale,
                     int max_ctas, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------- 8-bit KV cache with per-block scales ----
 * The 8-bit cache with one K scale and one V scale per (physical block, KV
 * head) instead of per KV head ([P2] 2.5 and 3.1 name KV quantisation as the
 * long-context lever; a per-block scale is the form that needs no
 * calibration and follows each block's range). Same E4M3 code format and
 * cache / metadata layouts as above; the scales are k_bscale and v_bscale,
 * [NB][Hkv] fp32 device arrays, read and written by the library: each entry
 * is a power of two 2^e (-126 <= e <= 127), or 0 for a block that holds
 * nothing yet (a new pool starts all zeros). A stored element stands for
 * decode(code) * scale[p][h] of its block p.
 *
 * Writing (pa_reshape_and_cache_fp8_block): for every physical block p a
 * call writes into, per KV head and for K and V separately,
 *   a      = the largest finite |x| over the call's tokens in p;
 *   e_call = the smallest integer e >= -126 with a <= 448 * 2^e;
 *   if a token of the call lands at offset 0 (the block restarts) or the
 *   stored scale is 0: e = e_call; else e = max(e_old, e_call) with
 *   2^e_old the stored scale;
 *   when e > e_old, every code of the block at an offset the call does not
 *   write is re-encoded as e4m3(decode(code) * 2^(e_old - e)): exact while
 *   the value stays in the E4M3 normal range (>= 2^-6), rounded to nearest
 *   (ties to even) below it;
 *   the call's elements are stored as e4m3(x / 2^e) (nearest, ties to even;
 *   infinities saturate to +-448, NaN becomes 0x7F) and the scale becomes 2^e.
 * The Quest metadata (quest_reshape_and_cache_fp8_block) follow the same
 * rule as quest_update_meta_fp8 on the re-encoded codes: on a restart the
 * min / max of the call's codes, else the stored min / max, re-encoded like
 * the codes when e grew, merged with the call's codes. The slots of one call
 * must be distinct. quest_rebuild_meta_fp8 works unchanged on this cache.
 *
 * Reading: the attention dequantises each block's K and V with its own
 * scales; the Quest score of a block is the score of its stored metadata
 * times the block's K scale (one fp32 product: the blocks' scales differ,
 * so it can change the top-K). */

/* ReshapeAndCache into an 8-bit cache with per-block scales (k_bscale,
 * v_bscale updated in place), one launch. Same argument rules as
 * pa_reshape_and_cache_fp8. */
PA_API int pa_reshape_and_cache_fp8_block(const pa_bf16 *key, const pa_bf16 *value,
                                          pa_e4m3 *key_cache, pa_e4m3 *value_cache,
                                          const int64_t *slot_mapping, int64_t num_tokens,
                                          float *k_bscale, float *v_bscale, int num_kv_heads,
                                          int head_dim, int block_size, int64_t num_blocks,
                                          void *stream);

/* pa_reshape_and_cache_fp8_block and the Quest metadata update, one launch. */
PA_API int quest_reshape_and_cache_fp8_block(const pa_bf16 *key, const pa_bf16 *value,
                                             pa_e4m3 *key_cache, pa_e4m3 *value_cache,
                                             pa_e4m3 *kmin, pa_e4m3 *kmax,
                                             const int64_t *slot_mapping, int64_t num_tokens,
                                             float *k_bscale, float *v_bscale, int num_kv_heads,
                                             int head_dim, int block_size, int64_t num_blocks,
                                             void *stream);

/* quest_select_topk_fp8 on a cache with per-block scales: every block's
 * score is the metadata score times k_bscale[p][kvh] (p its physical block),
 * then the same top-K rule and workspace. */
PA_API int quest_select_topk_fp8_block(int32_t *selected, const pa_bf16 *query,
                                       const pa_e4m3 *kmin, const pa_e4m3 *kmax,
                                       const float *k_bscale, const int32_t *block_tables,
                                       int max_blocks_per_seq, const int32_t *context_lens,
                                       int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int64_t num_blocks, int topk,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* pa_decode_fp8 on a cache with per-block scales: K and V of physical block
 * p read as decode(code) * k_bscale[p][kvh] (v_bscale alike). */
PA_API int pa_decode_fp8_block(pa_bf16 *out, const pa_bf16 *query,
                               const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                               const float *k_bscale, const float *v_bscale,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int batch, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               float scale, void *workspace, size_t workspace_bytes, void *stream);

/* pa_decode_fp8_block on at most max_ctas CTAs (as pa_decode_budget). */
PA_API int pa_decode_fp8_block_budget(pa_bf16 *out, const pa_bf16 *query,
                               const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                               const float *k_bscale, const float *v_bscale,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int batch, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               float scale, int max_ctas, void *workspace, size_t workspace_bytes,
                               void *stream);

/* quest_sparse_decode_fp8_budget on a cache with per-block scales
 * (max_ctas 0: the default). */
PA_API int quest_sparse_decode_fp8_block(pa_bf16 *out, const pa_bf16 *query,
                                         const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                                         const float *k_bscale, const float *v_bscale,
                                         const int32_t *block_tables, int max_blocks_per_seq,
                                         const int32_t *context_lens, const int32_t *selected,
                                         int topk, int batch, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int64_t num_blocks,
                                         float scale, int max_ctas, void *workspace,
                                         size_t workspace_bytes, void *stream);

/* quest_decode_fp8 on a cache with per-block scales: the block-scaled scores,
 * then the fused selection and sparse decode (or, for a large selection,
 * quest_select_topk_fp8_block and quest_sparse_decode_fp8_block). */
PA_API int quest_decode_fp8_block(pa_bf16 *out, int32_t *selected, const pa_bf16 *query,
                                  const pa_e4m3 *kmin, const pa_e4m3 *kmax,
                                  const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                                  const float *k_bscale, const float *v_bscale,
                                  const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *context_lens, int batch, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                  int topk, float scale, int max_ctas, void *workspace,
                                  size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_DECODE_H */
