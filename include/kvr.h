/*
 * kvr.h -- C ABI of libkvr: the online hot path of precomputed-KV RAG on one
 * GPU (GB300, sm_103a).
 *
 * A request's prefix is stitched out of token spans [start, end) of per-chunk
 * KV caches that were computed offline at chunk-local positions; keys are
 * re-rotated (RoPE) so the spans form one contiguous prefix, values are copied
 * unchanged; then the request's query tokens run prefill attention over that
 * prefix, seeing the whole prefix and, causally, each other.
 *
 *   CoinRAG blog (liuzhao09.github.io, "CoinRAG: contextualized information
 *   nugget KV cache reuse"), section 2.2: a retrieval result is a list of
 *   triples (chunk b_i, start s_i, end e_i);
 *   section 2.3: C_ctx = C_p (+) Rot(C_b1[s1:e1]; D1) (+) ... (+) Rot(C_bk[sk:ek]; Dk),
 *   with D_i = |p| + sum_{j<i} len_j, and KV_CoinRAG = C_ctx (+) KV_M(q; C_ctx).
 *   TurboRAG blog (shibing624), "Attention Mask" and "Position ID": chunks are
 *   independent, the query attends to every chunk and to itself; positions
 *   are reordered to be contiguous, RoPE re-applied at the new positions.
 *   SemPIC page (agihunt.info): on a cache hit, re-rotate the compiled
 *   document keys at their final positions and interleave the request's own
 *   inline tokens under a causal mask.
 *
 * Conventions shared by every call:
 *   - Device pointers are CUDA device memory owned by the caller.  The library
 *     never frees them and keeps none past the call, except the pool pointers
 *     that a registered pool holds until kvr_pool_unregister.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls enqueue work on it and return without waiting for the GPU, with
 *     these exceptions, which are the library's only allocations and waits:
 *       1. kvr_check synchronizes the stream.
 *       2. The first call that enqueues work on a pool (or kvr_pool_reserve)
 *          binds it to the current device: it allocates the RoPE tables
 *          (4 MiB for head_dim 128) and an error word and builds the tables,
 *          synchronously.
 *       3. Staging slots.  A call whose span, local-source or request tables
 *          do not fit inside its kernels' parameters (more than 64 spans,
 *          local sources or requests) copies them up from one of the pool's
 *          8 pinned staging slots, taken in turn.  A slot is allocated on
 *          first use, and freed and allocated larger when a call needs more
 *          (cudaFreeHost / cudaFree synchronize the device).  If the slot's
 *          previous call has not yet run on the GPU (8 such calls queued
 *          ahead of it), the call waits on the host for it.
 *       4. Query scratch (tensor-core attention: bf16, head_dim 128).  The
 *          rotated query heads of a call need n_layers * T * n_q_heads *
 *          head_dim * 2 bytes of device memory (T = query tokens of the
 *          call).  A call with more than the scratch holds waits for the
 *          previous call's attention, frees it and allocates it larger.
 *       5. A pool in pinned host memory: the first kvr_prefill on it creates
 *          an internal stream and its events (kept until unregister).
 *     kvr_pool_reserve makes 3 and 4 happen up front: afterwards, calls
 *     within the reserved sizes allocate nothing and wait only in the one
 *     case of 3 (8 calls with uploaded tables still queued).  kvr_pool_unregister
 *     synchronizes the handle's work before it frees.
 *   - Every failure is a returned kvr_status; nothing aborts or traps.  Host
 *     validation runs before any launch, so an error status from validation
 *     means nothing was enqueued.  kvr_last_error() gives a one-line reason.
 *   - A pool handle may be used by one host thread at a time.
 *   - Layouts are row-major, head_dim contiguous; element strides are in
 *     elements, not bytes.
 */
#ifndef KVR_H
#define KVR_H

#include <stdint.h>

#if defined(__GNUC__)
#define KVR_API __attribute__((visibility("default")))
#else
#define KVR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVR_OK = 0,
    KVR_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, stride or alignment */
    KVR_ERR_OUT_OF_RANGE = 2,  /* span or offset outside its source / cache    */
    KVR_ERR_UNSUPPORTED = 3,   /* dtype / head_dim / GPU this build cannot run */
    KVR_ERR_CUDA = 4,          /* a CUDA runtime call failed                    */
    KVR_ERR_TIMEOUT = 5,       /* a kernel's bounded wait ran out (kvr_check)   */
    KVR_ERR_DEVICE_CHECK = 6   /* a kernel flagged bad device-side input        */
} kvr_status;

enum { KVR_DTYPE_BF16 = 0, KVR_DTYPE_FP32 = 1 };

/* Span source flag: src = KVR_SRC_LOCAL | i names request-local source i
 * (inline tokens) instead of pool entry src. */
#define KVR_SRC_LOCAL (1 << 30)

/* kvr_assemble flag: composite positions (every span keeps its chunk-local
 * ids, no re-rotation) instead of the default reordered contiguous positions.
 * TurboRAG blog, "Position ID", Figure 5. */
#define KVR_POSITIONS_COMPOSITE 1u

/* kvr_pool_desc flag: the pool keeps its keys before RoPE (the raw key
 * projections), and stitching applies RoPE at each token's new position
 * instead of turning stored keys by delta = position - start (TurboRAG blog,
 * "Position ID": keep the un-rotated K, re-apply RoPE at the new position
 * when stitching).  Applies to pool entries; request-local sources keep
 * their keys rotated at local positions 0..len-1. */
#define KVR_POOL_KEYS_UNROTATED 1u

/* kvr_pool_desc flag: RoPE pairs adjacent elements (x_2i, x_2i+1) (the
 * interleaved convention) instead of (x_i, x_i+D/2); pair i still turns at
 * frequency theta^(-2i/D).  Applies to every rotation the library makes for
 * this pool: stored keys, query keys and query heads. */
#define KVR_POOL_ROPE_INTERLEAVED 2u

/* kvr_prefill flag: no decode follows, so the stitched prefix values are not
 * kept.  The prefix keys are stitched (re-rotated) into the cache's K blocks
 * as usual, but the value rows [0, P_b) of the cache's V blocks are left as
 * they are: the attention reads the prefix values straight from the pool
 * (the query rows P_b.. are still appended, and pos_ids / src_map are still
 * written).  Half the stitch's traffic; the output is the same, bit for bit. */
#define KVR_PREFILL_SKIP_PREFIX_CACHE 2u

typedef struct kvr_pool *kvr_pool_t;

/*
 * Resident pool of precomputed chunk caches C_b (CoinRAG blog section 2.1:
 * one offline forward pass per full chunk; TurboRAG blog, Figure 3-b).
 * Entry e, layer l, kv-head h, token t, dim d lives at element
 *   e*stride[0] + l*stride[1] + h*stride[2] + t*stride[3] + d
 * of k (and of v).  Keys are RoPE-rotated at their entry-local positions
 * 0..entry_len-1.  A system-prompt cache C_p is simply another entry.
 */
typedef struct {
    int32_t n_layers;
    int32_t n_q_heads;    /* query heads; a multiple of n_kv_heads (GQA)        */
    int32_t n_kv_heads;
    int32_t head_dim;     /* 64 or 128 (128 for the tensor-core attention path) */
    int32_t dtype;        /* KVR_DTYPE_BF16 or KVR_DTYPE_FP32                   */
    int32_t flags;        /* KVR_POOL_KEYS_UNROTATED | KVR_POOL_ROPE_INTERLEAVED */
    int64_t n_entries;    /* chunks (plus prompt entries) in the pool           */
    int64_t entry_len;    /* tokens per entry                                   */
    const void *k;        /* caller-owned, valid until unregister: device memory,
                           * or pinned host memory the GPU reads through its
                           * unified address (over NVLink-C2C on Grace boards) */
    const void *v;
    int64_t stride[4];    /* elements: entry, layer, head, token; multiples of 8 */
    double rope_theta;    /* RoPE base (e.g. 1e6 for Qwen2)                     */
} kvr_pool_desc;

/* One retrieved span: tokens [start, end) of source src (CoinRAG (b, s, e)). */
typedef struct {
    int32_t src;
    int32_t start;
    int32_t end;
} kvr_span;

/* A request-local source (inline tokens, SemPIC): [n_layers, n_kv_heads, len,
 * head_dim] at the given element strides (layer, head, token), keys rotated
 * at local positions 0..len-1 exactly like a pool entry.  Device pointers. */
typedef struct {
    const void *k;
    const void *v;
    int64_t len;
    int64_t stride[3];
} kvr_local_src;

/*
 * kvr_pool_register -- validate a pool layout and create a handle (host only;
 * no CUDA call).  The first call that enqueues work on the pool binds it to
 * the then-current device and builds the RoPE cos/sin tables for
 * (rope_theta, head_dim) there, synchronously (so make that first call
 * outside any stream capture); the conventions above list every allocation
 * the handle makes afterwards.
 * Errors: KVR_ERR_INVALID_ARG (null, negative or unaligned strides, head_dim
 * odd, n_q_heads % n_kv_heads), KVR_ERR_UNSUPPORTED (dtype, head_dim).
 * On error *out is left NULL.
 */
KVR_API kvr_status kvr_pool_register(const kvr_pool_desc *desc, kvr_pool_t *out);

/* Release a handle and the library's own buffers (synchronizes the device
 * work the handle enqueued).  NULL is a no-op. */
KVR_API kvr_status kvr_pool_unregister(kvr_pool_t pool);

/*
 * kvr_pool_reserve -- bind the pool to the current device (if no call has
 * yet) and allocate, now, every buffer that calls within these limits need:
 * the 8 staging slots sized for the largest tables of a call with up to
 * max_batch requests, max_spans spans and max_locals local sources, and the
 * query scratch for up to max_query_tokens query tokens per call (tensor-core
 * path only).  It synchronizes (allocation and the wait for slots in use).
 * After it, kvr_assemble / kvr_query_attention / kvr_prefill calls within the
 * limits never allocate and never wait on the host, except on a staging slot
 * whose previous call is still queued (see the conventions above).  Calls
 * beyond the limits still work: they grow the buffers as described there.
 * Make it outside any stream capture.  Errors: KVR_ERR_INVALID_ARG (NULL pool,
 * a negative limit, max_query_tokens > 2^31 - 1), KVR_ERR_CUDA.
 */
KVR_API kvr_status kvr_pool_reserve(kvr_pool_t pool, int32_t max_batch, int32_t max_spans,
                                    int32_t max_locals, int64_t max_query_tokens);

/*
 * kvr_assemble -- gather + re-rotate + stitch (CoinRAG blog section 2.3).
 *
 * Request b owns spans[span_offsets[b] .. span_offsets[b+1]) in retrieval
 * order (a system prompt, if any, is its first span).  Its prefix length is
 * P_b = sum of its span lengths; span i lands at stitched row
 * row_i = sum_{j<i} len_j, with position id row_i (reordered) or its source
 * ids (KVR_POSITIONS_COMPOSITE), and its keys are rotated by
 * delta_i = position - start (values are copied bit for bit).
 *
 * Cache layout (device, caller-owned): request b's block holds
 * R_b = cache_offsets[b+1] - cache_offsets[b] rows per (layer, kv-head) and
 * starts at element cache_offsets[b] * n_layers * n_kv_heads * head_dim;
 * inside it, [n_layers][n_kv_heads][R_b][head_dim].  R_b must be >= P_b;
 * leave room for the query tokens if kvr_query_attention follows.
 *
 *   span_offsets  host [batch+1], non-decreasing, span_offsets[0] = 0
 *   spans         host [span_offsets[batch]]
 *   locals        host [n_locals] descriptors of request-local sources
 *                 (device data), or NULL when n_locals = 0
 *   cache_offsets host [batch+1] rows, non-decreasing
 *   pos_ids       device int32 [sum P_b] (request-major, stitched order) or NULL
 *   src_map       device int32 [sum P_b][2] = (src, source token) or NULL
 *   prefix_len    host out int32 [batch] = P_b, or NULL
 *   flags         0 or KVR_POSITIONS_COMPOSITE
 * Errors: KVR_ERR_INVALID_ARG, KVR_ERR_OUT_OF_RANGE (span outside its source,
 * unknown source, P_b > R_b, positions >= 2^24), KVR_ERR_CUDA.
 */
KVR_API kvr_status kvr_assemble(kvr_pool_t pool, int32_t batch, const int32_t *span_offsets,
                        const kvr_span *spans, const kvr_local_src *locals, int32_t n_locals,
                        const int64_t *cache_offsets, void *cache_k, void *cache_v,
                        int32_t *pos_ids, int32_t *src_map, int32_t *prefix_len,
                        uint32_t flags, void *stream);

/*
 * kvr_query_attention -- query prefill over the stitched prefix
 * (CoinRAG blog section 2.3, KV_M(q; C_ctx); TurboRAG blog "Attention Mask").
 *
 * Query token t (0-based) of request b sits at position P_b + t.  The call
 * rotates its query heads and its key at that position, appends its key and
 * value at cache row P_b + t of every (layer, kv-head) block, and computes
 *   O[l, q_offsets[b]+t, h] = sum_j softmax_j(scale * <q, k_j>) v_j
 * over the P_b prefix rows and query rows 0..t, kv-head = h / (H_q / H_kv).
 *
 *   cache_offsets host [batch+1] as in kvr_assemble; need P_b + Lq_b <= R_b
 *   prefix_len    host [batch] (P_b, e.g. from kvr_assemble)
 *   q_offsets     host [batch+1]: request b's query tokens are rows
 *                 q_offsets[b] .. q_offsets[b+1]-1 of the token axis
 *   q             [n_layers][T][n_q_heads][head_dim], T = q_offsets[batch],
 *                 not rotated
 *   kq, vq        [n_layers][T][n_kv_heads][head_dim], not rotated
 *   out           [n_layers][T][n_q_heads][head_dim], pool dtype
 *                 q, kq, vq and out are device memory or pinned host memory
 *                 (read, or written, once by the library's kernels through the
 *                 unified address, over the CPU-GPU link): a host `out` spares
 *                 the caller a copy back after the call.
 *   softmax_scale 0 means 1/sqrt(head_dim)
 *
 * A decode step -- every request with one query token, or none (CoinRAG
 * blog section 2.3: decoding continues normally on top of the stitched
 * cache) -- on a bf16 pool with head_dim 128 and at most 16 query heads per
 * kv head runs as a single kernel that rotates, appends and attends, each
 * (request, layer, kv-head) block streamed once by one CTA.  Other calls on the
 * tensor-core path (bf16, head_dim 128) also write zeros into the V rows
 * between a block's last query row and the end of its last 128-row key tile
 * (rows of the block, never past R_b); a decode step leaves those rows as
 * they are.
 * Errors: KVR_ERR_INVALID_ARG, KVR_ERR_OUT_OF_RANGE, KVR_ERR_UNSUPPORTED,
 * KVR_ERR_CUDA.  A kernel whose bounded wait ran out records
 * KVR_ERR_TIMEOUT, reported by kvr_check.
 */
KVR_API kvr_status kvr_query_attention(kvr_pool_t pool, int32_t batch, const int64_t *cache_offsets,
                               const int32_t *prefix_len, const int32_t *q_offsets,
                               const void *q, const void *kq, const void *vq,
                               void *cache_k, void *cache_v, void *out,
                               float softmax_scale, void *stream);

/*
 * kvr_prefill -- the whole precomputed-KV prefill in one call: kvr_assemble
 * followed by kvr_query_attention with P_b taken from the stitch
 * (CoinRAG blog section 2.3: KV_CoinRAG = C_ctx stitched from stored chunks,
 * then KV_M(q; C_ctx) computed online).  Arguments mean what they mean in
 * those two calls (cache_k / cache_v and cache_offsets are shared; the
 * blocks must hold P_b + Lq_b rows); prefix_len is an optional host output.
 * Results are identical, bit for bit, to the two calls in a row (a pool in
 * pinned host memory: see below).
 *
 * The difference is scheduling: every check of both halves runs before
 * anything is enqueued, the table uploads go first, and the kernels follow
 * one another on the stream with programmatic dependent launch, so the
 * query-side kernel (rotation and append of the query tokens, which touches
 * no prefix row) runs alongside the stitch, and the attention kernel's setup
 * overlaps it.  The timing hook (kvr_set_timing_events) serializes them.
 *
 * A pool in pinned host memory (on the tensor-core path, more than one query
 * token in some request, n_layers divisible by 2..8): the stitch, bound by
 * the CPU-GPU link, runs by groups of layers, last group first, on 64 CTAs of
 * an internal stream that starts after the work already on `stream`; the
 * attention of each group runs on `stream`, on the other SMs, beside the
 * stitch of the next group.  Before that stitch, zeros are written into the
 * first min(P_b, 128) V rows of the first block of requests 1..batch-1 (rows
 * the stitch then overwrites), so that the attention of the previous request's
 * last block, whose last key tile reaches into them with weight 0, reads
 * finite values.  When the call returns, all of its work is ordered before
 * later work on `stream`.  The output is that of the two calls up to rounding
 * order (the attention's last round of units splits differently on fewer SMs).
 *
 * flags: KVR_POSITIONS_COMPOSITE as in kvr_assemble; KVR_PREFILL_SKIP_PREFIX_CACHE
 * (above) needs a bf16 pool in device memory with head_dim 128 and the
 * tensor-core attention (any strides, request-local sources allowed);
 * otherwise the call returns KVR_ERR_UNSUPPORTED before any work.
 * Errors: those of the two calls; nothing is enqueued when a check fails.
 */
KVR_API kvr_status kvr_prefill(kvr_pool_t pool, int32_t batch, const int32_t *span_offsets,
                               const kvr_span *spans, const kvr_local_src *locals, int32_t n_locals,
                               const int64_t *cache_offsets, void *cache_k, void *cache_v,
                               int32_t *pos_ids, int32_t *src_map, int32_t *prefix_len,
                               uint32_t flags, const int32_t *q_offsets, const void *q,
                               const void *kq, const void *vq, void *out, float softmax_scale,
                               void *stream);

/* Attention kernels a pool can select (kvr_attention_path). */
enum { KVR_PATH_UNBOUND = -1, KVR_PATH_CUDA_CORES = 0, KVR_PATH_TCGEN05 = 1 };

/* Which attention kernel kvr_query_attention runs for this pool: the
 * tcgen05 tensor-core kernel (bf16, head_dim 128, sm_103) or the CUDA-core
 * kernel (fp32 or head_dim 64).  KVR_PATH_UNBOUND until the pool's first
 * call has bound it to a device; -2 for a NULL pool. */
KVR_API int32_t kvr_attention_path(kvr_pool_t pool);

/* Timing hook.  With events non-NULL, later calls on this pool record, on the
 * caller's stream, events[0] / events[1] right before / after the assemble
 * kernel, events[2] / events[3] around the query-append kernel (nothing
 * between them for a decode step, whose one kernel appends) and
 * events[4] / events[5] around the attention kernel.  The handles are
 * cudaEvent_t created by the caller (timing enabled); the array is copied.
 * NULL turns the hook off. */
KVR_API kvr_status kvr_set_timing_events(kvr_pool_t pool, void *const *events);

/*
 * kvr_selftest_wait -- exercise the bounded-wait error path.
 *
 * Every wait inside the library's kernels gives up after a time limit (2 s),
 * records KVR_ERR_TIMEOUT in the pool's error word and lets the kernel end,
 * so that a lost signal is reported by kvr_check rather than hanging the GPU.
 * This call enqueues, on `stream`, a one-CTA kernel that waits the same way on
 * a barrier that nothing completes, for limit_ns nanoseconds (1 us .. 2 s;
 * other values are clamped), and records KVR_ERR_TIMEOUT like the hot path.
 * The next kvr_check on the pool returns KVR_ERR_TIMEOUT and clears the word;
 * the pool and the CUDA context stay usable.  For tests of the error path.
 * Errors: KVR_ERR_INVALID_ARG (NULL pool), KVR_ERR_CUDA.
 */
KVR_API kvr_status kvr_selftest_wait(kvr_pool_t pool, uint64_t limit_ns, void *stream);

/*
 * kvr_assemble_noalloc -- kvr_assemble for callers that cannot allocate.
 *
 * The pages have no counterpart: this is a deployment variant.  Some callers
 * cannot call cudaMalloc (or any allocator) where they stitch a prefix -- an
 * engine whose caching allocator already holds the free device memory, a
 * latency-critical request loop that forbids allocations, a plug-in that may
 * only use its host program's allocator.  This call allocates nothing: it
 * takes the pool descriptor itself (no handle), builds its span table in a
 * fixed host array, and keeps its device scratch (span table, local-source
 * table, RoPE tables: 4.2 MiB) in one file-scope __device__ array that every
 * GPU loading the library holds until the process exits.  Same arguments,
 * layout and results as kvr_assemble otherwise (same kernel).
 *
 * Limits: at most 4096 non-empty spans and 256 local sources per call, and
 * head_dim <= 128; beyond them the call returns KVR_ERR_INVALID_ARG before
 * any GPU work, with the reason in kvr_last_error().  The first call on a
 * device looks up the scratch address (cudaGetSymbolAddress, a synchronous
 * runtime call) with that device current.  A call with at
 * most 64 spans and 64 local sources passes its tables inside the kernel's
 * parameters; a larger one copies them from the library's fixed host tables
 * into the scratch on the caller's stream.  All calls share the scratch and
 * the host tables: calls from several host threads, or calls that overlap on
 * the GPU (on different streams), race; the RoPE tables are rebuilt in the
 * scratch, on the caller's stream, whenever (rope_theta, head_dim) differs
 * from the previous call on that device.  Nothing in the scratch has to start
 * at zero.
 */
KVR_API kvr_status kvr_assemble_noalloc(const kvr_pool_desc *desc, int32_t batch,
                                        const int32_t *span_offsets, const kvr_span *spans,
                                        const kvr_local_src *locals, int32_t n_locals,
                                        const int64_t *cache_offsets, void *cache_k, void *cache_v,
                                        int32_t *pos_ids, int32_t *src_map, int32_t *prefix_len,
                                        uint32_t flags, void *stream);

/* Synchronize `stream` and return (then clear) the first error a kernel of
 * this pool recorded: KVR_OK, KVR_ERR_TIMEOUT (a bounded wait ran out),
 * KVR_ERR_DEVICE_CHECK or KVR_ERR_CUDA.  KVR_ERR_DEVICE_CHECK: the
 * tensor-core prefill or decode attention found a query row whose softmax
 * denominator was not a finite positive number -- a NaN or an infinity in
 * its query heads or in a key it attends to (inputs the host cannot see
 * without reading device memory); the row's output is written as computed
 * (not finite) and the rest of the call is unaffected. */
KVR_API kvr_status kvr_check(kvr_pool_t pool, void *stream);

/* Static string naming a status. */
KVR_API const char *kvr_status_string(kvr_status s);

/* One-line description of the last error raised on this host thread. */
KVR_API const char *kvr_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVR_H */
