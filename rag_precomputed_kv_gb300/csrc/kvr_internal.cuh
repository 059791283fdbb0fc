// kvr_internal.cuh -- types shared by the libkvr translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvr.h"

#ifdef __CUDACC__
#include <cuda_bf16.h>
#endif

namespace kvr {

// RoPE tables: angle(n, i) = n * theta^(-2i/D) for n in [0, 2^24) is split as
// n = hi * 4096 + lo; the table holds (cos, sin) of hi * 4096 * w_i
// (rows 0..4095) and of lo * w_i (rows 4096..8191), each computed in double
// precision and rounded to float.  One complex product in float recombines
// them: the angle-addition identity, with error of a few float ulps for
// every position (a float product n * w_i would be off by up to ~2e-3 rad at
// n ~ 3e4).
constexpr int kRopeSplit = 4096;
constexpr int kMaxPosition = kRopeSplit * kRopeSplit;  // 2^24

#ifdef __CUDACC__
// Programmatic dependent launch: let the next kernel of the stream (launched
// with programmatic serialization) start its grid now / wait until the
// previous kernel of the stream has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// (cos, sin) of pos * w_i for |pos| < 2^24 from the two table halves (angle
// addition, one complex product in float); a negative pos is the conjugate.
// Below 2^12 the high half's entry is row 0, exactly (1, 0): the product is
// the low entry itself, bit for bit, and only that one is read.
__device__ __forceinline__ float2 rope_cs(const float2 *__restrict__ tab, int half, int pos, int i)
{
    const int a = pos < 0 ? -pos : pos;
    const float2 l = __ldg(tab + (kRopeSplit + (a & (kRopeSplit - 1))) * half + i);
    float c = l.x, s = l.y;
    if (a >= kRopeSplit) {
        const float2 h = __ldg(tab + (a >> 12) * half + i);
        c = fmaf(h.x, l.x, -h.y * l.y);
        s = fmaf(h.y, l.x, h.x * l.y);
    }
    return make_float2(c, pos < 0 ? -s : s);
}

// RoPE rotation of 8 bf16 pairs: lo holds elements [8j, 8j+8) of a row, hi
// their partners [D/2 + 8j, ...); (c, s) of each pair.  The stitch kernel's
// key re-rotation for bf16 caches.
// Per pair: x' = fma(x, c, -(y s)), y' = fma(x, s, y c), rounded once to bf16;
// computed two lanes at a time with the packed fp32 instructions (each lane
// is the IEEE operation of the scalar form).
__device__ __forceinline__ void rotate_bf16x8(uint4 &lo, uint4 &hi, const float *c, const float *s)
{
    uint32_t *pl = reinterpret_cast<uint32_t *>(&lo);
    uint32_t *ph = reinterpret_cast<uint32_t *>(&hi);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        // bf16 pair -> two fp32 lanes (a bf16 is the high half of its fp32)
        const uint64_t x = ((uint64_t)(pl[w] & 0xffff0000u) << 32) | (uint64_t)(pl[w] << 16);
        const uint64_t y = ((uint64_t)(ph[w] & 0xffff0000u) << 32) | (uint64_t)(ph[w] << 16);
        const uint64_t cc = ((uint64_t)__float_as_uint(c[2 * w + 1]) << 32) | __float_as_uint(c[2 * w]);
        const uint64_t ns = ((uint64_t)__float_as_uint(-s[2 * w + 1]) << 32) | __float_as_uint(-s[2 * w]);
        const uint64_t ss = ((uint64_t)__float_as_uint(s[2 * w + 1]) << 32) | __float_as_uint(s[2 * w]);
        uint64_t ys, yc, xo, yo;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(ys) : "l"(y), "l"(ns));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(yc) : "l"(y), "l"(cc));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(xo) : "l"(x), "l"(cc), "l"(ys));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(yo) : "l"(x), "l"(ss), "l"(yc));
        __nv_bfloat162 xb = __floats2bfloat162_rn(__uint_as_float((uint32_t)xo), __uint_as_float((uint32_t)(xo >> 32)));
        __nv_bfloat162 yb = __floats2bfloat162_rn(__uint_as_float((uint32_t)yo), __uint_as_float((uint32_t)(yo >> 32)));
        pl[w] = *reinterpret_cast<uint32_t *>(&xb);
        ph[w] = *reinterpret_cast<uint32_t *>(&yb);
    }
}

// The same rotation for the interleaved pairing: every bf16 word of lo and
// hi is a pair (x_2i, x_2i+1); c[w], s[w] belong to lo's word w and c[4 + w],
// s[4 + w] to hi's.
__device__ __forceinline__ void rotate_bf16x8_il(uint4 &lo, uint4 &hi, const float *c, const float *s)
{
    uint32_t *pw[2] = {reinterpret_cast<uint32_t *>(&lo), reinterpret_cast<uint32_t *>(&hi)};
#pragma unroll
    for (int v = 0; v < 2; ++v) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float2 xy = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&pw[v][w]));
            const float cc = c[4 * v + w], ss = s[4 * v + w];
            __nv_bfloat162 o = __floats2bfloat162_rn(fmaf(xy.x, cc, -xy.y * ss), fmaf(xy.x, ss, xy.y * cc));
            pw[v][w] = *reinterpret_cast<uint32_t *>(&o);
        }
    }
}

// Pair index of the e-th (cos, sin) of a thread that owns 16-byte chunk j of
// both row halves (E elements per chunk, head dim D): half-split pairs are
// elements (jE + e, D/2 + jE + e); interleaved pairs are whole inside a
// chunk, E/2 of them in the chunk of each half.
__device__ __forceinline__ int rope_pair(bool interleaved, int D, int E, int j, int e)
{
    if (!interleaved)
        return j * E + e;
    return e < E / 2 ? (E / 2) * j + e : D / 4 + (E / 2) * j + (e - E / 2);
}
#endif

// Device copy of one span (48 bytes).
struct alignas(16) DevSpan {
    int64_t dst_row0;  // first row of the request's cache block, in head_dim rows
    int64_t flat0;     // index of the span's first token in the flat pos / src maps
    int32_t src;       // pool entry, or KVR_SRC_LOCAL | local index
    int32_t start;     // first source token
    int32_t len;       // tokens
    int32_t row;       // first stitched row inside the request's block
    int32_t delta;     // rotation applied to the keys (positions)
    int32_t pos0;      // position id of the first token
    int32_t cap;       // rows per (layer, kv-head) block of the request
    int32_t dstep;     // 0: source keys carry their source positions (rotate all
                       //    tokens by delta); 1: source keys are un-rotated
                       //    (token t is rotated by delta + t)
};

// Device copy of one request-local source.
struct alignas(16) DevLocal {
    const void *k;
    const void *v;
    int64_t s_layer, s_head, s_tok;
    int64_t len;
};

// Per-request data for the attention kernels (48 bytes).  On the tensor-core
// path the table is in schedule order (longest prefix first) and unit0 is the
// request's first work unit; elsewhere it is in request order.
struct alignas(16) DevReq {
    int64_t cache_row0;  // cache_offsets[b] * L * H_kv
    int32_t cap;         // R_b
    int32_t prefix;      // P_b
    int32_t q_off;       // first query token (token axis of q / out)
    int32_t q_len;       // Lq_b
    int32_t unit0;       // first (layer, kv-head, 256-row block) unit (tensor-core path)
    int32_t span0;       // first non-empty span of this request (values-gathering attention)
    int32_t span_end;    // one past its last
    int32_t flags;       // kReqValuesTma (values-gathering attention)
    int32_t pad_[2];
};
static_assert(sizeof(DevReq) == 48, "request table layout");
// DevReq::flags: the values-gathering attention loads this request's prefix
// value tiles through TMA box loads (its spans are long and all from a
// contiguous pool) rather than with the gather warps' copies
constexpr int32_t kReqValuesTma = 1;

// Device error word codes (first error wins).  kDevBadInput: an attention
// row's softmax denominator came out non-finite or zero (a NaN or infinity in
// the query heads or the keys it saw); the row's output is written as computed.
enum : int { kDevOk = 0, kDevTimeout = 1, kDevBadInput = 2 };

// Records `msg` as this host thread's last error (kvr_last_error) and
// returns `st`; allocates nothing.
kvr_status record_error(kvr_status st, const char *msg);

struct AssembleArgs {
    const DevSpan *spans;
    const DevLocal *locals;
    const float2 *rope;
    const void *pool_k;
    const void *pool_v;
    int64_t ps_entry, ps_layer, ps_head, ps_tok;
    void *cache_k;
    void *cache_v;
    int32_t *pos_ids;
    int32_t *src_map;
    int32_t n_layers, n_heads;  // kv heads
    int32_t upc;                // (layer, head) units per CTA
    int32_t interleaved;        // RoPE pairs (x_2i, x_2i+1)
    // a slice of the (layer, kv-head) units, [lh_begin, lh_begin + lh_count)
    // (lh_count 0: all of them); the position ids and source map are written
    // with the slice that starts at unit 0
    int32_t lh_begin, lh_count;
    // > 0: at most this many CTAs, each looping over (span, unit group)
    // pieces (the stitch then leaves the other SMs to a concurrent kernel)
    int32_t max_ctas;
    int32_t n_spans;            // set by launch_assemble
    int32_t keys_only;          // stitch K (and the maps) only; V is gathered by the attention
};

// Span / local-source tables passed inside the kernel parameters (no upload)
// when a call has at most kInlineEntries of each.
constexpr int kInlineEntries = 64;
struct AssembleTables {
    DevSpan spans[kInlineEntries];
    DevLocal locals[kInlineEntries];
};

// Request table passed inside the attention kernels' parameters when
// batch <= kInlineEntries (AttnArgs::reqs is then NULL).
struct ReqTable {
    DevReq reqs[kInlineEntries];
};

struct AttnArgs {
    const DevReq *reqs;
    int32_t n_reqs;
    const float2 *rope;
    const void *q;              // [L][T][Hq][D]
    const void *cache_k;
    const void *cache_v;
    void *out;                  // [L][T][Hq][D]
    int32_t n_layers, n_q_heads, n_kv_heads;
    int32_t total_q;            // T
    float scale_log2;           // softmax scale * log2(e)
    int *err;
    // tensor-core kernel: units n_full.. (the last wave's, when two halves of
    // each fit one wave) run as two halves of their key range on the two CTAs
    // of a cluster, which merge them; n_full < units requires a launch in
    // two-CTA clusters
    int32_t n_full;
    int32_t interleaved;        // RoPE pairs (x_2i, x_2i+1)
    // tensor-core kernel: a slice of each request's (layer, kv-head) units,
    // [lh_base, lh_base + lh_count) (lh_count 0: all); the request table's
    // unit0 counts lh_count units per 256-row block
    int32_t lh_base, lh_count;
    // tensor-core kernel: the output goes out through TMA tensor stores (the
    // tmap_out parameter), a warp's 32 rows = 32 / G whole tokens of the G
    // query heads of one kv head; set when G is a power of two and `out` is
    // device memory
    int32_t out_tma;
};

struct QueryPrologueArgs {
    const DevReq *reqs;         // NULL: the ReqTable parameter holds the requests
    const float2 *rope;
    const void *q;              // [L][T][Hq][D], not rotated
    const void *kq;             // [L][T][Hkv][D], not rotated
    const void *vq;
    void *cache_k;
    void *cache_v;
    void *q_rot;                // out: [L][Hkv][T][G][D], rotated at P_b + t
    int32_t n_layers, n_q_heads, n_kv_heads;
    int32_t total_q;            // T
    int32_t max_q_len;          // longest query of the batch
    int32_t n_reqs;
    int32_t interleaved;        // RoPE pairs (x_2i, x_2i+1)
};

// ---- launchers (each returns the cudaGetLastError of its launch) ----
cudaError_t launch_rope_tables(float2 *tab, int head_dim, double theta, cudaStream_t s);
// `inl` (optional) carries the span and local tables; a.spans / a.locals are
// then ignored.
cudaError_t launch_assemble(const AssembleArgs &a, int dtype, int head_dim, int n_spans,
                            cudaStream_t s, const AssembleTables *inl = nullptr);
cudaError_t launch_attention_simt(const AttnArgs &a, const ReqTable &rt, int dtype, int head_dim,
                                  cudaStream_t s);

// Tensor-core attention (bf16, head_dim 128).  `tmaps` points to two
// CUtensorMap objects (K then V) describing the cache as a 2-D
// [rows, head_dim] bf16 tensor.
// The tensor-core attention's values-gathering variant (kvr_prefill): V tiles
// of prefix rows are gathered from the pool, seen as a 2-D
// [entries * L * H_kv * entry_len, D] tensor, through the batch's span table.
struct SpanTable {
    DevSpan spans[kInlineEntries];
};
struct GatherArgs {
    const DevSpan *spans;       // the batch's spans in global memory, or NULL: the SpanTable parameter
    const DevLocal *locals;     // the batch's request-local sources in global memory; NULL in calls with none
    int32_t n_spans;            // non-empty spans of the batch (request b's start at DevReq::span0)
    int32_t entry_len;          // pool tokens per entry
    const void *pool_v;         // the pool's values (bf16)
    int64_t ps_entry, ps_layer, ps_head, ps_tok;   // their strides, in elements
    int32_t tma_pool;           // the TMA maps of the pool's values are set (a contiguous pool)
};

struct TcAttnArgs {
    AttnArgs base;
    const ReqTable *rt;         // used when base.reqs is NULL
    const void *tmap_q;         // host CUtensorMaps, passed by value to the kernel:
    const void *tmap_k;         //   rotated packed Q [L*Hkv*T*G, D], cache K and V [rows, D]
    const void *tmap_v;
    int32_t n_m_blocks;         // total 256-row query blocks over all requests
    int32_t n_sms;              // persistent grid size bound
    bool gather_v;              // V tiles of prefix rows from the pool (g, st), K from the cache
    const void *tmap_pv;        // the pool's values as [rows, D] with a one-row box (gather4)
    const void *tmap_bv;        // the same with a 32-row box (runs of consecutive pool rows)
    GatherArgs g;
    const SpanTable *st;
    const void *tmap_out;       // out as [L*T][H_q][D] with a (64, G, 32 / G) box (base.out_tma)
};
// `pdl`: the kernel before it on the stream is the assemble kernel of the
// same prefill (which it may overlap: it reads only the caller's inputs and
// writes only query-side rows).
cudaError_t launch_query_prologue(const QueryPrologueArgs &a, const ReqTable &rt, int n_sms, bool pdl,
                                  cudaStream_t s);
// `pdl`: the kernel before it on the stream is the query prologue of the
// same call; the setup (barriers, TMEM) overlaps that kernel's tail.
// Launched in two-CTA clusters when a.base.n_full < units.
cudaError_t launch_attention_tc(const TcAttnArgs &a, bool pdl, cudaStream_t s);
bool attention_tc_supported(int dtype, int head_dim);
// A decode step (every request has one query token, or none): one CTA per
// (request, layer, kv-head) rotates the step's key and query heads, appends
// the key and value at row P_b and streams the cache block (the cache tensor
// maps of the prefill attention).  Replaces the query prologue for the step.
struct DecodeIO {
    const void *kq;             // [L][T][Hkv][D], not rotated
    const void *vq;
    void *cache_k;
    void *cache_v;
    int32_t interleaved;        // RoPE pairs (x_2i, x_2i+1)
};
bool decode_supported(int dtype, int head_dim, int group);
// One CTA whose only wait (bounded by limit_ns) is on a barrier nothing
// completes: records kDevTimeout in *err when the limit runs out.
cudaError_t launch_wait_selftest(int *err, unsigned long long limit_ns, cudaStream_t s);
// `pdl`: programmatic launch (the kernel sets up while the kernel before it
// finishes, and reads nothing before that kernel is done); a decode step lets
// the next one launch that way
cudaError_t launch_decode_attention(const AttnArgs &a, const ReqTable &rt, const void *tmap_k, const void *tmap_v,
                                    const DecodeIO &io, bool pdl, cudaStream_t s);
// Whether `n_sms` CTAs of the attention kernel (either variant) can be
// resident at once as two-CTA clusters.
bool attention_tc_pairs_fit(int n_sms);

}  // namespace kvr
