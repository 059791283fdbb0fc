// kvr_api.cu -- the C ABI: validation, span tables, staging and launches.
//
// Host work per call is bookkeeping only: validate every span against its
// source and every request against its cache block, lay the span / request
// tables out (the stitched row of span i is the prefix sum of the lengths
// before it -- CoinRAG blog section 2.3), copy them to the device with one
// asynchronous H2D copy from a pinned staging slot, and launch the kernels on
// the caller's stream.  Allocations and host waits happen only where the
// header lists them: binding the pool to a device, growing a staging slot or
// the query scratch past its size (kvr_pool_reserve sizes both up front), and
// reusing a staging slot that an earlier call's work still holds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "kvr_internal.cuh"

using namespace kvr;

namespace {

// One-line reason of the last failure on this thread (a fixed buffer: the
// error paths allocate nothing, the allocation-free entry point included).
thread_local char g_last_error[512];

kvr_status fail(kvr_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

kvr_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(KVR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

kvr_status kvr::record_error(kvr_status st, const char *msg)
{
    snprintf(g_last_error, sizeof g_last_error, "%s", msg ? msg : "");
    return st;
}

namespace {

// Staging slots per pool: a call whose tables do not fit its kernels'
// parameters takes the next slot in turn, and waits on the host only if that
// slot's previous call has not yet run (kSlots such calls queued ahead).
constexpr int kSlots = 8;

// Host-pool prefill pipeline: layer groups, and the CTAs its stitch keeps
// (the attention runs on the other SMs meanwhile).
constexpr int kMaxLayerParts = 8;
constexpr int kHostStitchCtas = 64;

// Scoped NVTX range (a profiler's timeline shows which library call and which
// kernel each stretch of host time enqueued; nothing without a profiler).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

struct Slot {
    void *host = nullptr;   // pinned: tables built by the host
    void *dev = nullptr;    // device: the uploaded tables, then per-call device scratch
    size_t host_cap = 0, dev_cap = 0;
    cudaEvent_t done = nullptr;
    bool used = false;
};

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev)
            cudaSetDevice(dev);
        else
            prev = -1;
    }
    ~DeviceGuard()
    {
        if (prev >= 0)
            cudaSetDevice(prev);
    }
};

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

struct kvr_pool {
    kvr_pool_desc d{};
    int device = 0;
    int cc = 0;               // compute capability, major * 10 + minor
    float2 *rope = nullptr;   // RoPE tables
    int *err = nullptr;       // device error word
    Slot slots[kSlots];
    int next = 0;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    bool ready = false;       // device-side setup done
    int n_sms = 1;
    // rotated, packed query heads for the tensor-core attention (grown on
    // demand); q_rot_done orders its reuse after the last call's attention
    void *q_rot = nullptr;
    size_t q_rot_cap = 0;
    cudaEvent_t q_rot_done = nullptr;
    bool q_rot_used = false;
    // a pool in pinned host memory: kvr_prefill stitches it by layer groups on
    // a second stream, each group's attention overlapping the next group's
    // stitch (which reads over the CPU-GPU link)
    bool host_pool = false;
    cudaStream_t side = nullptr;
    cudaEvent_t side_start = nullptr;
    cudaEvent_t part_ev[kMaxLayerParts] = {};
    cudaEvent_t timing[6] = {};  // optional kernel timing events (caller-owned)
    bool timed = false;

    void mark(int i, cudaStream_t s) const
    {
        if (timed && timing[i])
            cudaEventRecord(timing[i], s);
    }

    int elt() const { return d.dtype == KVR_DTYPE_BF16 ? 2 : 4; }
    int vec_elems() const { return 16 / elt(); }

    // A staging slot with at least `host_bytes` of pinned and `dev_bytes` of
    // device memory; waits until the slot's last upload and the kernels that
    // read it are done (only when kSlots later calls have been enqueued since
    // and that work has not run yet).  A slot smaller than asked is freed and
    // allocated again (cudaFreeHost / cudaFree synchronize the device).
    kvr_status acquire(size_t host_bytes, size_t dev_bytes, Slot **out)
    {
        Slot &s = slots[next];
        next = (next + 1) % kSlots;
        cudaError_t e;
        if (s.used && cudaEventQuery(s.done) != cudaSuccess) {
            NvtxRange r("kvr.staging_slot_wait");
            if ((e = cudaEventSynchronize(s.done)) != cudaSuccess)
                return cuda_fail(e, "staging slot wait");
        }
        kvr_status st = grow(s, host_bytes, dev_bytes);
        if (st == KVR_OK)
            *out = &s;
        return st;
    }

    // Slot `s` (idle) with at least the given capacities, and its event.
    static kvr_status grow(Slot &s, size_t host_bytes, size_t dev_bytes)
    {
        cudaError_t e;
        if (s.host_cap < host_bytes) {
            NvtxRange r("kvr.staging_alloc");
            const size_t cap = std::max<size_t>({host_bytes, 2 * s.host_cap, 65536});
            if (s.host)
                cudaFreeHost(s.host);
            s.host = nullptr;
            s.host_cap = 0;
            if ((e = cudaMallocHost(&s.host, cap)) != cudaSuccess)
                return cuda_fail(e, "staging host buffer");
            s.host_cap = cap;
        }
        if (s.dev_cap < dev_bytes) {
            NvtxRange r("kvr.staging_alloc");
            const size_t cap = std::max<size_t>({dev_bytes, 2 * s.dev_cap, 65536});
            if (s.dev)
                cudaFree(s.dev);
            s.dev = nullptr;
            s.dev_cap = 0;
            if ((e = cudaMalloc(&s.dev, cap)) != cudaSuccess)
                return cuda_fail(e, "staging device buffer");
            s.dev_cap = cap;
        }
        if (!s.done && (e = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "staging event");
        return KVR_OK;
    }

    // The rotated-query scratch with at least `bytes`: a smaller one is freed
    // (after the last call's attention is done with it) and allocated again.
    kvr_status grow_query_scratch(size_t bytes)
    {
        cudaError_t e;
        if (q_rot_cap < bytes) {
            NvtxRange r("kvr.query_scratch_alloc");
            if (q_rot_used && (e = cudaEventSynchronize(q_rot_done)) != cudaSuccess)
                return cuda_fail(e, "query scratch wait");
            if (q_rot)
                cudaFree(q_rot);
            q_rot = nullptr;
            q_rot_cap = 0;
            q_rot_used = false;
            if ((e = cudaMalloc(&q_rot, bytes)) != cudaSuccess)
                return cuda_fail(e, "query scratch");
            q_rot_cap = bytes;
        }
        if (!q_rot_done && (e = cudaEventCreateWithFlags(&q_rot_done, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "query scratch event");
        return KVR_OK;
    }
};

// ---------------------------------------------------------------------------
// registration
// ---------------------------------------------------------------------------
extern "C" kvr_status kvr_pool_register(const kvr_pool_desc *desc, kvr_pool_t *out)
{
    if (!out)
        return fail(KVR_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!desc)
        return fail(KVR_ERR_INVALID_ARG, "desc is NULL");
    const kvr_pool_desc &d = *desc;
    if (d.dtype != KVR_DTYPE_BF16 && d.dtype != KVR_DTYPE_FP32)
        return fail(KVR_ERR_UNSUPPORTED, "dtype %d", d.dtype);
    if (d.head_dim != 64 && d.head_dim != 128)
        return fail(KVR_ERR_UNSUPPORTED, "head_dim %d (64 or 128)", d.head_dim);
    if (d.n_layers < 1 || d.n_kv_heads < 1 || d.n_q_heads < 1 || d.n_q_heads % d.n_kv_heads)
        return fail(KVR_ERR_INVALID_ARG, "layers %d, q heads %d, kv heads %d", d.n_layers,
                    d.n_q_heads, d.n_kv_heads);
    if (d.n_entries < 1 || d.entry_len < 1 || d.entry_len > kMaxPosition)
        return fail(KVR_ERR_INVALID_ARG, "n_entries %lld, entry_len %lld",
                    (long long)d.n_entries, (long long)d.entry_len);
    if (d.flags & ~(KVR_POOL_KEYS_UNROTATED | KVR_POOL_ROPE_INTERLEAVED))
        return fail(KVR_ERR_INVALID_ARG, "unknown pool flags 0x%x", (unsigned)d.flags);
    if (!d.k || !d.v)
        return fail(KVR_ERR_INVALID_ARG, "pool k / v is NULL");
    if (!aligned16(d.k) || !aligned16(d.v))
        return fail(KVR_ERR_INVALID_ARG, "pool k / v not 16-byte aligned");
    if (!(d.rope_theta > 1.0) || !std::isfinite(d.rope_theta))
        return fail(KVR_ERR_INVALID_ARG, "rope_theta %g", d.rope_theta);
    const int vec = 16 / (d.dtype == KVR_DTYPE_BF16 ? 2 : 4);
    for (int i = 0; i < 4; ++i)
        if (d.stride[i] < 0 || d.stride[i] % vec)
            return fail(KVR_ERR_INVALID_ARG, "stride[%d] = %lld must be >= 0 and a multiple of %d",
                        i, (long long)d.stride[i], vec);

    kvr_pool *p = new kvr_pool();
    p->d = d;
    *out = p;
    return KVR_OK;
}

// Device-side setup, done by the first call that launches work: the RoPE
// tables for (rope_theta, head_dim), the error word, the tensor-map encoder.
static kvr_status ensure_device(kvr_pool *p)
{
    if (p->ready)
        return KVR_OK;
    cudaError_t e;
    if ((e = cudaGetDevice(&p->device)) != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int maj = 0, min = 0;
    cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, p->device);
    cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, p->device);
    p->cc = maj * 10 + min;
    cudaDeviceGetAttribute(&p->n_sms, cudaDevAttrMultiProcessorCount, p->device);
    const size_t tab = sizeof(float2) * 2 * kRopeSplit * (p->d.head_dim / 2);
    if ((e = cudaMalloc(&p->rope, tab)) != cudaSuccess ||
        (e = cudaMalloc(&p->err, sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(p->err, 0, sizeof(int))) != cudaSuccess ||
        (e = launch_rope_tables(p->rope, p->d.head_dim, p->d.rope_theta, 0)) != cudaSuccess ||
        (e = cudaStreamSynchronize(0)) != cudaSuccess)
        return cuda_fail(e, "pool device setup");
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        p->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, p->d.k) == cudaSuccess)
        p->host_pool = pa.type == cudaMemoryTypeHost;
    else
        cudaGetLastError();
    p->ready = true;
    return KVR_OK;
}

extern "C" kvr_status kvr_pool_unregister(kvr_pool_t p)
{
    if (!p)
        return KVR_OK;
    if (!p->ready) {  // device setup never completed: free what it got
        if (p->rope)
            cudaFree(p->rope);
        if (p->err)
            cudaFree(p->err);
        delete p;
        return KVR_OK;
    }
    DeviceGuard g(p->device);
    for (Slot &s : p->slots) {
        if (s.done) {
            cudaEventSynchronize(s.done);
            cudaEventDestroy(s.done);
        }
        if (s.host)
            cudaFreeHost(s.host);
        if (s.dev)
            cudaFree(s.dev);
    }
    if (p->q_rot_done) {
        cudaEventSynchronize(p->q_rot_done);
        cudaEventDestroy(p->q_rot_done);
    }
    if (p->q_rot)
        cudaFree(p->q_rot);
    if (p->side) {
        cudaStreamSynchronize(p->side);
        cudaStreamDestroy(p->side);
    }
    if (p->side_start)
        cudaEventDestroy(p->side_start);
    for (cudaEvent_t e : p->part_ev)
        if (e)
            cudaEventDestroy(e);
    if (p->rope)
        cudaFree(p->rope);
    if (p->err)
        cudaFree(p->err);
    delete p;
    return KVR_OK;
}

// The tcgen05 kernel runs for bf16 pools with head_dim 128 on sm_103.
static bool use_tensor_cores(const kvr_pool &p);

extern "C" kvr_status kvr_pool_reserve(kvr_pool_t p, int32_t max_batch, int32_t max_spans, int32_t max_locals,
                                       int64_t max_query_tokens)
{
    if (!p)
        return fail(KVR_ERR_INVALID_ARG, "pool is NULL");
    if (max_batch < 0 || max_spans < 0 || max_locals < 0 || max_query_tokens < 0 ||
        max_query_tokens > INT32_MAX)
        return fail(KVR_ERR_INVALID_ARG, "negative or too large reservation (batch %d, spans %d, locals %d, "
                    "query tokens %lld)", max_batch, max_spans, max_locals, (long long)max_query_tokens);
    NvtxRange call("kvr_pool_reserve");
    kvr_status st;
    if ((st = ensure_device(p)) != KVR_OK)
        return st;
    DeviceGuard g(p->device);
    // the largest table a call within the limits uploads: an assemble's spans
    // and local sources, or a query attention's request / append tables
    const size_t asm_bytes = align16((size_t)max_spans * sizeof(DevSpan)) + (size_t)max_locals * sizeof(DevLocal);
    const size_t qa_bytes = align16((size_t)max_batch * sizeof(DevReq)) +
                            align16((size_t)max_batch * sizeof(DevSpan)) + (size_t)max_batch * sizeof(DevLocal);
    const size_t bytes = std::max(asm_bytes, qa_bytes);
    cudaError_t e;
    for (Slot &s : p->slots) {
        if (s.used && (e = cudaEventSynchronize(s.done)) != cudaSuccess)
            return cuda_fail(e, "staging slot wait");
        if ((st = kvr_pool::grow(s, bytes, bytes)) != KVR_OK)
            return st;
    }
    if (use_tensor_cores(*p)) {
        const size_t q_bytes = (size_t)p->d.n_layers * (size_t)max_query_tokens * p->d.n_q_heads * p->d.head_dim * 2;
        if (q_bytes > 0 && (st = p->grow_query_scratch(q_bytes)) != KVR_OK)
            return st;
    }
    return KVR_OK;
}

static bool use_tensor_cores(const kvr_pool &p)
{
    return attention_tc_supported(p.d.dtype, p.d.head_dim) && p.cc == 103 && p.encode;
}

// ---------------------------------------------------------------------------
// assemble
// ---------------------------------------------------------------------------
namespace {

kvr_status check_offsets32(const int32_t *o, int32_t batch, const char *name)
{
    if (!o)
        return fail(KVR_ERR_INVALID_ARG, "%s is NULL", name);
    if (o[0] != 0)
        return fail(KVR_ERR_INVALID_ARG, "%s[0] = %d, must be 0", name, o[0]);
    for (int b = 0; b < batch; ++b)
        if (o[b + 1] < o[b])
            return fail(KVR_ERR_INVALID_ARG, "%s decreases at %d", name, b);
    return KVR_OK;
}

kvr_status check_cache_offsets(const int64_t *o, int32_t batch)
{
    if (!o)
        return fail(KVR_ERR_INVALID_ARG, "cache_offsets is NULL");
    if (o[0] < 0)
        return fail(KVR_ERR_INVALID_ARG, "cache_offsets[0] < 0");
    for (int b = 0; b < batch; ++b)
        if (o[b + 1] < o[b] || o[b + 1] - o[b] > kMaxPosition)
            return fail(KVR_ERR_INVALID_ARG, "cache_offsets[%d..%d] invalid", b, b + 1);
    return KVR_OK;
}

kvr_status check_local(const kvr_pool &p, const kvr_local_src &lc, int i)
{
    if (!lc.k || !lc.v || !aligned16(lc.k) || !aligned16(lc.v))
        return fail(KVR_ERR_INVALID_ARG, "local source %d: k / v NULL or not 16-byte aligned", i);
    if (lc.len < 0 || lc.len > kMaxPosition)
        return fail(KVR_ERR_INVALID_ARG, "local source %d: len %lld", i, (long long)lc.len);
    for (int s = 0; s < 3; ++s)
        if (lc.stride[s] < 0 || lc.stride[s] % p.vec_elems())
            return fail(KVR_ERR_INVALID_ARG, "local source %d: stride[%d] = %lld", i, s,
                        (long long)lc.stride[s]);
    return KVR_OK;
}

// Units of (layer, kv-head) per assemble CTA: about 256 rows per CTA.
int units_per_cta(int LH, int64_t rows, int64_t n_spans)
{
    const int64_t avg = std::max<int64_t>(1, rows / std::max<int64_t>(1, n_spans));
    return (int)std::min<int64_t>(LH, std::max<int64_t>(1, 256 / avg));
}

}  // namespace

// One assemble call, validated (host tables built), then staged (device
// tables in kernel parameters or uploaded), then launched.
struct AsmPlan {
    std::vector<DevSpan> ds;
    std::vector<int32_t> plen;
    std::vector<int32_t> span0;   // request b's first entry of ds
    int64_t flat = 0;
    const kvr_local_src *locals = nullptr;
    int32_t n_locals = 0;
    void *cache_k = nullptr, *cache_v = nullptr;
    int32_t *pos_ids = nullptr, *src_map = nullptr;
    AssembleArgs a{};
    bool inl = false;
    bool upload = false;   // upload the tables even for a small call (a later kernel reads them)
    AssembleTables tab;
    Slot *slot = nullptr;
};

static kvr_status asm_validate(const kvr_pool &p, int32_t batch, const int32_t *span_offsets,
                               const kvr_span *spans, const kvr_local_src *locals, int32_t n_locals,
                               const int64_t *cache_offsets, uint32_t flags, AsmPlan &pl)
{
    if (flags & ~(uint32_t)KVR_POSITIONS_COMPOSITE)
        return fail(KVR_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    kvr_status st;
    if ((st = check_offsets32(span_offsets, batch, "span_offsets")) != KVR_OK ||
        (st = check_cache_offsets(cache_offsets, batch)) != KVR_OK)
        return st;
    const int32_t n_spans = span_offsets[batch];
    if (n_spans > 0 && !spans)
        return fail(KVR_ERR_INVALID_ARG, "spans is NULL");
    if (n_locals < 0 || (n_locals > 0 && !locals))
        return fail(KVR_ERR_INVALID_ARG, "locals NULL with n_locals %d", n_locals);
    for (int i = 0; i < n_locals; ++i)
        if ((st = check_local(p, locals[i], i)) != KVR_OK)
            return st;
    const bool composite = flags & KVR_POSITIONS_COMPOSITE;
    const int LH = p.d.n_layers * p.d.n_kv_heads;

    pl.locals = locals;
    pl.n_locals = n_locals;
    pl.ds.reserve(n_spans);
    pl.plen.assign(batch, 0);
    pl.span0.assign(batch, 0);
    int64_t flat = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t cap = cache_offsets[b + 1] - cache_offsets[b];
        int64_t row = 0;
        pl.span0[b] = (int32_t)pl.ds.size();
        for (int i = span_offsets[b]; i < span_offsets[b + 1]; ++i) {
            const kvr_span s = spans[i];
            int64_t src_len;
            if (s.src < 0)
                return fail(KVR_ERR_OUT_OF_RANGE, "span %d: negative source id %d", i, s.src);
            if (s.src & KVR_SRC_LOCAL) {
                const int idx = s.src & ~KVR_SRC_LOCAL;
                if (idx >= n_locals)
                    return fail(KVR_ERR_OUT_OF_RANGE, "span %d: local source %d of %d", i, idx,
                                n_locals);
                src_len = locals[idx].len;
            } else {
                if (s.src >= p.d.n_entries)
                    return fail(KVR_ERR_OUT_OF_RANGE, "span %d: pool entry %d of %lld", i, s.src,
                                (long long)p.d.n_entries);
                src_len = p.d.entry_len;
            }
            if (s.start < 0 || s.end < s.start || s.end > src_len)
                return fail(KVR_ERR_OUT_OF_RANGE, "span %d: [%d, %d) outside source of %lld tokens",
                            i, s.start, s.end, (long long)src_len);
            const int32_t len = s.end - s.start;
            const int64_t pos0 = composite ? s.start : row;
            if (pos0 + len > kMaxPosition)
                return fail(KVR_ERR_OUT_OF_RANGE, "span %d: positions beyond 2^24", i);
            if (len > 0) {
                DevSpan d{};
                d.dst_row0 = cache_offsets[b] * LH;
                d.flat0 = flat;
                d.src = s.src;
                d.start = s.start;
                d.len = len;
                d.row = (int32_t)row;
                d.pos0 = (int32_t)pos0;
                d.delta = (int32_t)(pos0 - s.start);
                d.cap = (int32_t)cap;
                d.dstep = 0;
                if (!(s.src & KVR_SRC_LOCAL) && (p.d.flags & KVR_POOL_KEYS_UNROTATED)) {
                    d.delta = (int32_t)pos0;   // token t turns by its position pos0 + t
                    d.dstep = 1;
                }
                pl.ds.push_back(d);
            }
            row += len;
            flat += len;
        }
        if (row > cap)
            return fail(KVR_ERR_OUT_OF_RANGE, "request %d: prefix %lld rows > cache block %lld", b,
                        (long long)row, (long long)cap);
        pl.plen[b] = (int32_t)row;
    }
    pl.flat = flat;
    return KVR_OK;
}

static kvr_status asm_check_outputs(AsmPlan &pl, void *cache_k, void *cache_v, int32_t *pos_ids,
                                    int32_t *src_map)
{
    if (!cache_k || !cache_v || !aligned16(cache_k) || !aligned16(cache_v))
        return fail(KVR_ERR_INVALID_ARG, "cache_k / cache_v NULL or not 16-byte aligned");
    pl.cache_k = cache_k;
    pl.cache_v = cache_v;
    pl.pos_ids = pos_ids;
    pl.src_map = src_map;
    return KVR_OK;
}

// Kernel arguments and tables; large tables go up by one H2D copy from a
// pinned staging slot.  Device setup must be done.
static kvr_status asm_stage(kvr_pool *p, AsmPlan &pl, cudaStream_t s)
{
    const int LH = p->d.n_layers * p->d.n_kv_heads;
    AssembleArgs &a = pl.a;
    a.rope = p->rope;
    a.pool_k = p->d.k;
    a.pool_v = p->d.v;
    a.ps_entry = p->d.stride[0];
    a.ps_layer = p->d.stride[1];
    a.ps_head = p->d.stride[2];
    a.ps_tok = p->d.stride[3];
    a.cache_k = pl.cache_k;
    a.cache_v = pl.cache_v;
    a.pos_ids = pl.pos_ids;
    a.src_map = pl.src_map;
    a.n_layers = p->d.n_layers;
    a.n_heads = p->d.n_kv_heads;
    a.upc = units_per_cta(LH, pl.flat, (int64_t)pl.ds.size());
    a.interleaved = (p->d.flags & KVR_POOL_ROPE_INTERLEAVED) ? 1 : 0;
    const int n_locals = pl.n_locals;
    const kvr_local_src *locals = pl.locals;
    pl.inl = !pl.upload && (int)pl.ds.size() <= kInlineEntries && n_locals <= kInlineEntries;
    if (pl.inl) {
        // small call: the tables travel inside the kernel parameters
        std::memcpy(pl.tab.spans, pl.ds.data(), pl.ds.size() * sizeof(DevSpan));
        for (int i = 0; i < n_locals; ++i)
            pl.tab.locals[i] = DevLocal{locals[i].k, locals[i].v, locals[i].stride[0], locals[i].stride[1],
                                        locals[i].stride[2], locals[i].len};
        return KVR_OK;
    }
    const size_t off_loc = align16(pl.ds.size() * sizeof(DevSpan));
    const size_t bytes = off_loc + sizeof(DevLocal) * std::max(n_locals, 0);
    kvr_status st;
    if ((st = p->acquire(bytes, bytes, &pl.slot)) != KVR_OK)
        return st;
    char *h = static_cast<char *>(pl.slot->host);
    std::memcpy(h, pl.ds.data(), pl.ds.size() * sizeof(DevSpan));
    for (int i = 0; i < n_locals; ++i) {
        DevLocal l{locals[i].k, locals[i].v, locals[i].stride[0], locals[i].stride[1],
                   locals[i].stride[2], locals[i].len};
        std::memcpy(h + off_loc + i * sizeof(DevLocal), &l, sizeof l);
    }
    cudaError_t e = cudaMemcpyAsync(pl.slot->dev, h, bytes, cudaMemcpyHostToDevice, s);
    cudaEventRecord(pl.slot->done, s);   // the slot is busy from here on
    pl.slot->used = true;
    if (e != cudaSuccess)
        return cuda_fail(e, "span table upload");
    a.spans = static_cast<const DevSpan *>(pl.slot->dev);
    a.locals = reinterpret_cast<const DevLocal *>(static_cast<char *>(pl.slot->dev) + off_loc);
    return KVR_OK;
}

// `record_slot` false: the caller records the staging slot's event after the
// kernels that follow (nothing may sit between this kernel and a dependent
// launched programmatically after it).
static kvr_status asm_launch(kvr_pool *p, AsmPlan &pl, cudaStream_t s, bool record_slot = true)
{
    NvtxRange r("kvr.k_assemble");
    p->mark(0, s);
    cudaError_t e = launch_assemble(pl.a, p->d.dtype, p->d.head_dim, (int)pl.ds.size(), s,
                                    pl.inl ? &pl.tab : nullptr);
    p->mark(1, s);
    if (pl.slot && record_slot)
        cudaEventRecord(pl.slot->done, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "assemble launch");
    return KVR_OK;
}

extern "C" kvr_status kvr_assemble(kvr_pool_t p, int32_t batch, const int32_t *span_offsets,
                                   const kvr_span *spans, const kvr_local_src *locals,
                                   int32_t n_locals, const int64_t *cache_offsets, void *cache_k,
                                   void *cache_v, int32_t *pos_ids, int32_t *src_map,
                                   int32_t *prefix_len, uint32_t flags, void *stream)
{
    if (!p)
        return fail(KVR_ERR_INVALID_ARG, "pool is NULL");
    if (batch < 0)
        return fail(KVR_ERR_INVALID_ARG, "batch %d", batch);
    if (batch == 0)
        return KVR_OK;
    NvtxRange call("kvr_assemble");
    AsmPlan pl;
    kvr_status st;
    if ((st = asm_validate(*p, batch, span_offsets, spans, locals, n_locals, cache_offsets, flags,
                           pl)) != KVR_OK)
        return st;
    if (prefix_len)
        std::copy(pl.plen.begin(), pl.plen.end(), prefix_len);
    if (pl.ds.empty())
        return KVR_OK;
    if ((st = asm_check_outputs(pl, cache_k, cache_v, pos_ids, src_map)) != KVR_OK ||
        (st = ensure_device(p)) != KVR_OK)
        return st;
    DeviceGuard g(p->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = asm_stage(p, pl, s)) != KVR_OK)
        return st;
    return asm_launch(p, pl, s);
}

// ---------------------------------------------------------------------------
// query attention
// ---------------------------------------------------------------------------
namespace {

kvr_status encode_cache_map(const kvr_pool &p, void *base, int64_t rows, CUtensorMap *m)
{
    if (!p.encode)
        return fail(KVR_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled not available");
    const cuuint64_t dims[2] = {(cuuint64_t)p.d.head_dim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)p.d.head_dim * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = p.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(KVR_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return KVR_OK;
}

// The output [L * T][H_q][D] as a 3-D tensor with a box of one 64-column half
// of G heads x 32 / G tokens (a warp's 32 packed rows), 128-byte swizzle.
kvr_status encode_out_map(const kvr_pool &p, void *base, int64_t tokens, CUtensorMap *m)
{
    if (!p.encode)
        return fail(KVR_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled not available");
    const int G = p.d.n_q_heads / p.d.n_kv_heads;
    const cuuint64_t dims[3] = {(cuuint64_t)p.d.head_dim, (cuuint64_t)p.d.n_q_heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)p.d.head_dim * 2, (cuuint64_t)p.d.n_q_heads * p.d.head_dim * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(32 / G)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = p.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(KVR_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", (int)r);
    return KVR_OK;
}

// The pool as a 2-D [entries * L * H_kv * entry_len, D] tensor with a box of
// `box_rows` rows (64 columns): the values-gathering attention's TMA source.
kvr_status encode_gather_map(const kvr_pool &p, const void *base, CUtensorMap *m, uint32_t box_rows)
{
    if (!p.encode)
        return fail(KVR_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled not available");
    const int64_t rows = p.d.n_entries * p.d.n_layers * p.d.n_kv_heads * p.d.entry_len;
    const cuuint64_t dims[2] = {(cuuint64_t)p.d.head_dim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)p.d.head_dim * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = p.encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(KVR_ERR_CUDA, "cuTensorMapEncodeTiled (pool values) failed (%d)", (int)r);
    return KVR_OK;
}

// What the values-gathering attention needs beyond a query-attention launch:
// the pool's values (as a pointer, and as gather4 / 32-row box TMA sources)
// and the span table.
struct GatherLaunch {
    CUtensorMap mpv{}, mbv{};
    GatherArgs g{};
    SpanTable st;
    bool inl = false;
};

}  // namespace

// One query-attention call, validated, staged, launched (as the assemble).
struct QaPlan {
    int32_t batch = 0, T = 0, m_blocks = 0, max_lq = 0;
    const int64_t *cache_offsets = nullptr;
    const int32_t *q_offsets = nullptr;
    const void *q = nullptr, *kq = nullptr, *vq = nullptr;
    void *cache_k = nullptr, *cache_v = nullptr, *out = nullptr;
    float scale = 0.f;
    std::vector<DevReq> rq;
    std::vector<DevSpan> ap;     // the query keys / values as append spans (CUDA-core path)
    std::vector<DevLocal> al;
    bool tc = false, inl = false;
    int32_t parts = 1;           // layer groups of a host-pool prefill (attention per group)
    CUtensorMap mq, mk, mv, mo;
    ReqTable rt_inl;
    AssembleTables tab;
    AssembleArgs a{};
    AttnArgs at{};
    Slot *slot = nullptr;
};

// Host checks and tables.  T = 0 (no query token) leaves nothing to do.
static kvr_status qa_validate(const kvr_pool &p, int32_t batch, const int64_t *cache_offsets,
                              const int32_t *prefix_len, const int32_t *q_offsets, const void *q,
                              const void *kq, const void *vq, void *cache_k, void *cache_v, void *out,
                              float softmax_scale, QaPlan &pl)
{
    kvr_status st;
    if ((st = check_cache_offsets(cache_offsets, batch)) != KVR_OK ||
        (st = check_offsets32(q_offsets, batch, "q_offsets")) != KVR_OK)
        return st;
    if (!prefix_len)
        return fail(KVR_ERR_INVALID_ARG, "prefix_len is NULL");
    if (!(softmax_scale >= 0.f) || !std::isfinite(softmax_scale))
        return fail(KVR_ERR_INVALID_ARG, "softmax_scale %g", (double)softmax_scale);
    pl.T = q_offsets[batch];
    if (pl.T == 0)
        return KVR_OK;
    const void *ptrs[] = {q, kq, vq, cache_k, cache_v, out};
    for (const void *x : ptrs)
        if (!x || !aligned16(x))
            return fail(KVR_ERR_INVALID_ARG, "q / kq / vq / cache / out NULL or not 16-byte aligned");
    for (int b = 0; b < batch; ++b) {
        const int64_t cap = cache_offsets[b + 1] - cache_offsets[b];
        const int32_t P = prefix_len[b];
        const int32_t Lq = q_offsets[b + 1] - q_offsets[b];
        if (P < 0 || (int64_t)P + Lq > cap)
            return fail(KVR_ERR_OUT_OF_RANGE, "request %d: prefix %d + query %d > cache block %lld",
                        b, P, Lq, (long long)cap);
    }
    pl.batch = batch;
    pl.cache_offsets = cache_offsets;
    pl.q_offsets = q_offsets;
    pl.q = q;
    pl.kq = kq;
    pl.vq = vq;
    pl.cache_k = cache_k;
    pl.cache_v = cache_v;
    pl.out = out;
    pl.scale = softmax_scale;

    const int L = p.d.n_layers, Hkv = p.d.n_kv_heads, Hq = p.d.n_q_heads, D = p.d.head_dim;
    const int LH = L * Hkv;
    const int G = Hq / Hkv;
    const int64_t T = pl.T;
    pl.rq.resize(batch);
    for (int b = 0; b < batch; ++b) {
        const int64_t cap = cache_offsets[b + 1] - cache_offsets[b];
        const int32_t P = prefix_len[b];
        const int32_t Lq = q_offsets[b + 1] - q_offsets[b];
        pl.max_lq = std::max(pl.max_lq, Lq);
        DevReq &r = pl.rq[b];
        r.cache_row0 = cache_offsets[b] * LH;
        r.cap = (int32_t)cap;
        r.prefix = P;
        r.q_off = q_offsets[b];
        r.q_len = Lq;
        r.unit0 = 0;   // set by the schedule (tensor-core path)
        r.span0 = r.span_end = 0;
        pl.m_blocks += (int32_t)((int64_t(G) * Lq + 255) / 256);
        if (Lq > 0) {
            // the query tokens' keys / values become cache rows P..P+Lq-1;
            // their keys arrive un-rotated, so token t turns by P + t
            DevSpan d{};
            d.dst_row0 = r.cache_row0;
            d.flat0 = 0;
            d.src = KVR_SRC_LOCAL | (int32_t)pl.al.size();
            d.start = 0;
            d.len = Lq;
            d.row = P;
            d.pos0 = P;
            d.delta = P;
            d.cap = (int32_t)cap;
            d.dstep = 1;
            pl.ap.push_back(d);
            const int64_t off = (int64_t)q_offsets[b] * Hkv * D * p.elt();
            DevLocal l{static_cast<const char *>(kq) + off, static_cast<const char *>(vq) + off,
                       T * Hkv * D, D, (int64_t)Hkv * D, Lq};
            pl.al.push_back(l);
        }
    }
    return KVR_OK;
}

// Scratch, tensor maps and tables.  Device setup must be done.
static kvr_status qa_stage(kvr_pool *p, QaPlan &pl, cudaStream_t s)
{
    const int L = p->d.n_layers, Hkv = p->d.n_kv_heads, Hq = p->d.n_q_heads, D = p->d.head_dim;
    const int LH = L * Hkv;
    const int32_t batch = pl.batch, T = pl.T;
    kvr_status st;
    cudaError_t e;
    pl.tc = use_tensor_cores(*p);
    if (pl.tc) {
        // rotated packed Q scratch and the three tensor maps
        const int64_t rows = pl.cache_offsets[batch] * LH;
        const int64_t q_rows = (int64_t)L * T * Hq;
        if (rows > (int64_t)INT32_MAX - 256 || q_rows > (int64_t)INT32_MAX - 256)   // int32 TMA coordinates
            return fail(KVR_ERR_UNSUPPORTED, "cache or query rows exceed the int32 TMA coordinate range");
        if ((st = p->grow_query_scratch((size_t)q_rows * D * 2)) != KVR_OK)
            return st;
        if ((st = encode_cache_map(*p, p->q_rot, q_rows, &pl.mq)) != KVR_OK ||
            (st = encode_cache_map(*p, pl.cache_k, rows, &pl.mk)) != KVR_OK ||
            (st = encode_cache_map(*p, pl.cache_v, rows, &pl.mv)) != KVR_OK)
            return st;
        // G a power of two and `out` in device memory: the attention's epilogue
        // writes each warp's 32 rows (32 / G whole tokens) with one TMA store
        const int G = Hq / Hkv;
        pl.at.out_tma = 0;
        if ((G & (G - 1)) == 0 && G <= 32) {
            cudaPointerAttributes pa{};
            if (cudaPointerGetAttributes(&pa, pl.out) == cudaSuccess && pa.type == cudaMemoryTypeDevice) {
                if ((st = encode_out_map(*p, pl.out, (int64_t)L * T, &pl.mo)) != KVR_OK)
                    return st;
                pl.at.out_tma = 1;
            } else {
                cudaGetLastError();
            }
        }
        // the previous call's attention must be done with the query scratch
        if (p->q_rot_used && (e = cudaStreamWaitEvent(s, p->q_rot_done, 0)) != cudaSuccess)
            return cuda_fail(e, "query scratch ordering");
    }

    if (pl.tc) {
        // schedule: requests with the longest key range first (requests
        // without query tokens last), each request's units numbered after the
        // previous one's; the table goes up in this order
        std::stable_sort(pl.rq.begin(), pl.rq.end(), [](const DevReq &x, const DevReq &y) {
            if ((x.q_len > 0) != (y.q_len > 0))
                return x.q_len > 0;
            return x.prefix + x.q_len > y.prefix + y.q_len;
        });
        int64_t u0 = 0;
        for (DevReq &r : pl.rq) {
            r.unit0 = (int32_t)u0;
            u0 += ((int64_t)(Hq / Hkv) * r.q_len + 255) / 256 * (LH / pl.parts);
        }
    }

    pl.inl = batch <= kInlineEntries;   // then ap, al have <= batch entries too
    AssembleArgs &a = pl.a;
    AttnArgs &at = pl.at;
    if (pl.inl) {
        std::memcpy(pl.rt_inl.reqs, pl.rq.data(), pl.rq.size() * sizeof(DevReq));
        std::memcpy(pl.tab.spans, pl.ap.data(), pl.ap.size() * sizeof(DevSpan));
        std::memcpy(pl.tab.locals, pl.al.data(), pl.al.size() * sizeof(DevLocal));
        at.reqs = nullptr;
    } else {
        const size_t off_sp = align16(pl.rq.size() * sizeof(DevReq));
        const size_t off_lc = off_sp + align16(pl.ap.size() * sizeof(DevSpan));
        const size_t bytes = off_lc + pl.al.size() * sizeof(DevLocal);
        if ((st = p->acquire(bytes, bytes, &pl.slot)) != KVR_OK)
            return st;
        char *h = static_cast<char *>(pl.slot->host);
        char *dv = static_cast<char *>(pl.slot->dev);
        std::memcpy(h, pl.rq.data(), pl.rq.size() * sizeof(DevReq));
        std::memcpy(h + off_sp, pl.ap.data(), pl.ap.size() * sizeof(DevSpan));
        std::memcpy(h + off_lc, pl.al.data(), pl.al.size() * sizeof(DevLocal));
        e = cudaMemcpyAsync(dv, h, bytes, cudaMemcpyHostToDevice, s);
        cudaEventRecord(pl.slot->done, s);   // the slot is busy from here on
        pl.slot->used = true;
        if (e != cudaSuccess)
            return cuda_fail(e, "request table upload");
        a.spans = reinterpret_cast<const DevSpan *>(dv + off_sp);
        a.locals = reinterpret_cast<const DevLocal *>(dv + off_lc);
        at.reqs = reinterpret_cast<const DevReq *>(dv);
    }

    at.n_reqs = batch;
    at.rope = p->rope;
    at.q = pl.q;
    at.cache_k = pl.cache_k;
    at.cache_v = pl.cache_v;
    at.out = pl.out;
    at.n_layers = L;
    at.n_q_heads = Hq;
    at.n_kv_heads = Hkv;
    at.total_q = T;
    at.scale_log2 = (pl.scale > 0.f ? pl.scale : 1.f / std::sqrt((float)D)) * 1.4426950408889634f;
    at.err = p->err;
    at.interleaved = (p->d.flags & KVR_POOL_ROPE_INTERLEAVED) ? 1 : 0;
    // CUDA-core path: the query keys / values are appended by the assemble
    // kernel (un-rotated source, token t turned by P + t); the query heads
    // are rotated inside the CUDA-core attention kernel
    a.rope = p->rope;
    a.cache_k = pl.cache_k;
    a.cache_v = pl.cache_v;
    a.n_layers = L;
    a.n_heads = Hkv;
    a.upc = 1;
    a.interleaved = at.interleaved;
    return KVR_OK;
}

// `after_assemble`: the kernel just enqueued on `s` is the assemble kernel of
// the same prefill, so the query prologue may overlap it.  Without the timing
// hook the attention kernel always overlaps the prologue's tail.
static kvr_status qa_launch(kvr_pool *p, QaPlan &pl, cudaStream_t s, bool after_assemble,
                            const GatherLaunch *gl = nullptr)
{
    static const ReqTable no_reqs{};
    const ReqTable &rt = pl.inl ? pl.rt_inl : no_reqs;
    const int D = p->d.head_dim;
    cudaError_t e;
    if (pl.tc) {
        // a host-pool prefill in layer groups, stitched last group first: the
        // attention of group g runs on the SMs the stitch leaves, beside the
        // stitch of group g - 1, once the stitch of group g is done
        const int n_sms = pl.parts > 1 ? p->n_sms - kHostStitchCtas : p->n_sms;
        const int lh_part = p->d.n_layers * p->d.n_kv_heads / pl.parts;
        TcAttnArgs ta{pl.at, &rt, &pl.mq, &pl.mk, &pl.mv, pl.m_blocks, n_sms};
        ta.tmap_out = &pl.mo;
        if (pl.parts > 1)
            ta.base.lh_count = lh_part;
        // the last wave's units split in two halves of their keys when two
        // halves of each fit one wave and the grid can run as two-CTA clusters
        const int64_t units = (int64_t)pl.m_blocks * lh_part;
        const int64_t tail = units % n_sms;
        ta.base.n_full = (int32_t)units;
        if (tail > 0 && 2 * tail <= n_sms && attention_tc_pairs_fit(n_sms))
            ta.base.n_full = (int32_t)(units - tail);
        QueryPrologueArgs qp{pl.at.reqs, p->rope, pl.q, pl.kq, pl.vq, pl.cache_k, pl.cache_v, p->q_rot,
                             p->d.n_layers, p->d.n_q_heads, p->d.n_kv_heads, pl.T, pl.max_lq, pl.batch,
                             pl.at.interleaved};
        // a decode step (one query token per request): one kernel rotates,
        // appends and streams each cache block
        const bool decode = !gl && pl.max_lq == 1 &&
                            decode_supported(p->d.dtype, D, p->d.n_q_heads / p->d.n_kv_heads);
        p->mark(2, s);
        if (!decode) {
            NvtxRange r("kvr.k_query_prologue");
            e = launch_query_prologue(qp, rt, p->n_sms, after_assemble && !p->timed, s);
        } else {
            e = cudaSuccess;
        }
        p->mark(3, s);
        if (e == cudaSuccess && decode) {
            const DecodeIO io{pl.kq, pl.vq, pl.cache_k, pl.cache_v, pl.at.interleaved};
            p->mark(4, s);
            {
                NvtxRange r("kvr.k_decode_attention");
                e = launch_decode_attention(pl.at, rt, &pl.mk, &pl.mv, io, !p->timed, s);
            }
            p->mark(5, s);
        } else if (e == cudaSuccess) {
            NvtxRange r(gl ? "kvr.k_attention_tc_values_gathered" : "kvr.k_attention_tc");
            if (pl.parts > 1) {
                p->mark(4, s);
                for (int g = pl.parts - 1; g >= 0 && e == cudaSuccess; --g) {
                    if ((e = cudaStreamWaitEvent(s, p->part_ev[g], 0)) != cudaSuccess)
                        break;
                    ta.base.lh_base = g * lh_part;
                    e = launch_attention_tc(ta, false, s);
                }
                p->mark(5, s);
            } else {
                if (gl) {
                    ta.gather_v = true;
                    ta.tmap_pv = &gl->mpv;
                    ta.tmap_bv = &gl->mbv;
                    ta.g = gl->g;
                    ta.st = gl->inl ? &gl->st : nullptr;
                }
                p->mark(4, s);
                e = launch_attention_tc(ta, !p->timed, s);
                p->mark(5, s);
            }
        }
        cudaEventRecord(p->q_rot_done, s);
        p->q_rot_used = true;
    } else {
        NvtxRange r("kvr.k_attention_simt");
        p->mark(2, s);
        e = launch_assemble(pl.a, p->d.dtype, D, (int)pl.ap.size(), s, pl.inl ? &pl.tab : nullptr);
        p->mark(3, s);
        if (e == cudaSuccess) {
            p->mark(4, s);
            e = launch_attention_simt(pl.at, rt, p->d.dtype, D, s);
            p->mark(5, s);
        }
    }
    if (pl.slot)
        cudaEventRecord(pl.slot->done, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "attention launch");
    return KVR_OK;
}

extern "C" kvr_status kvr_query_attention(kvr_pool_t p, int32_t batch, const int64_t *cache_offsets,
                                          const int32_t *prefix_len, const int32_t *q_offsets,
                                          const void *q, const void *kq, const void *vq,
                                          void *cache_k, void *cache_v, void *out,
                                          float softmax_scale, void *stream)
{
    if (!p)
        return fail(KVR_ERR_INVALID_ARG, "pool is NULL");
    if (batch < 0)
        return fail(KVR_ERR_INVALID_ARG, "batch %d", batch);
    if (batch == 0)
        return KVR_OK;
    NvtxRange call("kvr_query_attention");
    QaPlan pl;
    kvr_status st;
    if ((st = qa_validate(*p, batch, cache_offsets, prefix_len, q_offsets, q, kq, vq, cache_k, cache_v,
                          out, softmax_scale, pl)) != KVR_OK)
        return st;
    if (pl.T == 0)
        return KVR_OK;
    if ((st = ensure_device(p)) != KVR_OK)
        return st;
    DeviceGuard g(p->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = qa_stage(p, pl, s)) != KVR_OK)
        return st;
    return qa_launch(p, pl, s, false);
}

// ---------------------------------------------------------------------------
// prefill = assemble + query attention in one call
// ---------------------------------------------------------------------------
extern "C" kvr_status kvr_prefill(kvr_pool_t p, int32_t batch, const int32_t *span_offsets,
                                  const kvr_span *spans, const kvr_local_src *locals, int32_t n_locals,
                                  const int64_t *cache_offsets, void *cache_k, void *cache_v,
                                  int32_t *pos_ids, int32_t *src_map, int32_t *prefix_len,
                                  uint32_t flags, const int32_t *q_offsets, const void *q,
                                  const void *kq, const void *vq, void *out, float softmax_scale,
                                  void *stream)
{
    if (!p)
        return fail(KVR_ERR_INVALID_ARG, "pool is NULL");
    if (batch < 0)
        return fail(KVR_ERR_INVALID_ARG, "batch %d", batch);
    if (batch == 0)
        return KVR_OK;
    NvtxRange call("kvr_prefill");
    // every check of both halves before anything is enqueued
    const bool gather = flags & KVR_PREFILL_SKIP_PREFIX_CACHE;
    // the pool seen as one 2-D [rows, D] tensor for TMA box loads of value tiles
    bool tma_pool = false;
    if (gather) {
        const kvr_pool_desc &d = p->d;
        const int64_t E = d.entry_len, D = d.head_dim;
        tma_pool = d.stride[3] == D && d.stride[2] == E * D && d.stride[1] == d.n_kv_heads * E * D &&
                   d.stride[0] == (int64_t)d.n_layers * d.n_kv_heads * E * D &&
                   d.n_entries * d.n_layers * d.n_kv_heads * E <= INT32_MAX;
        if (d.dtype != KVR_DTYPE_BF16 || D != 128)
            return fail(KVR_ERR_UNSUPPORTED, "KVR_PREFILL_SKIP_PREFIX_CACHE needs a bf16 pool with head_dim 128");
    }
    AsmPlan ap;
    QaPlan qp;
    kvr_status st;
    if ((st = asm_validate(*p, batch, span_offsets, spans, locals, n_locals, cache_offsets,
                           flags & ~(uint32_t)KVR_PREFILL_SKIP_PREFIX_CACHE, ap)) != KVR_OK ||
        (st = qa_validate(*p, batch, cache_offsets, ap.plen.data(), q_offsets, q, kq, vq, cache_k,
                          cache_v, out, softmax_scale, qp)) != KVR_OK)
        return st;
    const bool stitch = !ap.ds.empty();
    if (stitch && (st = asm_check_outputs(ap, cache_k, cache_v, pos_ids, src_map)) != KVR_OK)
        return st;
    if (prefix_len)
        std::copy(ap.plen.begin(), ap.plen.end(), prefix_len);
    if (!stitch && qp.T == 0)
        return KVR_OK;
    if ((st = ensure_device(p)) != KVR_OK)
        return st;
    DeviceGuard g(p->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (gather) {
        // the stitch writes the prefix keys (re-rotated) and the maps only; the
        // attention reads the keys from the cache and gathers the prefix values
        // from the pool
        if (!use_tensor_cores(*p))
            return fail(KVR_ERR_UNSUPPORTED, "KVR_PREFILL_SKIP_PREFIX_CACHE needs the tensor-core attention");
        cudaPointerAttributes pa{};
        if (cudaPointerGetAttributes(&pa, p->d.k) != cudaSuccess || pa.type != cudaMemoryTypeDevice) {
            cudaGetLastError();
            return fail(KVR_ERR_UNSUPPORTED, "KVR_PREFILL_SKIP_PREFIX_CACHE needs the pool in device memory");
        }
        if (qp.T == 0)
            return KVR_OK;
        GatherLaunch gl;
        gl.g.pool_v = p->d.v;
        gl.g.ps_entry = p->d.stride[0];
        gl.g.ps_layer = p->d.stride[1];
        gl.g.ps_head = p->d.stride[2];
        gl.g.ps_tok = p->d.stride[3];
        gl.g.tma_pool = tma_pool ? 1 : 0;
        if (tma_pool && ((st = encode_gather_map(*p, p->d.v, &gl.mpv, 1)) != KVR_OK ||
                         (st = encode_gather_map(*p, p->d.v, &gl.mbv, 32)) != KVR_OK))
            return st;
        for (int b = 0; b < batch; ++b) {
            DevReq &r = qp.rq[b];
            r.span0 = ap.span0[b];
            r.span_end = b + 1 < batch ? ap.span0[b + 1] : (int32_t)ap.ds.size();
            // spans of 96 rows or more on average, all from a pool that TMA can
            // address as one tensor: the prefix value tiles go through TMA box
            // loads (runs of 32 pool rows), else through the gather warps
            const int64_t n_sp = r.span_end - r.span0;
            bool long_pool_spans = tma_pool && n_sp > 0 && (int64_t)ap.plen[b] >= 96 * n_sp;
            for (int i = r.span0; long_pool_spans && i < r.span_end; ++i)
                long_pool_spans = (ap.ds[i].src & KVR_SRC_LOCAL) == 0;
            r.flags = long_pool_spans ? kReqValuesTma : 0;
        }
        // the attention reads the local-source table from device memory
        ap.upload = n_locals > 0;
        if ((stitch && (st = asm_stage(p, ap, s)) != KVR_OK) || (st = qa_stage(p, qp, s)) != KVR_OK)
            return st;
        gl.inl = !stitch || ap.inl;
        if (stitch && ap.inl)
            std::memcpy(gl.st.spans, ap.tab.spans, ap.ds.size() * sizeof(DevSpan));
        gl.g.spans = gl.inl ? nullptr : ap.a.spans;
        // (NULL when no span names a request-local source: the attention then
        // runs its pool-only variant)
        gl.g.locals = n_locals > 0 && !gl.inl ? ap.a.locals : nullptr;
        gl.g.n_spans = (int32_t)ap.ds.size();
        gl.g.entry_len = (int32_t)p->d.entry_len;
        if (stitch) {
            ap.a.keys_only = 1;
            if ((st = asm_launch(p, ap, s, false)) != KVR_OK) {
                if (ap.slot)
                    cudaEventRecord(ap.slot->done, s);
                return st;
            }
        }
        st = qa_launch(p, qp, s, stitch, &gl);
        if (ap.slot)
            cudaEventRecord(ap.slot->done, s);
        return st;
    }
    // a pool in pinned host memory: layer groups, whose stitch (bound by the
    // CPU-GPU link, on a bounded grid and a second stream) overlaps the
    // previous group's attention
    const int L = p->d.n_layers;
    if (p->host_pool && stitch && qp.max_lq > 1 && use_tensor_cores(*p))
        for (int n = kMaxLayerParts; n > 1; --n)
            if (L % n == 0) {
                qp.parts = n;
                break;
            }
    // uploads and stream waits first, so that the kernels follow one another
    // on the stream with nothing in between
    if ((stitch && (st = asm_stage(p, ap, s)) != KVR_OK) ||
        (qp.T > 0 && (st = qa_stage(p, qp, s)) != KVR_OK))
        return st;
    if (qp.parts > 1) {
        cudaError_t e = cudaSuccess;
        if (!p->side && (e = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e, "host-pool stitch stream");
        if (!p->side_start && (e = cudaEventCreateWithFlags(&p->side_start, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "host-pool stitch event");
        for (int g = 0; g < qp.parts; ++g)
            if (!p->part_ev[g] && (e = cudaEventCreateWithFlags(&p->part_ev[g], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e, "host-pool stitch event");
        // the stitch stream starts after everything the caller's stream holds
        if ((e = cudaEventRecord(p->side_start, s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(p->side, p->side_start, 0)) != cudaSuccess)
            return cuda_fail(e, "host-pool stitch ordering");
        // The last 128-key tile of a request's last block reaches into the
        // first rows of the next request's first block, which the last stitch
        // group (the first layers) writes: until then those prefix rows' values
        // must be finite, since a masked key has weight 0 but 0 x NaN is NaN.
        const int LHn = L * p->d.n_kv_heads;
        const size_t row_bytes = (size_t)p->d.head_dim * p->elt();
        for (int b = 1; b < batch && e == cudaSuccess; ++b) {
            const int64_t rows = std::min<int64_t>(ap.plen[b], 128);
            if (rows > 0)
                e = cudaMemsetAsync(static_cast<char *>(cache_v) + (size_t)cache_offsets[b] * LHn * row_bytes, 0,
                                    (size_t)rows * row_bytes, p->side);
        }
        const int lh_part = LHn / qp.parts;
        for (int g = qp.parts - 1; g >= 0 && e == cudaSuccess; --g) {
            NvtxRange r("kvr.k_assemble_loop");
            AssembleArgs a = ap.a;
            a.lh_begin = g * lh_part;
            a.lh_count = lh_part;
            a.max_ctas = kHostStitchCtas;
            if ((e = launch_assemble(a, p->d.dtype, p->d.head_dim, (int)ap.ds.size(), p->side,
                                     ap.inl ? &ap.tab : nullptr)) == cudaSuccess)
                e = cudaEventRecord(p->part_ev[g], p->side);
        }
        if (e != cudaSuccess) {
            if (ap.slot)
                cudaEventRecord(ap.slot->done, s);
            return cuda_fail(e, "host-pool stitch launch");
        }
        st = qa_launch(p, qp, s, false);
        if (ap.slot)   // after the last group's attention, which waited for every stitch group
            cudaEventRecord(ap.slot->done, s);
        return st;
    }
    if (stitch && (st = asm_launch(p, ap, s, false)) != KVR_OK) {
        if (ap.slot)
            cudaEventRecord(ap.slot->done, s);
        return st;
    }
    if (qp.T > 0)
        st = qa_launch(p, qp, s, stitch);
    if (ap.slot)
        cudaEventRecord(ap.slot->done, s);
    return st;
}

// ---------------------------------------------------------------------------
// status
// ---------------------------------------------------------------------------
extern "C" kvr_status kvr_check(kvr_pool_t p, void *stream)
{
    if (!p)
        return fail(KVR_ERR_INVALID_ARG, "pool is NULL");
    kvr_status st;
    if ((st = ensure_device(p)) != KVR_OK)
        return st;
    DeviceGuard g(p->device);
    cudaError_t e;
    if ((e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != cudaSuccess)
        return cuda_fail(e, "stream synchronize");
    int w = 0;
    if ((e = cudaMemcpy(&w, p->err, sizeof w, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "error word read");
    if (w == kDevOk)
        return KVR_OK;
    cudaMemset(p->err, 0, sizeof(int));
    if (w == kDevTimeout)
        return fail(KVR_ERR_TIMEOUT, "a kernel's bounded wait ran out");
    if (w == kDevBadInput)
        return fail(KVR_ERR_DEVICE_CHECK, "an attention row's softmax denominator was not finite and positive "
                                          "(NaN or infinity in the query heads or the keys it attends to)");
    return fail(KVR_ERR_DEVICE_CHECK, "a kernel flagged device-side input (code %d)", w);
}

extern "C" const char *kvr_status_string(kvr_status s)
{
    switch (s) {
    case KVR_OK: return "KVR_OK";
    case KVR_ERR_INVALID_ARG: return "KVR_ERR_INVALID_ARG";
    case KVR_ERR_OUT_OF_RANGE: return "KVR_ERR_OUT_OF_RANGE";
    case KVR_ERR_UNSUPPORTED: return "KVR_ERR_UNSUPPORTED";
    case KVR_ERR_CUDA: return "KVR_ERR_CUDA";
    case KVR_ERR_TIMEOUT: return "KVR_ERR_TIMEOUT";
    case KVR_ERR_DEVICE_CHECK: return "KVR_ERR_DEVICE_CHECK";
    }
    return "KVR_ERR_UNKNOWN";
}

extern "C" const char *kvr_last_error(void) { return g_last_error; }

extern "C" kvr_status kvr_set_timing_events(kvr_pool_t p, void *const *events)
{
    if (!p)
        return fail(KVR_ERR_INVALID_ARG, "pool is NULL");
    p->timed = events != nullptr;
    for (int i = 0; i < 6; ++i)
        p->timing[i] = events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
    return KVR_OK;
}

extern "C" kvr_status kvr_selftest_wait(kvr_pool_t p, uint64_t limit_ns, void *stream)
{
    if (!p)
        return fail(KVR_ERR_INVALID_ARG, "pool is NULL");
    kvr_status st;
    if ((st = ensure_device(p)) != KVR_OK)
        return st;
    DeviceGuard g(p->device);
    const unsigned long long lim = std::min<uint64_t>(std::max<uint64_t>(limit_ns, 1000ull), 2000000000ull);
    const cudaError_t e = launch_wait_selftest(p->err, lim, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "self-test launch");
    return KVR_OK;
}

extern "C" int32_t kvr_attention_path(kvr_pool_t p)
{
    if (!p)
        return -2;
    if (!p->ready)
        return KVR_PATH_UNBOUND;
    return use_tensor_cores(*p) ? KVR_PATH_TCGEN05 : KVR_PATH_CUDA_CORES;
}
