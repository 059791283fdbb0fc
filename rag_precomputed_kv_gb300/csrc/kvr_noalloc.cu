// kvr_noalloc.cu -- kvr_assemble_noalloc: the assemble step for callers that
// cannot allocate memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they stitch a prefix: a serving engine whose caching allocator already
// holds all free device memory, so a raw cudaMalloc would fail or fragment
// its pool; a latency-critical request loop where an allocation (and the
// synchronization it can imply) is not allowed; a plug-in loaded into a host
// program that forbids allocations outside its own allocator.  For them this
// entry point runs the same k_assemble kernel as kvr_assemble but allocates
// nothing: no pool handle, no staging buffers, no cudaMalloc / cudaFree, no
// host heap.  Its scratch -- the device span table, the local-source table and
// the RoPE tables -- lives in one file-scope __device__ array of fixed size
// that every GPU which loads this library holds until the process exits.
#include <cmath>

#include "kvr_internal.cuh"

using namespace kvr;

namespace {

constexpr int kNaMaxSpans = 4096;    // non-empty spans per call
constexpr int kNaMaxLocals = 256;    // request-local sources per call
constexpr int kNaMaxHalf = 64;       // head_dim / 2 (head_dim <= 128)
constexpr int kNaMaxDevices = 64;
constexpr size_t kNaRopeBytes = sizeof(float2) * 2 * kRopeSplit * kNaMaxHalf;   // 4 MiB
constexpr size_t kNaSpanBytes = sizeof(DevSpan) * kNaMaxSpans;                  // 192 KiB
constexpr size_t kNaLocalBytes = sizeof(DevLocal) * kNaMaxLocals;               // 12 KiB
constexpr size_t kNaScratchBytes = kNaRopeBytes + kNaSpanBytes + kNaLocalBytes;

// Per-device state of the scratch: its device address and the RoPE table it
// currently holds.
struct NaDevice {
    void *scratch;
    double theta;
    int head_dim;
    bool have_table;
};

NaDevice g_na_dev[kNaMaxDevices];
DevSpan g_na_spans[kNaMaxSpans];     // host-side tables, built per call
DevLocal g_na_locals[kNaMaxLocals];

// The status, with its reason recorded for kvr_last_error (a fixed
// thread-local buffer: no allocation).
kvr_status na_fail(kvr_status st, const char *why) { return record_error(st, why); }

bool na_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

// The scratch itself.  In host code this name is only a host-side stand-in,
// never a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_kvr_noalloc_scratch[kNaScratchBytes];

extern "C" kvr_status kvr_assemble_noalloc(const kvr_pool_desc *desc, int32_t batch,
                                           const int32_t *span_offsets, const kvr_span *spans,
                                           const kvr_local_src *locals, int32_t n_locals,
                                           const int64_t *cache_offsets, void *cache_k,
                                           void *cache_v, int32_t *pos_ids, int32_t *src_map,
                                           int32_t *prefix_len, uint32_t flags, void *stream)
{
    if (!desc)
        return na_fail(KVR_ERR_INVALID_ARG, "desc is NULL");
    const kvr_pool_desc &d = *desc;
    if (d.dtype != KVR_DTYPE_BF16 && d.dtype != KVR_DTYPE_FP32)
        return na_fail(KVR_ERR_UNSUPPORTED, "dtype");
    if (d.head_dim != 64 && d.head_dim != 128)
        return na_fail(KVR_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (d.n_layers < 1 || d.n_kv_heads < 1 || d.n_q_heads < 1 || d.n_q_heads % d.n_kv_heads ||
        d.n_entries < 1 || d.entry_len < 1 || d.entry_len > kMaxPosition || (d.flags & ~(KVR_POOL_KEYS_UNROTATED | KVR_POOL_ROPE_INTERLEAVED)) != 0 || !d.k ||
        !d.v || !na_aligned16(d.k) || !na_aligned16(d.v) || !(d.rope_theta > 1.0) ||
        !std::isfinite(d.rope_theta))
        return na_fail(KVR_ERR_INVALID_ARG, "invalid pool descriptor");
    const int vec = 16 / (d.dtype == KVR_DTYPE_BF16 ? 2 : 4);
    for (int i = 0; i < 4; ++i)
        if (d.stride[i] < 0 || d.stride[i] % vec)
            return na_fail(KVR_ERR_INVALID_ARG, "pool stride must be >= 0 and a multiple of 16 bytes");
    if (batch < 0)
        return na_fail(KVR_ERR_INVALID_ARG, "batch < 0");
    if (batch == 0)
        return KVR_OK;
    if (flags & ~KVR_POSITIONS_COMPOSITE)
        return na_fail(KVR_ERR_INVALID_ARG, "unknown flags");
    if (!span_offsets || !cache_offsets || span_offsets[0] != 0 || cache_offsets[0] < 0)
        return na_fail(KVR_ERR_INVALID_ARG, "span_offsets / cache_offsets");
    for (int b = 0; b < batch; ++b)
        if (span_offsets[b + 1] < span_offsets[b] || cache_offsets[b + 1] < cache_offsets[b] ||
            cache_offsets[b + 1] - cache_offsets[b] > kMaxPosition)
            return na_fail(KVR_ERR_INVALID_ARG, "offsets must be non-decreasing");
    if (span_offsets[batch] > 0 && !spans)
        return na_fail(KVR_ERR_INVALID_ARG, "spans is NULL");
    if (n_locals < 0 || (n_locals > 0 && !locals))
        return na_fail(KVR_ERR_INVALID_ARG, "locals");
    if (n_locals > kNaMaxLocals)
        return na_fail(KVR_ERR_INVALID_ARG, "more than 256 local sources (the fixed scratch limit)");
    for (int i = 0; i < n_locals; ++i) {
        const kvr_local_src &lc = locals[i];
        if (!lc.k || !lc.v || !na_aligned16(lc.k) || !na_aligned16(lc.v) || lc.len < 0 ||
            lc.len > kMaxPosition)
            return na_fail(KVR_ERR_INVALID_ARG, "local source");
        for (int s = 0; s < 3; ++s)
            if (lc.stride[s] < 0 || lc.stride[s] % vec)
                return na_fail(KVR_ERR_INVALID_ARG, "local source stride");
    }

    // span table (same layout and semantics as kvr_assemble)
    const bool composite = flags & KVR_POSITIONS_COMPOSITE;
    const int LH = d.n_layers * d.n_kv_heads;
    int n = 0;
    int64_t flat = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t cap = cache_offsets[b + 1] - cache_offsets[b];
        int64_t row = 0;
        for (int i = span_offsets[b]; i < span_offsets[b + 1]; ++i) {
            const kvr_span s = spans[i];
            int64_t src_len;
            if (s.src < 0)
                return na_fail(KVR_ERR_OUT_OF_RANGE, "negative source id");
            if (s.src & KVR_SRC_LOCAL) {
                const int idx = s.src & ~KVR_SRC_LOCAL;
                if (idx >= n_locals)
                    return na_fail(KVR_ERR_OUT_OF_RANGE, "unknown local source");
                src_len = locals[idx].len;
            } else {
                if (s.src >= d.n_entries)
                    return na_fail(KVR_ERR_OUT_OF_RANGE, "unknown pool entry");
                src_len = d.entry_len;
            }
            if (s.start < 0 || s.end < s.start || s.end > src_len)
                return na_fail(KVR_ERR_OUT_OF_RANGE, "span outside its source");
            const int32_t len = s.end - s.start;
            const int64_t pos0 = composite ? s.start : row;
            if (pos0 + len > kMaxPosition)
                return na_fail(KVR_ERR_OUT_OF_RANGE, "positions beyond 2^24");
            if (len > 0) {
                if (n == kNaMaxSpans)
                    return na_fail(KVR_ERR_INVALID_ARG, "more than 4096 non-empty spans (the fixed scratch limit)");
                DevSpan &t = g_na_spans[n++];
                t.dst_row0 = cache_offsets[b] * LH;
                t.flat0 = flat;
                t.src = s.src;
                t.start = s.start;
                t.len = len;
                t.row = (int32_t)row;
                t.pos0 = (int32_t)pos0;
                t.delta = (int32_t)(pos0 - s.start);
                t.cap = (int32_t)cap;
                t.dstep = 0;
                if (!(s.src & KVR_SRC_LOCAL) && (d.flags & KVR_POOL_KEYS_UNROTATED)) {
                    t.delta = (int32_t)pos0;   // token t turns by its position pos0 + t
                    t.dstep = 1;
                }
            }
            row += len;
            flat += len;
        }
        if (row > cap)
            return na_fail(KVR_ERR_OUT_OF_RANGE, "prefix longer than its cache block");
    }
    if (prefix_len)   // written only once every request is valid
        for (int b = 0; b < batch; ++b) {
            int64_t row = 0;
            for (int i = span_offsets[b]; i < span_offsets[b + 1]; ++i)
                row += spans[i].end - spans[i].start;
            prefix_len[b] = (int32_t)row;
        }
    if (n == 0)
        return KVR_OK;
    if (!cache_k || !cache_v || !na_aligned16(cache_k) || !na_aligned16(cache_v))
        return na_fail(KVR_ERR_INVALID_ARG, "cache_k / cache_v NULL or not 16-byte aligned");

    // scratch address: once per device, with that device current
    int dev = -1;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess)
        return na_fail(KVR_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kNaMaxDevices)
        return na_fail(KVR_ERR_UNSUPPORTED, "device index beyond 63");
    NaDevice &st = g_na_dev[dev];
    if (!st.scratch) {
        void *ptr = nullptr;
        if ((e = cudaGetSymbolAddress(&ptr, g_kvr_noalloc_scratch)) != cudaSuccess)
            return na_fail(KVR_ERR_CUDA, cudaGetErrorString(e));
        st.scratch = ptr;
    }
    char *base = static_cast<char *>(st.scratch);
    float2 *rope = reinterpret_cast<float2 *>(base);
    DevSpan *dspans = reinterpret_cast<DevSpan *>(base + kNaRopeBytes);
    DevLocal *dlocals = reinterpret_cast<DevLocal *>(base + kNaRopeBytes + kNaSpanBytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // RoPE tables: rebuilt in place only when (theta, head_dim) changes
    if (!st.have_table || st.theta != d.rope_theta || st.head_dim != d.head_dim) {
        if ((e = launch_rope_tables(rope, d.head_dim, d.rope_theta, s)) != cudaSuccess)
            return na_fail(KVR_ERR_CUDA, cudaGetErrorString(e));
        st.have_table = true;
        st.theta = d.rope_theta;
        st.head_dim = d.head_dim;
    }
    for (int i = 0; i < n_locals; ++i)
        g_na_locals[i] = DevLocal{locals[i].k, locals[i].v, locals[i].stride[0], locals[i].stride[1],
                                  locals[i].stride[2], locals[i].len};
    // a small call's tables travel inside the kernel parameters (a stack copy,
    // like kvr_assemble's); a larger call's go up into the scratch from the
    // host tables above
    const bool inl = n <= kInlineEntries && n_locals <= kInlineEntries;
    AssembleTables tab;
    if (inl) {
        for (int i = 0; i < n; ++i)
            tab.spans[i] = g_na_spans[i];
        for (int i = 0; i < n_locals; ++i)
            tab.locals[i] = g_na_locals[i];
    } else if ((e = cudaMemcpyAsync(dspans, g_na_spans, sizeof(DevSpan) * n, cudaMemcpyHostToDevice, s)) !=
                   cudaSuccess ||
               (n_locals > 0 && (e = cudaMemcpyAsync(dlocals, g_na_locals, sizeof(DevLocal) * n_locals,
                                                     cudaMemcpyHostToDevice, s)) != cudaSuccess)) {
        return na_fail(KVR_ERR_CUDA, cudaGetErrorString(e));
    }

    AssembleArgs a{};
    a.spans = dspans;
    a.locals = dlocals;
    a.rope = rope;
    a.pool_k = d.k;
    a.pool_v = d.v;
    a.ps_entry = d.stride[0];
    a.ps_layer = d.stride[1];
    a.ps_head = d.stride[2];
    a.ps_tok = d.stride[3];
    a.cache_k = cache_k;
    a.cache_v = cache_v;
    a.pos_ids = pos_ids;
    a.src_map = src_map;
    a.n_layers = d.n_layers;
    a.n_heads = d.n_kv_heads;
    const int64_t avg = flat / n > 0 ? flat / n : 1;
    a.upc = (int)(256 / avg > LH ? LH : (256 / avg < 1 ? 1 : 256 / avg));
    a.interleaved = (d.flags & KVR_POOL_ROPE_INTERLEAVED) ? 1 : 0;
    if ((e = launch_assemble(a, d.dtype, d.head_dim, n, s, inl ? &tab : nullptr)) != cudaSuccess)
        return na_fail(KVR_ERR_CUDA, cudaGetErrorString(e));
    return KVR_OK;
}
