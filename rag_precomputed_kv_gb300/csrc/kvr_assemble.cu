// kvr_assemble.cu -- RoPE tables and the fused span-gather + RoPE re-rotation
// + stitch kernel.
//
// CoinRAG blog section 2.3: C_ctx = C_p (+) Rot(C_b1[s1:e1]; D1) (+) ...: each
// retrieved span is sliced out of its chunk's precomputed cache, its keys are
// turned to the span's new positions, values are carried over unchanged.
// TurboRAG blog, "Position ID": re-apply RoPE at the reordered positions.
// SemPIC page: the same re-rotation places compiled documents and request-side
// inline tokens at their final logical positions.
//
// The kernel is a pure HBM stream: every stitched (token, layer, kv-head) row
// is read once from the pool and written once into the request's cache.  A
// CTA owns one span and a group of (layer, kv-head) units; inside a unit the
// span's rows are contiguous both in the pool and in the cache, so each warp
// issues 16-byte loads/stores over whole 128-byte lines.
#include <cuda_bf16.h>

#include <algorithm>

#include "kvr_internal.cuh"

namespace kvr {

// ---------------------------------------------------------------------------
// RoPE tables (built once per pool registration)
// ---------------------------------------------------------------------------
__global__ void k_rope_tables(float2 *tab, int half, double theta, int head_dim)
{
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= 2 * kRopeSplit * half)
        return;
    const int i = idx % half;
    const int n = (idx / half) % kRopeSplit;
    const bool hi = idx < kRopeSplit * half;
    const double w = pow(theta, -2.0 * (double)i / (double)head_dim);
    const double ang = (hi ? (double)n * (double)kRopeSplit : (double)n) * w;
    double s, c;
    sincos(ang, &s, &c);
    tab[idx] = make_float2((float)c, (float)s);
}

cudaError_t launch_rope_tables(float2 *tab, int head_dim, double theta, cudaStream_t s)
{
    const int half = head_dim / 2;
    const int n = 2 * kRopeSplit * half;
    k_rope_tables<<<(n + 255) / 256, 256, 0, s>>>(tab, half, theta, head_dim);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// 16-byte vectors of E elements, rotation of a (lo, hi) pair of vectors
// ---------------------------------------------------------------------------
template <typename T>
struct Vec;

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int E = 8;
    __device__ static void rotate(uint4 &lo, uint4 &hi, const float *c, const float *s, bool il)
    {
        if (il)
            rotate_bf16x8_il(lo, hi, c, s);
        else
            rotate_bf16x8(lo, hi, c, s);
    }
};

template <>
struct Vec<float> {
    static constexpr int E = 4;
    __device__ static void rotate(uint4 &lo, uint4 &hi, const float *c, const float *s, bool il)
    {
        float *x = reinterpret_cast<float *>(&lo);
        float *y = reinterpret_cast<float *>(&hi);
        if (il) {
            // pairs (x0, x1), (x2, x3) of lo with c[0], c[1]; of hi with c[2], c[3]
            float *v[2] = {x, y};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const float a0 = v[h][2 * p], a1 = v[h][2 * p + 1];
                    const float cc = c[2 * h + p], ss = s[2 * h + p];
                    v[h][2 * p] = fmaf(a0, cc, -a1 * ss);
                    v[h][2 * p + 1] = fmaf(a0, ss, a1 * cc);
                }
            }
            return;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float xo = fmaf(x[e], c[e], -y[e] * s[e]);
            const float yo = fmaf(x[e], s[e], y[e] * c[e]);
            x[e] = xo;
            y[e] = yo;
        }
    }
};

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_vec(void *p, const uint4 &v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

constexpr int kAssembleThreads = 256;

// One CTA = one span x a group of `upc` (layer, kv-head) units.  A row of the
// span is handled by TPR threads; thread j of a row owns elements
// [j*E, j*E+E) and their RoPE partners [D/2 + j*E, D/2 + j*E + E).
template <typename T, int D>
__device__ __forceinline__ void assemble_body(const AssembleArgs &a, const DevSpan *spans,
                                              const DevLocal *locals, int span_i, int grp, int n_grp)
{
    constexpr int H2 = D / 2;
    constexpr int E = Vec<T>::E;
    constexpr int TPR = H2 / E;                   // threads per row
    constexpr int RPP = kAssembleThreads / TPR;   // rows per pass
    static_assert(H2 % E == 0 && kAssembleThreads % TPR == 0, "head_dim");
    // the per-token (cos, sin) lookup below reads pairs i0 / 2 .. and i1 / 2 ..
    // as 16-byte float4 vectors of two pairs: its pair indices must be even
    static_assert(E % 4 == 0 && H2 % 2 == 0 && (D / 4) % 2 == 0, "16-byte (cos, sin) vector alignment");

    // the next kernel (the query prologue) touches none of this kernel's
    // rows: it may start alongside
    pdl_launch_dependents();
    const DevSpan sp = spans[span_i];
    const int j = threadIdx.x % TPR;

    // this thread's E (cos, sin) pairs for the span's rotation
    float c[E], s[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float2 cs = rope_cs(a.rope, H2, sp.delta, rope_pair(a.interleaved, D, E, j, e));
        c[e] = cs.x;
        s[e] = cs.y;
    }

    const T *kb, *vb;
    int64_t sl, sh, st;
    if (sp.src & KVR_SRC_LOCAL) {
        const DevLocal lc = locals[sp.src & ~KVR_SRC_LOCAL];
        kb = static_cast<const T *>(lc.k);
        vb = static_cast<const T *>(lc.v);
        sl = lc.s_layer;
        sh = lc.s_head;
        st = lc.s_tok;
    } else {
        kb = static_cast<const T *>(a.pool_k) + (int64_t)sp.src * a.ps_entry;
        vb = static_cast<const T *>(a.pool_v) + (int64_t)sp.src * a.ps_entry;
        sl = a.ps_layer;
        sh = a.ps_head;
        st = a.ps_tok;
    }
    T *ck = static_cast<T *>(a.cache_k);
    T *cv = static_cast<T *>(a.cache_v);

    const int lh_end = a.lh_count > 0 ? a.lh_begin + a.lh_count : a.n_layers * a.n_heads;
    // last (layer, kv-head) groups first: what the kernel writes last stays in
    // L2, and the attention kernel that follows starts on the first groups
    const int u0 = a.lh_begin + (n_grp - 1 - grp) * a.upc;
    const int nu = min(a.upc, lh_end - u0);
    const int total = nu * sp.len;

    for (int r0 = threadIdx.x / TPR; r0 < total; r0 += 2 * RPP) {
        uint4 klo[2], khi[2], vlo[2], vhi[2];
        int64_t dst[2];
        bool ok[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int r = r0 + u * RPP;
            ok[u] = r < total;
            if (ok[u]) {
                const int unit = u0 + r / sp.len;
                const int row = r - (r / sp.len) * sp.len;
                const int l = unit / a.n_heads, h = unit - l * a.n_heads;
                const int64_t so = l * sl + h * sh + (int64_t)(sp.start + row) * st + j * E;
                klo[u] = ld_stream(kb + so);
                khi[u] = ld_stream(kb + so + H2);
                if (!a.keys_only) {
                    vlo[u] = ld_stream(vb + so);
                    vhi[u] = ld_stream(vb + so + H2);
                }
                dst[u] = (sp.dst_row0 + (int64_t)unit * sp.cap + sp.row + row) * D + j * E;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (ok[u]) {
                if (sp.dstep) {  // un-rotated source: token t turns by delta + t
                    const int r = r0 + u * RPP;
                    const int row = r - (r / sp.len) * sp.len;
                    const int pos = sp.delta + row;
                    if (pos >= 0 && pos < kRopeSplit) {
                        // the low table row alone (rope_cs below 2^12), its pairs
                        // of this chunk read as 16-byte vectors straight into (c, s)
                        const float4 *lo = reinterpret_cast<const float4 *>(a.rope + (kRopeSplit + pos) * H2);
                        const int i0 = a.interleaved ? (E / 2) * j : E * j;
                        const int i1 = a.interleaved ? D / 4 + (E / 2) * j : E * j + E / 2;
#pragma unroll
                        for (int q = 0; q < E / 4; ++q) {
                            const float4 v0 = __ldg(lo + i0 / 2 + q), v1 = __ldg(lo + i1 / 2 + q);
                            c[2 * q] = v0.x;
                            s[2 * q] = v0.y;
                            c[2 * q + 1] = v0.z;
                            s[2 * q + 1] = v0.w;
                            c[E / 2 + 2 * q] = v1.x;
                            s[E / 2 + 2 * q] = v1.y;
                            c[E / 2 + 2 * q + 1] = v1.z;
                            s[E / 2 + 2 * q + 1] = v1.w;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const float2 cs = rope_cs(a.rope, H2, pos, rope_pair(a.interleaved, D, E, j, e));
                            c[e] = cs.x;
                            s[e] = cs.y;
                        }
                    }
                }
                Vec<T>::rotate(klo[u], khi[u], c, s, a.interleaved);
                st_vec(ck + dst[u], klo[u]);
                st_vec(ck + dst[u] + H2, khi[u]);
                if (!a.keys_only) {
                    st_vec(cv + dst[u], vlo[u]);
                    st_vec(cv + dst[u] + H2, vhi[u]);
                }
            }
        }
    }

    // position ids and source map, written once per span
    if (grp == 0 && a.lh_begin == 0) {
        for (int t = threadIdx.x; t < sp.len; t += kAssembleThreads) {
            if (a.pos_ids)
                a.pos_ids[sp.flat0 + t] = sp.pos0 + t;
            if (a.src_map) {
                a.src_map[2 * (sp.flat0 + t)] = sp.src;
                a.src_map[2 * (sp.flat0 + t) + 1] = sp.start + t;
            }
        }
    }
}

// Tables in global memory (uploaded by the host).
// One CTA per (span, unit group): blockIdx.x, blockIdx.y.
template <typename T, int D>
__global__ void __launch_bounds__(kAssembleThreads) k_assemble(const __grid_constant__ AssembleArgs a)
{
    assemble_body<T, D>(a, a.spans, a.locals, blockIdx.x, blockIdx.y, gridDim.y);
}

// Tables inside the kernel parameters: nothing to upload for small calls.
template <typename T, int D>
__global__ void __launch_bounds__(kAssembleThreads)
    k_assemble_inl(const __grid_constant__ AssembleArgs a, const __grid_constant__ AssembleTables tab)
{
    assemble_body<T, D>(a, tab.spans, tab.locals, blockIdx.x, blockIdx.y, gridDim.y);
}

// A bounded grid (a.max_ctas) whose CTAs take the (span, unit group) pieces
// in turn, leaving the other SMs to a kernel that runs alongside.
template <typename T, int D>
__global__ void __launch_bounds__(kAssembleThreads)
    k_assemble_loop(const __grid_constant__ AssembleArgs a, const __grid_constant__ AssembleTables tab, bool inl)
{
    const DevSpan *spans = inl ? tab.spans : a.spans;
    const DevLocal *locals = inl ? tab.locals : a.locals;
    const int lh_n = a.lh_count > 0 ? a.lh_count : a.n_layers * a.n_heads;
    const int n_grp = (lh_n + a.upc - 1) / a.upc;
    for (int v = blockIdx.x; v < a.n_spans * n_grp; v += gridDim.x)
        assemble_body<T, D>(a, spans, locals, v % a.n_spans, v / a.n_spans, n_grp);
}

template <typename T, int D>
static void launch_one(const AssembleArgs &a, dim3 grid, cudaStream_t s, const AssembleTables *inl)
{
    static const AssembleTables no_tables{};
    if (a.max_ctas > 0)
        k_assemble_loop<T, D><<<grid, kAssembleThreads, 0, s>>>(a, inl ? *inl : no_tables, inl != nullptr);
    else if (inl)
        k_assemble_inl<T, D><<<grid, kAssembleThreads, 0, s>>>(a, *inl);
    else
        k_assemble<T, D><<<grid, kAssembleThreads, 0, s>>>(a);
}

cudaError_t launch_assemble(const AssembleArgs &args, int dtype, int head_dim, int n_spans,
                            cudaStream_t s, const AssembleTables *inl)
{
    if (n_spans == 0)
        return cudaSuccess;
    if (inl && n_spans > kInlineEntries)
        return cudaErrorInvalidValue;
    AssembleArgs a = args;
    a.n_spans = n_spans;
    const int lh_n = a.lh_count > 0 ? a.lh_count : a.n_layers * a.n_heads;
    dim3 grid(n_spans, (lh_n + a.upc - 1) / a.upc);
    if (a.max_ctas > 0)
        grid = dim3((unsigned)std::min<int64_t>((int64_t)grid.x * grid.y, a.max_ctas), 1);
    if (dtype == KVR_DTYPE_BF16 && head_dim == 128)
        launch_one<__nv_bfloat16, 128>(a, grid, s, inl);
    else if (dtype == KVR_DTYPE_BF16 && head_dim == 64)
        launch_one<__nv_bfloat16, 64>(a, grid, s, inl);
    else if (dtype == KVR_DTYPE_FP32 && head_dim == 128)
        launch_one<float, 128>(a, grid, s, inl);
    else if (dtype == KVR_DTYPE_FP32 && head_dim == 64)
        launch_one<float, 64>(a, grid, s, inl);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace kvr
