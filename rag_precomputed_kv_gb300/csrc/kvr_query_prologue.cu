// kvr_query_prologue.cu -- the query side of the prefill, before attention.
//
// CoinRAG blog section 2.3: the query is the only part computed online,
// KV_M(q; C_ctx), on top of the stitched prefix.  Query token t of request b
// sits at position P_b + t (reordered, contiguous positions: TurboRAG blog,
// "Position ID").  For every (request, layer, kv-head) this kernel
//   * rotates the token's key by P_b + t and appends it, with its value, at
//     row P_b + t of the cache block (so attention sees it like a prefix row);
//   * rotates the G query heads of that kv head by the same angles and writes
//     them packed as [layer][kv-head][token][G][head_dim] -- the 128-row tiles
//     the tensor-core attention kernel loads with TMA are then contiguous;
//   * zeroes spare V rows up to the end of the block's last 128-key tile.
// Memory-bound: each query-side row is read once and written once.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kQpTokens = 16;                 // query tokens per CTA
constexpr int kQpThreads = 8 * kQpTokens;     // 8 threads per token

__device__ __forceinline__ void rotate8(uint4 &lo, uint4 &hi, const float *c, const float *s, bool il)
{
    if (il) {
        rotate_bf16x8_il(lo, hi, c, s);
        return;
    }
    uint32_t *pl = reinterpret_cast<uint32_t *>(&lo);
    uint32_t *ph = reinterpret_cast<uint32_t *>(&hi);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&pl[w]));
        const float2 y = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&ph[w]));
        const float c0 = c[2 * w], s0 = s[2 * w], c1 = c[2 * w + 1], s1 = s[2 * w + 1];
        __nv_bfloat162 xo = __floats2bfloat162_rn(fmaf(x.x, c0, -y.x * s0), fmaf(x.y, c1, -y.y * s1));
        __nv_bfloat162 yo = __floats2bfloat162_rn(fmaf(x.x, s0, y.x * c0), fmaf(x.y, s1, y.y * c1));
        pl[w] = *reinterpret_cast<uint32_t *>(&xo);
        ph[w] = *reinterpret_cast<uint32_t *>(&yo);
    }
}

}  // namespace

// Work item = (request, 16-token chunk of its query, layer, kv-head); a
// grid-stride loop over the items (the grid fills the SMs once, so that when
// the kernel runs alongside the assemble kernel its resident CTAs keep
// working).  8 threads per token, thread j owns elements [8j, 8j+8) and
// their RoPE partners [64 + 8j, ...).
__global__ void __launch_bounds__(kQpThreads)
    k_query_prologue(const __grid_constant__ QueryPrologueArgs a, const __grid_constant__ ReqTable rt)
{
    constexpr int D = 128, H2 = 64, E = 8, TPR = 8, RPP = kQpThreads / TPR;
    const DevReq *reqs = a.reqs ? a.reqs : rt.reqs;
    const int n_chunks = (a.max_q_len + kQpTokens - 1) / kQpTokens;
    const int64_t n_rc = (int64_t)a.n_reqs * n_chunks;
    const int64_t n_items = n_rc * a.n_layers * a.n_kv_heads;
    const int G = a.n_q_heads / a.n_kv_heads;
    const int j = threadIdx.x % TPR;
    const int64_t T = a.total_q;
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *kq = static_cast<const __nv_bfloat16 *>(a.kq);
    const __nv_bfloat16 *vq = static_cast<const __nv_bfloat16 *>(a.vq);
    __nv_bfloat16 *ck = static_cast<__nv_bfloat16 *>(a.cache_k);
    __nv_bfloat16 *cv = static_cast<__nv_bfloat16 *>(a.cache_v);
    __nv_bfloat16 *qr = static_cast<__nv_bfloat16 *>(a.q_rot);
    for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int64_t rc = it % n_rc;
        const int lh = (int)(it / n_rc);
        const int chunk = (int)(rc % n_chunks);
        const DevReq rq = reqs[rc / n_chunks];
        const int t_end = min(rq.q_len, (chunk + 1) * kQpTokens);
        const int l = lh / a.n_kv_heads, h = lh - l * a.n_kv_heads;
        for (int t = chunk * kQpTokens + threadIdx.x / TPR; t < t_end; t += RPP) {
            const int64_t tok = rq.q_off + t;
            float c[E], s[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float2 cs = rope_cs(a.rope, H2, rq.prefix + t, rope_pair(a.interleaved, D, E, j, e));
                c[e] = cs.x;
                s[e] = cs.y;
            }
            const int64_t kv_src = ((l * T + tok) * a.n_kv_heads + h) * D + j * E;
            uint4 klo = *reinterpret_cast<const uint4 *>(kq + kv_src);
            uint4 khi = *reinterpret_cast<const uint4 *>(kq + kv_src + H2);
            const uint4 vlo = *reinterpret_cast<const uint4 *>(vq + kv_src);
            const uint4 vhi = *reinterpret_cast<const uint4 *>(vq + kv_src + H2);
            rotate8(klo, khi, c, s, a.interleaved);
            const int64_t dst = (rq.cache_row0 + (int64_t)lh * rq.cap + rq.prefix + t) * D + j * E;
            *reinterpret_cast<uint4 *>(ck + dst) = klo;
            *reinterpret_cast<uint4 *>(ck + dst + H2) = khi;
            *reinterpret_cast<uint4 *>(cv + dst) = vlo;
            *reinterpret_cast<uint4 *>(cv + dst + H2) = vhi;
            const int64_t q_src = ((l * T + tok) * a.n_q_heads + (int64_t)h * G) * D + j * E;
            const int64_t q_dst = (((int64_t)lh * T + tok) * G) * D + j * E;
            for (int g = 0; g < G; ++g) {
                uint4 lo = *reinterpret_cast<const uint4 *>(q + q_src + (int64_t)g * D);
                uint4 hi = *reinterpret_cast<const uint4 *>(q + q_src + (int64_t)g * D + H2);
                rotate8(lo, hi, c, s, a.interleaved);
                *reinterpret_cast<uint4 *>(qr + q_dst + (int64_t)g * D) = lo;
                *reinterpret_cast<uint4 *>(qr + q_dst + (int64_t)g * D + H2) = hi;
            }
        }
        // V rows between the block's data and the end of its last 128-row
        // key tile (present only when the block has spare capacity) are
        // zeroed, so that the attention kernel's masked keys (p = 0) never
        // meet a non-finite value; rows past the block belong to the next,
        // assembled, block.
        const int n_valid = rq.prefix + rq.q_len;
        const int pad_end = chunk == 0 ? min(rq.cap, (n_valid + 127) / 128 * 128) : 0;
        for (int row = n_valid + threadIdx.x / TPR; row < pad_end; row += RPP) {
            const int64_t dst = (rq.cache_row0 + (int64_t)lh * rq.cap + row) * D + j * E;
            *reinterpret_cast<uint4 *>(cv + dst) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(cv + dst + H2) = make_uint4(0, 0, 0, 0);
        }
    }
    // Launched after the assemble kernel of the same prefill, this grid may
    // run alongside it (the assemble kernel writes only prefix rows); it
    // completes only after that kernel has, so the attention kernel's wait on
    // this grid covers the stitched prefix too.  Without a programmatic
    // launch the wait returns at once.
    pdl_wait_prerequisites();
    pdl_launch_dependents();
}

cudaError_t launch_query_prologue(const QueryPrologueArgs &a, const ReqTable &rt, int n_sms, bool pdl,
                                  cudaStream_t s)
{
    const int64_t n_chunks = (a.max_q_len + kQpTokens - 1) / kQpTokens;
    const int64_t n_items = (int64_t)a.n_reqs * n_chunks * a.n_layers * a.n_kv_heads;
    if (n_items == 0)
        return cudaSuccess;
    // one wave: the resident CTAs per SM (registers decide) times the SMs
    static std::atomic<int> per_sm[64] = {};   // per device (host threads may race: same value)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    int occ = dev < 64 ? per_sm[dev].load(std::memory_order_relaxed) : 0;
    if (occ == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_query_prologue, kQpThreads, 0);
        if (e != cudaSuccess)
            return e;
        occ = std::max(occ, 1);
        if (dev < 64)
            per_sm[dev].store(occ, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(n_items, (int64_t)n_sms * occ));
    cfg.blockDim = dim3(kQpThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_query_prologue, a, rt);
}

}  // namespace kvr
