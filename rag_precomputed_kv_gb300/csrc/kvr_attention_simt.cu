// kvr_attention_simt.cu -- query prefill attention on the CUDA cores.
//
// The path for fp32 pools and for head dims the tensor-core kernel does not
// take.  Same definition as the tensor-core kernel: query token t of request b
// sits at position P_b + t, attends to the P_b stitched prefix rows and to
// query rows 0..t (CoinRAG blog section 2.3, KV_M(q; C_ctx); TurboRAG blog,
// "Attention Mask": the query sees every chunk and itself).
//
// One warp per (layer, query token, query head); each lane holds head_dim/32
// elements (lane + 32k), so a RoPE pair (i, i + D/2) stays inside one lane.
// Scores are reduced across the warp; softmax is online in fp32.
#include <cuda_bf16.h>

#include "kvr_internal.cuh"

namespace kvr {

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T, int D>
__global__ void __launch_bounds__(128)
    k_attention_simt(const __grid_constant__ AttnArgs a, const __grid_constant__ ReqTable rt)
{
    const DevReq *reqs = a.reqs ? a.reqs : rt.reqs;
    constexpr int PL = D / 32;  // elements per lane
    const int64_t w = (int64_t)blockIdx.x * 4 + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int Hq = a.n_q_heads;
    if (w >= (int64_t)a.n_layers * a.total_q * Hq)
        return;
    const int h = (int)(w % Hq);
    const int tok = (int)((w / Hq) % a.total_q);
    const int l = (int)(w / Hq / a.total_q);

    // request owning this token: last b with q_off <= tok and a non-empty range
    int lo = 0, hi = a.n_reqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (reqs[mid].q_off <= tok)
            lo = mid;
        else
            hi = mid - 1;
    }
    while (lo > 0 && reqs[lo].q_len == 0)
        --lo;
    const DevReq rq = reqs[lo];
    const int t = tok - rq.q_off;
    const int pos = rq.prefix + t;
    const int G = Hq / a.n_kv_heads;
    const int kvh = h / G;

    const T *qp = static_cast<const T *>(a.q) + (((int64_t)l * a.total_q + tok) * Hq + h) * D;
    float qv[PL];
#pragma unroll
    for (int k = 0; k < PL; ++k)
        qv[k] = to_f(qp[lane + 32 * k]);
    if (a.interleaved) {
        // pairs (x_2i, x_2i+1): element lane + 32k and its neighbour lane ^ 1
#pragma unroll
        for (int k = 0; k < PL; ++k) {
            const float2 cs = rope_cs(a.rope, D / 2, pos, (lane + 32 * k) >> 1);
            const float other = __shfl_xor_sync(0xffffffffu, qv[k], 1);
            qv[k] = (lane & 1) ? fmaf(other, cs.y, qv[k] * cs.x) : fmaf(qv[k], cs.x, -other * cs.y);
        }
    } else {
#pragma unroll
        for (int k = 0; k < PL / 2; ++k) {
            const float2 cs = rope_cs(a.rope, D / 2, pos, lane + 32 * k);
            const float x = qv[k], y = qv[k + PL / 2];
            qv[k] = fmaf(x, cs.x, -y * cs.y);
            qv[k + PL / 2] = fmaf(x, cs.y, y * cs.x);
        }
    }

    const int64_t blk = rq.cache_row0 + (int64_t)(l * a.n_kv_heads + kvh) * rq.cap;
    const T *kp = static_cast<const T *>(a.cache_k) + blk * D;
    const T *vp = static_cast<const T *>(a.cache_v) + blk * D;
    const int n_vis = pos + 1;
    float m = -INFINITY, lsum = 0.f, acc[PL];
#pragma unroll
    for (int k = 0; k < PL; ++k)
        acc[k] = 0.f;
    for (int j = 0; j < n_vis; ++j) {
        float d = 0.f;
#pragma unroll
        for (int k = 0; k < PL; ++k)
            d = fmaf(qv[k], to_f(kp[(int64_t)j * D + lane + 32 * k]), d);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            d += __shfl_xor_sync(0xffffffffu, d, off);
        const float s = d * a.scale_log2;
        const float mn = fmaxf(m, s);
        const float corr = exp2f(m - mn);
        const float p = exp2f(s - mn);
        lsum = lsum * corr + p;
#pragma unroll
        for (int k = 0; k < PL; ++k)
            acc[k] = fmaf(p, to_f(vp[(int64_t)j * D + lane + 32 * k]), acc[k] * corr);
        m = mn;
    }
    T *op = static_cast<T *>(a.out) + (((int64_t)l * a.total_q + tok) * Hq + h) * D;
    const float inv = 1.f / lsum;
#pragma unroll
    for (int k = 0; k < PL; ++k)
        op[lane + 32 * k] = from_f<T>(acc[k] * inv);
}

cudaError_t launch_attention_simt(const AttnArgs &a, const ReqTable &rt, int dtype, int head_dim,
                                  cudaStream_t s)
{
    const int64_t warps = (int64_t)a.n_layers * a.total_q * a.n_q_heads;
    if (warps == 0)
        return cudaSuccess;
    const int64_t blocks = (warps + 3) / 4;
    if (blocks > 0x7fffffff)
        return cudaErrorInvalidValue;
    if (dtype == KVR_DTYPE_BF16 && head_dim == 128)
        k_attention_simt<__nv_bfloat16, 128><<<(unsigned)blocks, 128, 0, s>>>(a, rt);
    else if (dtype == KVR_DTYPE_BF16 && head_dim == 64)
        k_attention_simt<__nv_bfloat16, 64><<<(unsigned)blocks, 128, 0, s>>>(a, rt);
    else if (dtype == KVR_DTYPE_FP32 && head_dim == 128)
        k_attention_simt<float, 128><<<(unsigned)blocks, 128, 0, s>>>(a, rt);
    else if (dtype == KVR_DTYPE_FP32 && head_dim == 64)
        k_attention_simt<float, 64><<<(unsigned)blocks, 128, 0, s>>>(a, rt);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace kvr
