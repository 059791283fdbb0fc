// kvr_decode.cu -- attention of a decode step over the stitched cache.
//
// CoinRAG blog section 2.3: after the query prefill the model decodes
// normally on top of KV_CoinRAG; each step appends one token at the next
// row and position P_b of every cache block and attends to rows 0..P_b.  For
// every (request, layer, kv-head) this kernel rotates the step's key by P_b
// and appends it and its value at row P_b (TurboRAG blog, "Position ID":
// contiguous positions), rotates the G query heads of the kv head by P_b, and
// computes
//     o_g = sum_j softmax_j(q_g . k_j * scale) v_j,  j <= P_b,
// all in one pass over the block.
//
// A decode step reads the whole cache block once and does only G (<= 16)
// rows of arithmetic per key: it is bound by HBM, not by the tensor cores.
// So the kernel streams: one CTA per (request, layer, kv-head), a three-stage
// ring of 128-key K and V tiles loaded by TMA (128B-swizzled 64-column
// panels, the tensor maps of the prefill attention), and four warps that each
// take 32 keys of a tile.  The G x 128 by 128 x 32 products are register-
// resident warp MMAs (mma.sync m16n8k16, the G heads padded to 16 rows): at
// 16 rows a tcgen05 MMA would round-trip every tile through TMEM for no
// throughput the step can use.  Each warp keeps an online softmax in registers
// (the score fragment of one MMA is the P operand of the next); at the end the
// four warps' states are combined in shared memory in a fixed order.
//
// The appended row reaches the computation through the kernel itself: the
// warp whose keys hold row P_b writes it into the last shared-memory tile
// (whatever the tile's copy read from memory), and every warp zeroes the V
// rows of that tile past P_b, so that masked keys (p = 0) never meet a
// non-finite value.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>

#include "kvr_decode_common.cuh"

namespace kvr {

namespace {

using namespace dec;

constexpr int kDecOffBar = kDecStages * kDecStageBytes;
constexpr int kDecNumBars = 2 * kDecStages;         // full[s], empty[s]
constexpr int kDecOffErr = kDecOffBar + 8 * kDecNumBars;
constexpr int kDecSmem = kDecOffErr + 16 + 1024;    // + alignment slack
// the four warps' final states over stage 0 of the ring
static_assert(kDecMergeBytes <= kDecStageBytes, "merge area");

}  // namespace

__global__ void __launch_bounds__(kDecThreads, 1)
    k_decode_attention(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ AttnArgs a, const __grid_constant__ ReqTable rt,
                       const __grid_constant__ DecodeIO io)
{
    extern __shared__ uint8_t dec_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dec_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = dec_smem_u32(smem);
    auto full = [&](int s) { return sbase + kDecOffBar + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return sbase + kDecOffBar + 8u * (uint32_t)(kDecStages + s); };
    volatile int *cta_err = reinterpret_cast<volatile int *>(smem + kDecOffErr);

    const DevReq *reqs = a.reqs ? a.reqs : rt.reqs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = (int)(blockIdx.x % (unsigned)a.n_reqs);
    const int lh = (int)(blockIdx.x / (unsigned)a.n_reqs);
    const int G = a.n_q_heads / a.n_kv_heads;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            dec_mbar_init(full(s), 1);
            dec_mbar_init(empty(s), kDecThreads);
        }
        *cta_err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x == 32) {   // descriptors only: nothing the previous kernel writes
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    __syncthreads();
    // a decode step launched after this one (programmatic launch) may now take
    // the SMs this grid leaves free and set up there: it reads and writes
    // nothing before its own wait below, which returns once this grid is done
    pdl_launch_dependents();
    // nothing the kernel before it on the stream writes (the step's query,
    // key and value, the cache rows, the request table) is read before this
    pdl_wait_prerequisites();

    const DevReq rq = reqs[b];
    if (rq.q_len == 0)
        return;   // uniform over the CTA: no barrier is waited on
    const int n_valid = rq.prefix + rq.q_len;
    const int n_t = (n_valid + kDecTile - 1) / kDecTile;
    const int64_t kv_row0 = rq.cache_row0 + (int64_t)lh * rq.cap;

    // producer: thread 0 keeps the ring kDecStages tiles ahead
    auto issue = [&](int j) {
        const int s = j % kDecStages;
        const uint32_t dst = sbase + (uint32_t)(s * kDecStageBytes);
        const int row = (int)(kv_row0 + (int64_t)j * kDecTile);
        dec_expect_tx(full(s), kDecStageBytes);
        dec_tma_load(dst, &tmk, 0, row, full(s));
        dec_tma_load(dst + kDecPanel, &tmk, 64, row, full(s));
        dec_tma_load(dst + kDecTileBytes, &tmv, 0, row, full(s));
        dec_tma_load(dst + kDecTileBytes + kDecPanel, &tmv, 64, row, full(s));
    };
    int n_issued = 0;   // thread 0
    if (threadIdx.x == 0)
        for (; n_issued < n_t && n_issued < kDecStages; ++n_issued)
            issue(n_issued);

    const int P = rq.prefix;   // the step's row and position
    const int l_idx = lh / a.n_kv_heads, h_idx = lh - l_idx * a.n_kv_heads;
    const int64_t tok = (int64_t)l_idx * a.total_q + rq.q_off;
    const bool il = io.interleaved != 0;
    auto rot = [](float &x, float &y, float2 cs) {
        const float xo = fmaf(x, cs.x, -(y * cs.y));
        y = fmaf(x, cs.y, y * cs.x);
        x = xo;
    };
    auto unpk = [](uint32_t u, float &lo, float &hi) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
        lo = f.x;
        hi = f.y;
    };

    // the step's key (rotated by P) and value: lane l holds RoPE pairs 2l and
    // 2l + 1, i.e. elements (2l, 2l + 1) and (64 + 2l, 65 + 2l), or (4l .. 4l + 3)
    // with adjacent pairs; the warp whose keys hold row P appends them
    const int w_new = (P & (kDecTile - 1)) >> 5;
    uint32_t kn[2] = {0u, 0u}, vn[2] = {0u, 0u};
    const int d_a = il ? 4 * lane : 2 * lane, d_b = il ? 4 * lane + 2 : 64 + 2 * lane;
    if (warp == w_new) {
        const int64_t src = (tok * a.n_kv_heads + h_idx) * kDecD;
        const __nv_bfloat16 *kq = static_cast<const __nv_bfloat16 *>(io.kq) + src;
        const __nv_bfloat16 *vq = static_cast<const __nv_bfloat16 *>(io.vq) + src;
        kn[0] = *reinterpret_cast<const uint32_t *>(kq + d_a);
        kn[1] = *reinterpret_cast<const uint32_t *>(kq + d_b);
        vn[0] = *reinterpret_cast<const uint32_t *>(vq + d_a);
        vn[1] = *reinterpret_cast<const uint32_t *>(vq + d_b);
        float x0, x1, y0, y1;
        unpk(kn[0], x0, x1);
        unpk(kn[1], y0, y1);
        const float2 c0 = rope_cs(a.rope, kDecD / 2, P, 2 * lane), c1 = rope_cs(a.rope, kDecD / 2, P, 2 * lane + 1);
        if (il) {   // pairs (x0, x1) and (y0, y1)
            rot(x0, x1, c0);
            rot(y0, y1, c1);
        } else {    // pairs (x0, y0) and (x1, y1)
            rot(x0, y0, c0);
            rot(x1, y1, c1);
        }
        kn[0] = pack2(x0, x1);
        kn[1] = pack2(y0, y1);
        __nv_bfloat16 *ck = static_cast<__nv_bfloat16 *>(io.cache_k) + (kv_row0 + P) * kDecD;
        __nv_bfloat16 *cv = static_cast<__nv_bfloat16 *>(io.cache_v) + (kv_row0 + P) * kDecD;
        *reinterpret_cast<uint32_t *>(ck + d_a) = kn[0];
        *reinterpret_cast<uint32_t *>(ck + d_b) = kn[1];
        *reinterpret_cast<uint32_t *>(cv + d_a) = vn[0];
        *reinterpret_cast<uint32_t *>(cv + d_b) = vn[1];
    }

    // Q fragments (A operand, 16 x 128, rows >= G zero), rotated by P: rows
    // lane/4 and lane/4 + 8, elements kb*16 + cq + {0, 1} and + 8 + {0, 1}
    const __nv_bfloat16 *qp = static_cast<const __nv_bfloat16 *>(a.q) + (tok * a.n_q_heads + h_idx * G) * kDecD;
    const int r0 = lane >> 2, r1 = r0 + 8, cq = (lane & 3) * 2;
    uint32_t qa[8][4];
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
        const int c0 = kb * 16 + cq;
        auto ld2 = [&](int r, int c) -> uint32_t {
            return r < G ? *reinterpret_cast<const uint32_t *>(qp + (int64_t)r * kDecD + c) : 0u;
        };
        qa[kb][0] = ld2(r0, c0);
        qa[kb][1] = ld2(r1, c0);
        qa[kb][2] = ld2(r0, c0 + 8);
        qa[kb][3] = ld2(r1, c0 + 8);
    }
    if (il) {   // the two elements of each register are a pair
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int d = kb * 16 + cq + ((i & 2) ? 8 : 0);
                const float2 cs = rope_cs(a.rope, kDecD / 2, P, d >> 1);
                float x, y;
                unpk(qa[kb][i], x, y);
                rot(x, y, cs);
                qa[kb][i] = pack2(x, y);
            }
        }
    } else {    // element d pairs with d + 64: register i of block kb with that of block kb + 4
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int d = kb * 16 + cq + ((i & 2) ? 8 : 0);
                const float2 cs0 = rope_cs(a.rope, kDecD / 2, P, d), cs1 = rope_cs(a.rope, kDecD / 2, P, d + 1);
                float x0, x1, y0, y1;
                unpk(qa[kb][i], x0, x1);
                unpk(qa[kb + 4][i], y0, y1);
                rot(x0, y0, cs0);
                rot(x1, y1, cs1);
                qa[kb][i] = pack2(x0, x1);
                qa[kb + 4][i] = pack2(y0, y1);
            }
        }
    }

    const float sc = a.scale_log2;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    bool ok = true;
    for (int j = 0; j < n_t; ++j) {
        const int s = j % kDecStages;
        if (!dec_wait(full(s), (uint32_t)((j / kDecStages) & 1))) {
            ok = false;
            break;
        }
        const uint32_t kt = sbase + (uint32_t)(s * kDecStageBytes), vt = kt + kDecTileBytes;
        const int key0 = 32 * warp;   // this warp's 32 keys of the tile
        if (j == n_t - 1) {
            // V rows past P are zero; row P is the step's own key and value
            for (int idx = lane; idx < 32 * 16; idx += 32) {
                const int row = key0 + (idx >> 4);
                if (j * kDecTile + row > P) {
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vt + sw_off(row, idx & 15)), "r"(0u)
                                 : "memory");
                }
            }
            if (warp == w_new) {
                const int row = P & (kDecTile - 1);
                auto put = [&](uint32_t tile, int d, uint32_t v) {
                    const uint32_t addr = tile + sw_off(row, d >> 3) + (uint32_t)((d & 7) * 2);
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
                };
                put(kt, d_a, kn[0]);
                put(kt, d_b, kn[1]);
                put(vt, d_a, vn[0]);
                put(vt, d_b, vn[1]);
            }
            __syncwarp();
        }
        // S = Q K^T for 32 keys: four 8-key column blocks
        float c[4][4];
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
            c[nb][0] = c[nb][1] = c[nb][2] = c[nb][3] = 0.f;
#pragma unroll
        for (int nb = 0; nb < 4; nb += 2) {
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
                // matrices: (nb, kb lo), (nb, kb hi), (nb+1, kb lo), (nb+1, kb hi)
                const int mi = lane >> 3;
                const int key = key0 + 8 * (nb + (mi >> 1)) + (lane & 7);
                const int chunk = 2 * kb + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kt + sw_off(key, chunk), b0, b1, b2, b3);
                mma_bf16(c[nb], qa[kb], b0, b1);
                mma_bf16(c[nb + 1], qa[kb], b2, b3);
            }
        }
        // scale to log2 units, mask keys >= n_valid, row maxima over the quad
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kk = j * kDecTile + key0 + 8 * nb + cq + (e & 1);
                c[nb][e] = kk < n_valid ? c[nb][e] * sc : -INFINITY;
                mx[e >> 1] = fmaxf(mx[e >> 1], c[nb][e]);
            }
        }
        float corr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            const float m_new = fmaxf(m_run[h], mx[h]);
            // a row that has seen no key yet keeps m = -inf and p = 0
            corr[h] = m_new == -INFINITY ? 1.f : dec_ex2(m_run[h] - m_new);
            m_run[h] = m_new;
        }
        const float nm[2] = {m_run[0] == -INFINITY ? 0.f : -m_run[0], m_run[1] == -INFINITY ? 0.f : -m_run[1]};
        float sum[2] = {0.f, 0.f};
        uint32_t pa[2][4];   // P as the A operand of two 16-key blocks
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
            const float p0 = dec_ex2(c[nb][0] + nm[0]), p1 = dec_ex2(c[nb][1] + nm[0]);
            const float p2 = dec_ex2(c[nb][2] + nm[1]), p3 = dec_ex2(c[nb][3] + nm[1]);
            sum[0] += p0 + p1;
            sum[1] += p2 + p3;
            pa[nb >> 1][(nb & 1) * 2 + 0] = pack2(p0, p1);
            pa[nb >> 1][(nb & 1) * 2 + 1] = pack2(p2, p3);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 1);
            sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 2);
            l_run[h] = l_run[h] * corr[h] + sum[h];
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            o[n][0] *= corr[0];
            o[n][1] *= corr[0];
            o[n][2] *= corr[1];
            o[n][3] *= corr[1];
        }
        // O += P V over the warp's 32 keys: two 16-key blocks x sixteen 8-column blocks
#pragma unroll
        for (int kb2 = 0; kb2 < 2; ++kb2) {
#pragma unroll
            for (int n = 0; n < 16; n += 2) {
                // matrices: (keys lo, n), (keys hi, n), (keys lo, n+1), (keys hi, n+1)
                const int mi = lane >> 3;
                const int key = key0 + 16 * kb2 + 8 * (mi & 1) + (lane & 7);
                const int chunk = n + (mi >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vt + sw_off(key, chunk), b0, b1, b2, b3);
                mma_bf16(o[n], pa[kb2], b0, b1);
                mma_bf16(o[n + 1], pa[kb2], b2, b3);
            }
        }
        // this stage is consumed; thread 0 refills it kDecStages tiles ahead
        dec_mbar_arrive(empty(s));
        if (threadIdx.x == 0 && j + kDecStages < n_t) {
            if (!dec_wait(empty(s), (uint32_t)((j / kDecStages) & 1))) {
                ok = false;
                break;
            }
            issue(j + kDecStages);
            ++n_issued;
        }
    }
    if (!ok)
        *cta_err = 1;
    __syncthreads();
    if (*cta_err) {
        if (threadIdx.x == 0 && a.err)
            atomicCAS(a.err, kDevOk, kDevTimeout);
        // copies in flight land before the CTA leaves (bounded)
        if (threadIdx.x == 0)
            for (int j = n_issued > kDecStages ? n_issued - kDecStages : 0; j < n_issued; ++j)
                dec_wait(full(j % kDecStages), (uint32_t)((j / kDecStages) & 1));
        return;
    }

    // combine the four warps' states (fixed order) over stage 0 of the ring
    float *mm = reinterpret_cast<float *>(smem);          // [4][16]
    float *ll = mm + 4 * 16;                              // [4][16]
    float *oo = ll + 4 * 16;                              // [4][16][128]
    if ((lane & 3) == 0) {
        mm[warp * 16 + r0] = m_run[0];
        mm[warp * 16 + r1] = m_run[1];
        ll[warp * 16 + r0] = l_run[0];
        ll[warp * 16 + r1] = l_run[1];
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int col = 8 * n + cq;
        *reinterpret_cast<float2 *>(oo + (warp * 16 + r0) * kDecD + col) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2 *>(oo + (warp * 16 + r1) * kDecD + col) = make_float2(o[n][2], o[n][3]);
    }
    __syncthreads();
    // thread t: row t / 8 (the G valid rows), columns 16 (t % 8) .. +15
    for (int rr = threadIdx.x >> 3; rr < G; rr += kDecThreads / 8) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w)
            M = fmaxf(M, mm[w * 16 + rr]);
        float wgt[4], L = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float mw = mm[w * 16 + rr];
            wgt[w] = mw == -INFINITY ? 0.f : dec_ex2(mw - M);
            L += ll[w * 16 + rr] * wgt[w];
        }
        const float inv = 1.f / L;
        // a NaN or infinity among the row's query or key elements leaves no
        // finite positive denominator: report it (the row is written as computed)
        if (!(L > 0.f && L < INFINITY) && (threadIdx.x & 7) == 0 && a.err)
            atomicCAS(a.err, kDevOk, kDevBadInput);
        const int c0 = 16 * (threadIdx.x & 7);
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                v0 += oo[(w * 16 + rr) * kDecD + c0 + e] * wgt[w];
                v1 += oo[(w * 16 + rr) * kDecD + c0 + e + 1] * wgt[w];
            }
            pk[e >> 1] = pack2(v0 * inv, v1 * inv);
        }
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                             (((int64_t)l_idx * a.total_q + rq.q_off) * a.n_q_heads + h_idx * G + rr) * kDecD + c0;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
}

bool decode_supported(int dtype, int head_dim, int group) { return dtype == KVR_DTYPE_BF16 && head_dim == kDecD && group <= 16; }

cudaError_t launch_decode_attention(const AttnArgs &a, const ReqTable &rt, const void *tmap_k, const void *tmap_v,
                                    const DecodeIO &io, bool pdl, cudaStream_t s)
{
    const int64_t ctas = (int64_t)a.n_reqs * a.n_layers * a.n_kv_heads;
    if (ctas == 0)
        return cudaSuccess;
    if (ctas > 0x7fffffff)
        return cudaErrorInvalidValue;
    static std::atomic<bool> attr_set[64] = {};   // per device (host threads may race: same value)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k_decode_attention, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            attr_set[dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = kDecSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_decode_attention, *static_cast<const CUtensorMap *>(tmap_k),
                              *static_cast<const CUtensorMap *>(tmap_v), a, rt, io);
}

}  // namespace kvr
