// kvr_decode_stream.cu -- a decode step over few cache blocks, spread over
// every SM.
//
// The same step as k_decode_attention (CoinRAG blog section 2.3: decoding
// continues on top of the stitched cache; each step appends one token at row
// and position P_b and attends to rows 0..P_b): rotate the step's key and
// query heads by P_b, append the key and value, and stream the block once.
// With one CTA per (request, layer, kv-head) a small batch leaves SMs idle
// (batch 1 of a 28-layer, 4-kv-head model: 112 blocks on 152 SMs), so here a
// persistent grid of one CTA per SM takes equal, contiguous shares of all the
// blocks' 128-key tiles (the tiles of request b, kv block lh, in request-major
// order).  A CTA streams its share through one three-stage TMA ring without a
// break at block boundaries.  A block whose tiles fall to one CTA is finished
// there; a block split between CTAs (at most the first and the last block of
// each share) leaves each part's combined state -- running max m, sum l and
// unnormalised O for its G rows -- in a per-CTA workspace slot, and the CTA
// that completes the block's arrival count merges the parts in part order (a
// fixed rounding order, whichever CTA finishes last) and writes the output.
// No CTA ever waits for another.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>

#include "kvr_decode_common.cuh"

namespace kvr {

namespace {

using namespace dec;

// shared memory: ring of kDecStages (K tile, V tile) stages, the four warps'
// states for a segment's combine, barriers, flags
constexpr int kDsOffMerge = kDecStages * kDecStageBytes;
constexpr int kDsOffBar = kDsOffMerge + kDecMergeBytes;
constexpr int kDsNumBars = 2 * kDecStages;
constexpr int kDsOffFlags = kDsOffBar + 8 * kDsNumBars;   // [0] error, [1] merger
constexpr int kDsSmem = kDsOffFlags + 16 + 1024;          // + alignment slack
static_assert(kDsSmem <= 227 * 1024, "shared memory budget");

// A workspace slot: m[16], l[16], O[16][128] fp32.
constexpr int kPartFloats = 16 + 16 + 16 * kDecD;

__device__ __forceinline__ int64_t share_start(int c, int n_cta, int64_t total)
{
    return (int64_t)c * total / n_cta;
}

// Workspace slot of a block's part computed by the CTA whose share starts at
// `share0` (a CTA holds at most two partial blocks: the one it starts inside,
// slot 1, and the one it ends inside, slot 0, or a single one).
__device__ __forceinline__ int part_slot(int64_t blk_g0, int64_t share0) { return blk_g0 >= share0 ? 0 : 1; }

// The CTA whose share holds tile g.
__device__ __forceinline__ int share_of(int64_t g, int n_cta, int64_t total)
{
    return (int)(((g + 1) * n_cta - 1) / total);
}

// Tiles of request r's blocks (the step's row P is the last key).
__device__ __forceinline__ int req_tiles(const DevReq &r)
{
    return r.q_len > 0 ? (r.prefix + 1 + kDecTile - 1) / kDecTile : 0;
}

// A position in the step's tile sequence, with the request fields its tiles
// need held in registers: the request table (kernel parameters or global
// memory, whose lines the K/V stream evicts) is read once per request, not
// once per tile.
struct TileCursor {
    int b, lh, j, n_t;
    int prefix, cap, q_off;
    int64_t cache_row0;

    __device__ __forceinline__ void load_req(const DevReq *reqs, int bb)
    {
        const DevReq r = reqs[bb];
        b = bb;
        n_t = req_tiles(r);
        prefix = r.prefix;
        cap = r.cap;
        q_off = r.q_off;
        cache_row0 = r.cache_row0;
    }
    // tile g: the last request (table order) whose first tile is <= g
    __device__ __forceinline__ void seek(const DevReq *reqs, int n_reqs, int64_t g)
    {
        int lo = 0, hi = n_reqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (reqs[mid].tile0 <= g)
                lo = mid;
            else
                hi = mid - 1;
        }
        load_req(reqs, lo);
        const int64_t rel = g - reqs[lo].tile0;
        lh = (int)(rel / n_t);
        j = (int)(rel - (int64_t)lh * n_t);
    }
    // the next tile (within the step's sequence: requests without a token
    // have no tiles and come last)
    __device__ __forceinline__ void next(const DevReq *reqs, int LH)
    {
        if (++j < n_t)
            return;
        j = 0;
        if (++lh < LH)
            return;
        lh = 0;
        load_req(reqs, b + 1);
    }
};

}  // namespace

__global__ void __launch_bounds__(kDecThreads, 1)
    k_decode_stream(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ AttnArgs a, const __grid_constant__ ReqTable rt,
                    const __grid_constant__ DecodeIO io, const __grid_constant__ DecodeStream ds)
{
    extern __shared__ uint8_t ds_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(ds_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = dec_smem_u32(smem);
    auto full = [&](int s) { return sbase + kDsOffBar + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return sbase + kDsOffBar + 8u * (uint32_t)(kDecStages + s); };
    volatile int *flags = reinterpret_cast<volatile int *>(smem + kDsOffFlags);

    const DevReq *reqs = a.reqs ? a.reqs : rt.reqs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.n_q_heads / a.n_kv_heads;
    const int c = blockIdx.x;
    const int64_t g0 = share_start(c, ds.n_cta, ds.total), g1 = share_start(c + 1, ds.n_cta, ds.total);
    if (g0 >= g1)
        return;   // uniform over the CTA: no barrier is waited on

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            dec_mbar_init(full(s), 1);
            dec_mbar_init(empty(s), kDecThreads);
        }
        flags[0] = 0;
        flags[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x == 32) {   // descriptors only: nothing the previous kernel writes
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    __syncthreads();
    // the cache rows of earlier steps and the caller's inputs are read from here on
    pdl_wait_prerequisites();

    // producer: thread 0 keeps the ring kDecStages tiles ahead of the share
    const int n_mine = (int)(g1 - g0);
    TileCursor pc;   // thread 0: the next tile to load
    if (threadIdx.x == 0)
        pc.seek(reqs, a.n_reqs, g0);
    auto issue = [&](int i) {
        const int s = i % kDecStages;
        const uint32_t dst = sbase + (uint32_t)(s * kDecStageBytes);
        const int row = (int)(pc.cache_row0 + (int64_t)pc.lh * pc.cap + (int64_t)pc.j * kDecTile);
        if (i + 1 < n_mine)
            pc.next(reqs, ds.LH);
        dec_expect_tx(full(s), kDecStageBytes);
        dec_tma_load(dst, &tmk, 0, row, full(s));
        dec_tma_load(dst + kDecPanel, &tmk, 64, row, full(s));
        dec_tma_load(dst + kDecTileBytes, &tmv, 0, row, full(s));
        dec_tma_load(dst + kDecTileBytes + kDecPanel, &tmv, 64, row, full(s));
    };
    int n_issued = 0;   // thread 0
    if (threadIdx.x == 0)
        for (; n_issued < n_mine && n_issued < kDecStages; ++n_issued)
            issue(n_issued);

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
    const int r0 = lane >> 2, r1 = r0 + 8, cq = (lane & 3) * 2;
    const int d_a = il ? 4 * lane : 2 * lane, d_b = il ? 4 * lane + 2 : 64 + 2 * lane;
    const float sc = a.scale_log2;
    float *mm = reinterpret_cast<float *>(smem + kDsOffMerge);   // [4][16]
    float *ll = mm + 4 * 16;                                      // [4][16]
    float *oo = ll + 4 * 16;                                      // [4][16][128]

    // state of the current segment (the share's tiles of one block)
    int b = -1, lh = 0, n_t = 0, P = 0, n_valid = 0, w_new = 0, seg_j0 = 0;
    int64_t kv_row0 = 0, tok = 0, blk_g0 = 0;
    uint32_t kn[2] = {0u, 0u}, vn[2] = {0u, 0u};
    uint32_t qa[8][4];
    float m_run[2], l_run[2], o[16][4];

    // A failed (timed-out) wait stops this thread's work but not its walk
    // through the loop: every thread reaches every barrier of the loop, and
    // the segment ends read the CTA's failure flag after a barrier.
    bool ok = true;
    TileCursor t;   // the consumers' tile
    t.seek(reqs, a.n_reqs, g0);
    for (int i = 0; i < n_mine; ++i) {
        const int64_t g = g0 + i;
        if (i > 0)
            t.next(reqs, ds.LH);
        if (i == 0 || t.j == 0) {
            // ---- a new segment: block (t.b, t.lh) from its tile t.j ----
            b = t.b;
            lh = t.lh;
            n_t = t.n_t;
            seg_j0 = t.j;
            blk_g0 = g - t.j;
            P = t.prefix;
            n_valid = P + 1;
            kv_row0 = t.cache_row0 + (int64_t)lh * t.cap;
            const int l_idx = lh / a.n_kv_heads, h_idx = lh - l_idx * a.n_kv_heads;
            tok = (int64_t)l_idx * a.total_q + t.q_off;
            w_new = (P & (kDecTile - 1)) >> 5;
            // the step's key (rotated by P) and value, written to the cache by
            // the CTA that holds the block's last tile
            if (warp == w_new && blk_g0 + n_t - 1 < g1) {
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
                if (il) {
                    rot(x0, x1, c0);
                    rot(y0, y1, c1);
                } else {
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
            // Q fragments (A operand, 16 x 128, rows >= G zero), rotated by P
            const __nv_bfloat16 *qp = static_cast<const __nv_bfloat16 *>(a.q) + (tok * a.n_q_heads + h_idx * G) * kDecD;
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
                const int col = kb * 16 + cq;
                auto ld2 = [&](int r, int cc) -> uint32_t {
                    return r < G ? *reinterpret_cast<const uint32_t *>(qp + (int64_t)r * kDecD + cc) : 0u;
                };
                qa[kb][0] = ld2(r0, col);
                qa[kb][1] = ld2(r1, col);
                qa[kb][2] = ld2(r0, col + 8);
                qa[kb][3] = ld2(r1, col + 8);
            }
            if (il) {
#pragma unroll
                for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int d = kb * 16 + cq + ((e & 2) ? 8 : 0);
                        const float2 cs = rope_cs(a.rope, kDecD / 2, P, d >> 1);
                        float x, y;
                        unpk(qa[kb][e], x, y);
                        rot(x, y, cs);
                        qa[kb][e] = pack2(x, y);
                    }
                }
            } else {
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int d = kb * 16 + cq + ((e & 2) ? 8 : 0);
                        const float2 cs0 = rope_cs(a.rope, kDecD / 2, P, d), cs1 = rope_cs(a.rope, kDecD / 2, P, d + 1);
                        float x0, x1, y0, y1;
                        unpk(qa[kb][e], x0, x1);
                        unpk(qa[kb + 4][e], y0, y1);
                        rot(x0, y0, cs0);
                        rot(x1, y1, cs1);
                        qa[kb][e] = pack2(x0, x1);
                        qa[kb + 4][e] = pack2(y0, y1);
                    }
                }
            }
            m_run[0] = m_run[1] = -INFINITY;
            l_run[0] = l_run[1] = 0.f;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        }

        // ---- tile t.j of the block ----
        const int j = t.j;
        const int s = i % kDecStages;
        if (ok && !dec_wait(full(s), (uint32_t)((i / kDecStages) & 1))) {
            ok = false;
            flags[0] = 1;
        }
        const uint32_t kt = sbase + (uint32_t)(s * kDecStageBytes), vt = kt + kDecTileBytes;
        const int key0 = 32 * warp;   // this warp's 32 keys of the tile
        if (ok) {
        if (j == n_t - 1) {
            // V rows past P are zero; row P is the step's own key and value
            for (int idx = lane; idx < 32 * 16; idx += 32) {
                const int row = key0 + (idx >> 4);
                if (j * kDecTile + row > P)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vt + sw_off(row, idx & 15)), "r"(0u)
                                 : "memory");
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
        float cs_[4][4];
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
            cs_[nb][0] = cs_[nb][1] = cs_[nb][2] = cs_[nb][3] = 0.f;
#pragma unroll
        for (int nb = 0; nb < 4; nb += 2) {
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
                const int mi = lane >> 3;
                const int key = key0 + 8 * (nb + (mi >> 1)) + (lane & 7);
                const int chunk = 2 * kb + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kt + sw_off(key, chunk), b0, b1, b2, b3);
                mma_bf16(cs_[nb], qa[kb], b0, b1);
                mma_bf16(cs_[nb + 1], qa[kb], b2, b3);
            }
        }
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kk = j * kDecTile + key0 + 8 * nb + cq + (e & 1);
                cs_[nb][e] = kk < n_valid ? cs_[nb][e] * sc : -INFINITY;
                mx[e >> 1] = fmaxf(mx[e >> 1], cs_[nb][e]);
            }
        }
        float corr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            const float m_new = fmaxf(m_run[h], mx[h]);
            corr[h] = m_new == -INFINITY ? 1.f : dec_ex2(m_run[h] - m_new);
            m_run[h] = m_new;
        }
        const float nm[2] = {m_run[0] == -INFINITY ? 0.f : -m_run[0], m_run[1] == -INFINITY ? 0.f : -m_run[1]};
        float sum[2] = {0.f, 0.f};
        uint32_t pa[2][4];
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
            const float p0 = dec_ex2(cs_[nb][0] + nm[0]), p1 = dec_ex2(cs_[nb][1] + nm[0]);
            const float p2 = dec_ex2(cs_[nb][2] + nm[1]), p3 = dec_ex2(cs_[nb][3] + nm[1]);
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
#pragma unroll
        for (int kb2 = 0; kb2 < 2; ++kb2) {
#pragma unroll
            for (int n = 0; n < 16; n += 2) {
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
        }
        if (threadIdx.x == 0 && ok && i + kDecStages < n_mine) {
            if (!dec_wait(empty(s), (uint32_t)((i / kDecStages) & 1))) {
                ok = false;
                flags[0] = 1;
            } else {
                issue(i + kDecStages);
                ++n_issued;
            }
        }

        if (j != n_t - 1 && i != n_mine - 1)
            continue;
        // ---- end of the segment: the four warps' states, combined in a fixed order ----
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
        if (flags[0]) {   // uniform: no wait of this segment is pending any more
            __syncthreads();
            continue;
        }
        const bool whole = seg_j0 == 0 && j == n_t - 1;
        const int blk = b * ds.LH + lh;
        const int l_idx = lh / a.n_kv_heads, h_idx = lh - l_idx * a.n_kv_heads;
        const int c0 = 16 * (threadIdx.x & 7);
        // this part's workspace slot (when the block is split between CTAs)
        float *mine = ds.ws + ((int64_t)c * 2 + part_slot(blk_g0, g0)) * kPartFloats;
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
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    acc += oo[(w * 16 + rr) * kDecD + c0 + e] * wgt[w];
                v[e] = acc;
            }
            if (whole) {
                const float inv = 1.f / L;
                if (!(L > 0.f && L < INFINITY) && (threadIdx.x & 7) == 0 && a.err)
                    atomicCAS(a.err, kDevOk, kDevBadInput);
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2)
                    pk[e >> 1] = pack2(v[e] * inv, v[e + 1] * inv);
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                     ((tok * a.n_q_heads) + h_idx * G + rr) * kDecD + c0;
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            } else {
                if ((threadIdx.x & 7) == 0) {
                    mine[rr] = M;
                    mine[16 + rr] = L;
                }
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4 *>(mine + 32 + rr * kDecD + c0 + e) =
                        make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
            }
        }
        if (!whole) {
            // arrive on the block's count; the part that completes it merges
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) {
                const int c_first = share_of(blk_g0, ds.n_cta, ds.total);
                const int c_last = share_of(blk_g0 + n_t - 1, ds.n_cta, ds.total);
                const int old = atomicAdd(ds.cnt + blk, 1);
                flags[1] = old == c_last - c_first ? 1 : 0;
            }
            __syncthreads();
            if (flags[1]) {
                __threadfence();
                const int c_first = share_of(blk_g0, ds.n_cta, ds.total);
                const int c_last = share_of(blk_g0 + n_t - 1, ds.n_cta, ds.total);
                for (int rr = threadIdx.x >> 3; rr < G; rr += kDecThreads / 8) {
                    float M = -INFINITY;
                    for (int cp = c_first; cp <= c_last; ++cp) {
                        const float *part = ds.ws +
                            ((int64_t)cp * 2 + part_slot(blk_g0, share_start(cp, ds.n_cta, ds.total))) * kPartFloats;
                        M = fmaxf(M, __ldcg(part + rr));
                    }
                    float L = 0.f, v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        v[e] = 0.f;
                    for (int cp = c_first; cp <= c_last; ++cp) {
                        const float *part = ds.ws +
                            ((int64_t)cp * 2 + part_slot(blk_g0, share_start(cp, ds.n_cta, ds.total))) * kPartFloats;
                        const float wgt = dec_ex2(__ldcg(part + rr) - M);
                        L += __ldcg(part + 16 + rr) * wgt;
#pragma unroll
                        for (int e = 0; e < 16; e += 4) {
                            const float4 x = __ldcg(reinterpret_cast<const float4 *>(part + 32 + rr * kDecD + c0 + e));
                            v[e] += x.x * wgt;
                            v[e + 1] += x.y * wgt;
                            v[e + 2] += x.z * wgt;
                            v[e + 3] += x.w * wgt;
                        }
                    }
                    const float inv = 1.f / L;
                    if (!(L > 0.f && L < INFINITY) && (threadIdx.x & 7) == 0 && a.err)
                        atomicCAS(a.err, kDevOk, kDevBadInput);
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2)
                        pk[e >> 1] = pack2(v[e] * inv, v[e + 1] * inv);
                    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                         ((tok * a.n_q_heads) + h_idx * G + rr) * kDecD + c0;
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
                if (threadIdx.x == 0)
                    ds.cnt[blk] = 0;   // ready for the next step
            }
        }
        __syncthreads();   // the merge area is free again
    }
    __syncthreads();
    if (flags[0]) {
        if (threadIdx.x == 0 && a.err)
            atomicCAS(a.err, kDevOk, kDevTimeout);
        // copies in flight land before the CTA leaves (bounded)
        if (threadIdx.x == 0)
            for (int k = n_issued > kDecStages ? n_issued - kDecStages : 0; k < n_issued; ++k)
                dec_wait(full(k % kDecStages), (uint32_t)((k / kDecStages) & 1));
    }
}

cudaError_t launch_decode_stream(const AttnArgs &a, const ReqTable &rt, const void *tmap_k, const void *tmap_v,
                                 const DecodeIO &io, const DecodeStream &ds, cudaStream_t s)
{
    if (ds.total == 0 || ds.n_cta == 0)
        return cudaSuccess;
    static std::atomic<bool> attr_set[64] = {};   // per device (host threads may race: same value)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k_decode_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, kDsSmem);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            attr_set[dev].store(true, std::memory_order_release);
    }
    k_decode_stream<<<(unsigned)ds.n_cta, kDecThreads, kDsSmem, s>>>(*static_cast<const CUtensorMap *>(tmap_k),
                                                                   *static_cast<const CUtensorMap *>(tmap_v), a, rt,
                                                                   io, ds);
    return cudaGetLastError();
}

int decode_stream_part_floats() { return kPartFloats; }

}  // namespace kvr
