// kvr_attention_tc.cu -- query prefill attention on the 5th-generation tensor
// cores: tcgen05.mma with TMEM accumulators, K/V tiles fed by TMA, online
// softmax in registers.
//
// What it computes (CoinRAG blog section 2.3, KV_M(q; C_ctx); TurboRAG blog,
// "Attention Mask"; SemPIC page, causal interleave): query token t of request
// b sits at position P_b + t and attends to the P_b stitched prefix rows and
// to query rows 0..t of its (layer, kv-head) block of the cache (the query
// rows were appended, rotated, by the assemble kernel just before).
//
// Tiling.  A CTA owns one (request, 128-row M-tile, layer, kv-head).  The
// G = H_q / H_kv query heads sharing a kv head are packed into M (row
// r = t * G + g), so each K/V tile feeds all of them.  Per 128-key tile j:
//   S_j = Q K_j^T      (tcgen05.mma, A = Q smem, B = K smem, D = TMEM, fp32)
//   P_j = exp2(S_j * scale*log2e - m)   (softmax warps; row r = TMEM lane r)
//   O  += P_j V_j      (tcgen05.mma, A = P smem, B = V smem (MN-major), D = TMEM)
// S is double-buffered in TMEM so S_{j+1} runs while the softmax warps work on
// S_j.  The running max is rescaled lazily: O is rescaled in TMEM only when a
// row's max grows by more than 8 (log2 units), so that p <= 2^8 stays exact
// enough in bf16 and the rescale is rare.
//
// Warp roles (192 threads): warps 0-3 load + rotate Q, run the softmax and
// the epilogue (one row per thread = one TMEM lane); warp 4 issues the TMA
// loads; warp 5 owns TMEM and issues the MMAs (one thread).
//
// Every mbarrier wait is bounded (2 s of %globaltimer); on expiry the CTA
// records KVR_ERR_TIMEOUT in the pool's error word, all roles leave their
// loops, in-flight copies and MMAs are drained (again bounded) and TMEM is
// freed before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kThreads = 192;
constexpr int kTileM = 128;      // query rows per CTA
constexpr int kTileN = 128;      // keys per K/V tile
constexpr int kD = 128;          // head dim
constexpr int kSlots = 4;        // K/V tile ring (K_j, V_j, K_j+1, ...)
constexpr int kTileBytes = kTileN * kD * 2;   // 32 KB
constexpr int kPanelBytes = kTileBytes / 2;   // 16 KB: 128 rows x 64 columns
constexpr int kTmemCols = 512;
constexpr int kColS = 0;         // S buffers at columns 0 and 128
constexpr int kColO = 256;       // O at columns 256..383
constexpr float kRescaleThreshold = 8.0f;
constexpr unsigned long long kWaitNs = 2000000000ull;

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kTileBytes;
constexpr int kOffKV = kOffP + kTileBytes;
constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
// barriers: full[kSlots], empty[kSlots], s_full[2], s_empty[2], p_full, o_done, q_ready, drain
constexpr int kBarFull = 0, kBarEmpty = kSlots, kBarSFull = 2 * kSlots, kBarSEmpty = 2 * kSlots + 2,
              kBarPFull = 2 * kSlots + 4, kBarODone = 2 * kSlots + 5, kBarQReady = 2 * kSlots + 6,
              kBarDrain = 2 * kSlots + 7, kNumBars = 2 * kSlots + 8;
constexpr int kOffTmemAddr = kOffBar + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemAddr + 4;
constexpr int kSmemBytes = kOffAbort + 4 + 1024;   // + alignment slack

// instruction descriptors (kind::f16): D fp32, A and B bf16, M = 128, N = 128
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTileN >> 3) << 17) |
                                ((uint32_t)(kTileM >> 4) << 24);
constexpr uint32_t kIdescS = kIdescBase;               // A, B K-major
constexpr uint32_t kIdescPV = kIdescBase | (1u << 16); // B (V) MN-major

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: false if the CTA aborted or the wait ran past kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (globaltimer() - t0 > kWaitNs)
            return false;
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version
    d |= (uint64_t)2 << 61;   // SWIZZLE_128B
    return d;
}

// Byte offset of 16-byte chunk `c` (0..15 over 128 columns) of row r in a
// [128 rows x 128 bf16] tile stored as two 128B-swizzled 64-column panels.
__device__ __forceinline__ uint32_t sw128_off(int r, int c)
{
    return (uint32_t)((c >> 3) * kPanelBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void flag_timeout(int *err, volatile int *abort_flag)
{
    *abort_flag = 1;
    atomicCAS(err, 0, kDevTimeout);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_attention_tc(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const AttnArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kOffBar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemAddr);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- which (request, M-tile, layer, kv-head) ----
    const int mt = blockIdx.x;
    const int lh = blockIdx.y;
    int lo = 0, hi = a.n_reqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.reqs[mid].m_tile0 <= mt)
            lo = mid;
        else
            hi = mid - 1;
    }
    const DevReq rq = a.reqs[lo];
    const int G = a.n_q_heads / a.n_kv_heads;
    const int l = lh / a.n_kv_heads, h = lh - l * a.n_kv_heads;
    const int row0 = (mt - rq.m_tile0) * kTileM;            // first packed row of the tile
    const int m_rows = G * rq.q_len;                        // packed rows of the request
    const int t_max = min(rq.q_len - 1, (row0 + kTileM - 1) / G);
    const int n_keys = rq.prefix + t_max + 1;               // keys any row of the tile sees
    const int n_tiles = (n_keys + kTileN - 1) / kTileN;
    const int n_valid = rq.prefix + rq.q_len;               // rows of the block that hold data
    const int64_t unit_row0 = rq.cache_row0 + (int64_t)lh * rq.cap;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(bar(i), (i == kBarSEmpty || i == kBarSEmpty + 1 || i == kBarPFull || i == kBarQReady)
                                  ? 128u
                                  : 1u);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5)
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        // =================== softmax / epilogue warpgroup ===================
        const int r = threadIdx.x;                 // row of the tile = TMEM lane
        const int rr = row0 + r;                   // packed row in the request
        const bool row_ok = rr < m_rows;
        const int t = row_ok ? rr / G : t_max;     // query token of this row
        const int g = row_ok ? rr - (rr / G) * G : 0;
        const int pos = rq.prefix + t;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);

        // Q row: load, rotate at position P + t, store bf16 into the swizzled tile
        {
            const __nv_bfloat16 *qp = static_cast<const __nv_bfloat16 *>(a.q) +
                                      (((int64_t)l * a.total_q + rq.q_off + t) * a.n_q_heads + h * G + g) * kD;
#pragma unroll
            for (int c = 0; c < 8; ++c) {          // chunk c (cols 8c..8c+7) with partner chunk c+8
                uint4 x = make_uint4(0, 0, 0, 0), y = make_uint4(0, 0, 0, 0);
                if (row_ok) {
                    x = *reinterpret_cast<const uint4 *>(qp + 8 * c);
                    y = *reinterpret_cast<const uint4 *>(qp + 64 + 8 * c);
                    uint32_t *px = reinterpret_cast<uint32_t *>(&x);
                    uint32_t *py = reinterpret_cast<uint32_t *>(&y);
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float2 fx = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&px[w]));
                        const float2 fy = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&py[w]));
                        const float2 c0 = rope_cs(a.rope, kD / 2, pos, 8 * c + 2 * w);
                        const float2 c1 = rope_cs(a.rope, kD / 2, pos, 8 * c + 2 * w + 1);
                        __nv_bfloat162 ox = __floats2bfloat162_rn(fmaf(fx.x, c0.x, -fy.x * c0.y),
                                                                  fmaf(fx.y, c1.x, -fy.y * c1.y));
                        __nv_bfloat162 oy = __floats2bfloat162_rn(fmaf(fx.x, c0.y, fy.x * c0.x),
                                                                  fmaf(fx.y, c1.y, fy.y * c1.x));
                        px[w] = *reinterpret_cast<uint32_t *>(&ox);
                        py[w] = *reinterpret_cast<uint32_t *>(&oy);
                    }
                }
                *reinterpret_cast<uint4 *>(smem + kOffQ + sw128_off(r, c)) = x;
                *reinterpret_cast<uint4 *>(smem + kOffQ + sw128_off(r, c + 8)) = y;
            }
            fence_async_smem();
            mbar_arrive(bar(kBarQReady));
        }

        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int sb = j & 1;
            if (!mbar_wait(bar(kBarSFull + sb), (j >> 1) & 1, abort_flag)) {
                flag_timeout(a.err, abort_flag);
                ok = false;
                break;
            }
            tc_fence_after();
            float s[kTileN];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tmem_ld32(lane_base + kColS + sb * kTileN + 32 * q, s + 32 * q);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(kBarSEmpty + sb));

            // mask: key 128j + c is visible to this row iff it is <= P + t
            const int lim = pos + 1 - j * kTileN;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kTileN; ++c) {
                s[c] = (c < lim) ? s[c] * a.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[c]);
            }
            bool waited = false;
            if (j == 0) {
                m_run = mx;
            } else if (mx > m_run + kRescaleThreshold) {
                // O must hold PV_{j-1} before it is rescaled
                if (!mbar_wait(bar(kBarODone), (j - 1) & 1, abort_flag)) {
                    flag_timeout(a.err, abort_flag);
                    ok = false;
                    break;
                }
                waited = true;
                tc_fence_after();
                const float corr = ex2(m_run - mx);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float o[32];
                    tmem_ld32(lane_base + kColO + 32 * q, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] *= corr;
                    tmem_st32(lane_base + kColO + 32 * q, o);
                }
                tmem_wait_st();
                l_run *= corr;
                m_run = mx;
            }
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < kTileN; ++c) {
                s[c] = ex2(s[c] - m_run);
                sum += s[c];
            }
            l_run += sum;
            // the P buffer is free once PV_{j-1} completed
            if (j > 0 && !waited) {
                if (!mbar_wait(bar(kBarODone), (j - 1) & 1, abort_flag)) {
                    flag_timeout(a.err, abort_flag);
                    ok = false;
                    break;
                }
            }
            // last tile: zero V rows past the block's data so that p = 0
            // never meets a non-finite value
            if (j == n_tiles - 1 && j * kTileN + r >= n_valid) {
                const int tv = 2 * j + 1;
                if (!mbar_wait(bar(kBarFull + tv % kSlots), (tv / kSlots) & 1, abort_flag)) {
                    flag_timeout(a.err, abort_flag);
                    ok = false;
                    break;
                }
                uint8_t *vt = smem + kOffKV + (tv % kSlots) * kTileBytes;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<uint4 *>(vt + sw128_off(r, c)) = make_uint4(0, 0, 0, 0);
            }
            uint8_t *pt = smem + kOffP;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint4 v;
                uint32_t *pv = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(s[8 * c + 2 * w], s[8 * c + 2 * w + 1]);
                    pv[w] = *reinterpret_cast<uint32_t *>(&b2);
                }
                *reinterpret_cast<uint4 *>(pt + sw128_off(r, c)) = v;
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar(kBarPFull));
        }
        // epilogue: O / l -> bf16 -> out[l][q_off + t][h*G + g][:]
        if (ok) {
            if (!mbar_wait(bar(kBarODone), (n_tiles - 1) & 1, abort_flag)) {
                flag_timeout(a.err, abort_flag);
            } else {
                tc_fence_after();
                const float inv = 1.f / l_run;
                __nv_bfloat16 *op = static_cast<__nv_bfloat16 *>(a.out) +
                                    (((int64_t)l * a.total_q + rq.q_off + t) * a.n_q_heads + h * G + g) * kD;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float o[32];
                    tmem_ld32(lane_base + kColO + 32 * q, o);
                    tmem_wait_ld();
                    if (row_ok) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint4 v;
                            uint32_t *pv = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                __nv_bfloat162 b2 = __floats2bfloat162_rn(o[8 * c + 2 * w] * inv,
                                                                          o[8 * c + 2 * w + 1] * inv);
                                pv[w] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            *reinterpret_cast<uint4 *>(op + 32 * q + 8 * c) = v;
                        }
                    }
                }
            }
        }
    } else if (warp == 4) {
        // =================== TMA producer ===================
        if (lane == 0) {
            int issued = 0;
            for (int tt = 0; tt < 2 * n_tiles; ++tt) {
                const int slot = tt % kSlots;
                if (tt >= kSlots && !mbar_wait(bar(kBarEmpty + slot), ((tt / kSlots) - 1) & 1, abort_flag)) {
                    flag_timeout(a.err, abort_flag);
                    break;
                }
                const uint32_t dst = sbase + kOffKV + slot * kTileBytes;
                const CUtensorMap *map = (tt & 1) ? &tmv : &tmk;
                const int row = (int)(unit_row0 + (int64_t)(tt >> 1) * kTileN);
                mbar_expect_tx(bar(kBarFull + slot), kTileBytes);
                tma_load_2d(dst, map, 0, row, bar(kBarFull + slot));
                tma_load_2d(dst + kPanelBytes, map, 64, row, bar(kBarFull + slot));
                issued = tt + 1;
            }
            // drain: every issued copy lands before the CTA leaves
            for (int tt = (issued > kSlots ? issued - kSlots : 0); tt < issued; ++tt) {
                uint64_t t0 = globaltimer();
                while (!mbar_try_wait(bar(kBarFull + tt % kSlots), (tt / kSlots) & 1) &&
                       globaltimer() - t0 < kWaitNs) {
                }
            }
        }
    } else {
        // =================== MMA issuer ===================
        if (lane == 0) {
            bool ok = mbar_wait(bar(kBarQReady), 0, abort_flag);
            if (!ok)
                flag_timeout(a.err, abort_flag);
            tc_fence_after();
            const uint32_t q_base = sbase + kOffQ, p_base = sbase + kOffP;
            auto issue_s = [&](int j) -> bool {
                const int tt = 2 * j, slot = tt % kSlots;
                if (!mbar_wait(bar(kBarFull + slot), (tt / kSlots) & 1, abort_flag))
                    return false;
                if (j >= 2 && !mbar_wait(bar(kBarSEmpty + (j & 1)), ((j >> 1) - 1) & 1, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t kb = sbase + kOffKV + slot * kTileBytes;
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t off = (k >> 2) * kPanelBytes + (k & 3) * 32;
                    umma_f16(tmem + kColS + (j & 1) * kTileN, sdesc(q_base + off, 16, 1024),
                             sdesc(kb + off, 16, 1024), kIdescS, k > 0);
                }
                umma_commit(bar(kBarSFull + (j & 1)));
                umma_commit(bar(kBarEmpty + slot));
                return true;
            };
            if (ok)
                ok = issue_s(0);
            for (int j = 0; j < n_tiles && ok; ++j) {
                if (j + 1 < n_tiles && !(ok = issue_s(j + 1)))
                    break;
                const int tt = 2 * j + 1, slot = tt % kSlots;
                if (!mbar_wait(bar(kBarPFull), j & 1, abort_flag) ||
                    !mbar_wait(bar(kBarFull + slot), (tt / kSlots) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t vb = sbase + kOffKV + slot * kTileBytes;
#pragma unroll
                for (int k = 0; k < kTileN / 16; ++k) {
                    const uint32_t aoff = (k >> 2) * kPanelBytes + (k & 3) * 32;
                    umma_f16(tmem + kColO, sdesc(p_base + aoff, 16, 1024),
                             sdesc(vb + k * 2048, kPanelBytes, 1024), kIdescPV, (j > 0 || k > 0));
                }
                umma_commit(bar(kBarEmpty + slot));
                umma_commit(bar(kBarODone));
            }
            if (!ok)
                flag_timeout(a.err, abort_flag);
            // drain: all issued MMAs complete before TMEM is released
            umma_commit(bar(kBarDrain));
            uint64_t t0 = globaltimer();
            while (!mbar_try_wait(bar(kBarDrain), 0) && globaltimer() - t0 < kWaitNs) {
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

bool attention_tc_supported(int dtype, int head_dim) { return dtype == KVR_DTYPE_BF16 && head_dim == kD; }

cudaError_t launch_attention_tc(const TcAttnArgs &ta, cudaStream_t s)
{
    if (ta.n_m_tiles == 0)
        return cudaSuccess;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_attention_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    const int LH = ta.base.n_layers * ta.base.n_kv_heads;
    dim3 grid(ta.n_m_tiles, LH);
    k_attention_tc<<<grid, kThreads, kSmemBytes, s>>>(*static_cast<const CUtensorMap *>(ta.tmap_k),
                                                      *static_cast<const CUtensorMap *>(ta.tmap_v), ta.base);
    return cudaGetLastError();
}

}  // namespace kvr
