// kvr_attention_tc.cu -- query prefill attention on the 5th-generation tensor
// cores: tcgen05.mma with TMEM accumulators, K/V tiles fed by TMA, online
// softmax in registers.
//
// What it computes (CoinRAG blog section 2.3, KV_M(q; C_ctx); TurboRAG blog,
// "Attention Mask"; SemPIC page, causal interleave): query token t of request
// b sits at position P_b + t and attends to the P_b stitched prefix rows and
// to query rows 0..t of its (layer, kv-head) block of the cache (the query
// rows were appended, rotated, by the query prologue just before).
//
// Tiling.  A work unit is one (request, 256-row query block, layer, kv-head),
// split into two 128-row tiles A and B; the kernel is persistent (one CTA per
// SM walks the units), so the next unit's Q and K/V loads overlap the current
// unit's last softmax and its epilogue; a tile's first S MMA of the next unit
// follows that tile's epilogue.  The G = H_q / H_kv query heads that
// share a kv head are packed into the rows (row r = t * G + g), so each K/V
// tile is read once for all of them, and once for both tiles.  Per 128-key
// tile j and tile X in {A, B}:
//   S_X = Q_X K_j^T          tcgen05.mma, A = Q_X (smem), B = K_j (smem), D = TMEM
//   P_X = exp2(S_X * c - m)  softmax warpgroup X, one row per thread = TMEM lane;
//                            P_X is written back into TMEM over S_X as bf16
//   O_X += P_X V_j           tcgen05.mma, A = P_X (TMEM), B = V_j (smem, MN-major)
// The MMA warp issues S_A(0), S_B(0), then per tile PV_A(j), S_A(j+1),
// PV_B(j), S_B(j+1): the tensor core works on one tile while the other
// tile's warpgroup runs its softmax.  MMAs of one thread execute in issue
// order, so S_X(j+1) (issued after PV_X(j)) never overwrites P_X(j) before
// PV_X(j) has read it; and the commit that signals S_X(j+1) covers PV_X(j), so
// O_X is stable whenever its warpgroup sees a new S_X.  The running max is
// rescaled lazily: O_X is rescaled in TMEM only when a row's max grows by more
// than 8 (log2 units).
//
// Warp roles (384 threads, one CTA per SM): warps 0-3 and 4-7 are the
// warpgroups of tiles A and B (softmax, epilogue); warp 8 issues the TMA loads
// of Q (already rotated and packed by the query-prologue kernel; the next
// unit's Q is prefetched into L2) and of the K/V tiles into a 4-slot ring;
// warp 9 owns the 512 TMEM columns and runs the MMA schedule on all 32 lanes,
// one lane (elected once) issuing the tcgen05 instructions: with the
// schedule's descriptor arithmetic warp-uniform, one MMA issues about as fast
// as the tensor core retires it (issued from a single-lane branch it was the
// bottleneck); warps 10-11 complete the third warpgroup, so that the
// registers can be split by warpgroup (setmaxnreg): the softmax warpgroups
// hold a whole row of S and run without spills (in the values-gathering
// variant they are the gather warps).  Barrier phases run on across units.
//
// Epilogue: each softmax thread holds one output row; its warp stages 32 rows
// x 64 columns at a time in shared memory and writes them back with one TMA
// tensor store (32 / G whole tokens, G a power of two) or as whole 128-byte
// lines (row-per-thread stores touch one line per lane); then it releases O_x
// (and, through the MMA warp's wait, the shared memory the next S MMA reads).
//
// Values-gathering variant (a prefill whose stitched prefix is not kept): the
// keys come from the cache, stitched by a keys-only stitch; each value tile
// that holds prefix rows is read from the pool through the span table, which
// halves the stitch's traffic.  For a request of long spans the producer loads
// those tiles (runs of 32 consecutive pool rows as one box load, other rows as
// gather4); for one of short spans warps 10-11 copy them with 16-byte
// cp.async copies.  The gather warps also fill the tile that holds the first
// query rows (from the cache) and zero the rows past a request's keys where a
// tile reaches past its cache block, whose value rows this variant does not
// write.
//
// Every mbarrier wait is bounded (2 s of %globaltimer); on expiry the CTA
// records KVR_ERR_TIMEOUT in the pool's error word, all roles leave their
// loops, in-flight copies and MMAs are drained (again bounded) and TMEM is
// freed before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "kvr_internal.cuh"

namespace kvr {

namespace {

// stitched-cache variant: 10 working warps and 2 idle ones completing the
// third warpgroup; launched at 168 registers a thread (the most for 384), the
// softmax warpgroups take 200 and the third gives up to 104 (setmaxnreg):
// 2 x 128 x 200 + 128 x 104 = 384 x 168.  At 320 threads and a flat 168 the
// softmax loop spilled, and G = 7 workloads ran 6-15 % slower.
constexpr int kThreads = 384;
constexpr int kRegsLaunchS = 168, kRegsSoftmaxS = 200, kRegsOtherS = 104;
static_assert(2 * 128 * kRegsSoftmaxS + 128 * kRegsOtherS <= kThreads * kRegsLaunchS, "register split");
constexpr int kTileM = 128;      // query rows per tile (two tiles per CTA)
constexpr int kTileN = 128;      // keys per K/V tile
constexpr int kD = 128;          // head dim
constexpr int kSlots = 4;        // K/V ring: K_j, V_j, K_j+1, V_j+1
constexpr int kTileBytes = kTileN * kD * 2;   // 32 KB
constexpr int kPanelBytes = kTileBytes / 2;   // 16 KB: 128 rows x 64 columns
constexpr int kTmemCols = 512;
// TMEM columns of tile x: S_x (P_x over its first 64) and O_x
__host__ __device__ constexpr uint32_t col_s(int x) { return 128u * (uint32_t)x; }
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u + 128u * (uint32_t)x; }
constexpr float kRescaleThreshold = 8.0f;
constexpr unsigned long long kWaitNs = 2000000000ull;

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;                          // Q_A, Q_B
constexpr int kOffKV = kOffQ + 2 * kTileBytes;
constexpr int kOffStage = kOffKV + kSlots * kTileBytes;
constexpr int kStageBytes = 8 * 32 * 128;
constexpr int kOffBar = kOffStage + kStageBytes;
// barriers
constexpr int kBarFull = 0;                       // [kSlots] K/V tile landed
constexpr int kBarEmpty = kBarFull + kSlots;      // [kSlots] K/V tile consumed
constexpr int kBarSFull = kBarEmpty + kSlots;     // [2] S_x computed
constexpr int kBarPFull = kBarSFull + 2;          // [2] P_x written (128 arrivals)
constexpr int kBarOFull = kBarPFull + 2;          // [2] O_x final for the unit
constexpr int kBarOEmpty = kBarOFull + 2;         // [2] O_x out, staged and stored (128 arrivals)
constexpr int kBarQFull = kBarOEmpty + 2;         // Q tiles landed
constexpr int kBarQEmpty = kBarQFull + 1;         // all S of the unit done with Q
constexpr int kBarDrain = kBarQEmpty + 1;
// split units (two-CTA cluster, half h on CTA rank h; rank x merges tile x):
// the partner's half of this CTA's tile has landed in its shared memory (128
// arrivals); the partner's MMAs are all done, so its K/V ring and Q tiles may
// take this CTA's half of the partner's tile
constexpr int kBarPeerData = kBarDrain + 1;
constexpr int kBarPeerFree = kBarPeerData + 1;
// the geometry of the CTA's next items, written by the producer warp (two
// slots): full (1 arrival), read by every consumer warp (one arrival each)
constexpr int kBarGeoFull = kBarPeerFree + 1;     // [2]
constexpr int kBarGeoEmpty = kBarGeoFull + 2;     // [2]
// values-gathering variant, one of each per V ring slot (odd slots), so that
// none runs more than a phase ahead of its waiters (a slot is refilled only
// after the MMAs consumed it): the slot is free for the gather warps' next
// tile (1 arrival, the producer); the gather warps' tile has landed (2
// arrivals, one a gather warp)
constexpr int kBarGatherJob = kBarGeoEmpty + 2;   // [2]
constexpr int kBarGathered = kBarGatherJob + 2;   // [2]
constexpr int kNumBars = kBarGathered + 2;
constexpr int kOffTmemAddr = kOffBar + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemAddr + 4;
constexpr int kOffGeo = (kOffAbort + 4 + 15) & ~15;   // [2] Item
constexpr int kGeoBytes = 128;
constexpr int kSmemBytes = kOffGeo + 2 * kGeoBytes + 1024;   // + alignment slack
// where a split unit's partner CTA leaves its half of this CTA's tile: O as
// fp16 with a power-of-two scale per row ([16-byte piece of 8][row]) over the
// K/V ring; the running max, sum and scale (fp32 [3][128]) over the Q tiles
constexpr int kOffPeerO = kOffKV;
constexpr int kPeerOBytes = kTileM * kD * 2;
constexpr int kOffPeerML = kOffQ;
static_assert(kPeerOBytes <= kSlots * kTileBytes && 3 * kTileM * 4 <= 2 * kTileBytes, "peer state");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

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

// Generic-proxy writes to shared memory become visible to the async proxy
// (the tensor core reads its operands through it).
// Fetch a tensor map (a kernel parameter) ahead of its first copy.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bring a tile into L2 ahead of its load into shared memory.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int c0, int c1)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
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

// Shared memory -> global through a 3-D tensor map (bulk async-group of the
// issuing thread); commit, and wait until the group no longer reads shared
// memory / has completed.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// 16 bytes global -> shared, asynchronous (this thread's copies complete at
// cp_async_wait_all); no register holds the data
// Four rows (given by row coordinate) x 64 columns of a 2-D tensor whose box
// is one row high, into four consecutive 128-byte rows of shared memory.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, int c0, const int *rows,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(rows[0]), "r"(rows[1]), "r"(rows[2]), "r"(rows[3]),
        "r"(bar)
        : "memory");
}

// (src_bytes 0: the 16 bytes are zero-filled and nothing is read)
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

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

// The MMA role runs on all 32 lanes of its warp (descriptor arithmetic stays
// warp-uniform); one lane, elected once, issues the tcgen05 instructions.
__device__ __forceinline__ uint32_t elect_one()
{
    uint32_t p;
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(p));
    return p;
}

template <bool ACC>
__device__ __forceinline__ void mma_ss(uint32_t lead, uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc)
{
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "n"(ACC ? 1 : 0), "r"(lead)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t lead, uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                         uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(lead)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t lead, uint32_t bar)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
                 "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
                 "r"(lead)
                 : "memory");
}


// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// MMA issue with precomputed descriptors: a descriptor's address field is in
// its low word, so a K-step or a ring slot only adds to the low word (the
// issuing thread shares its SM sub-partition with two softmax warps, so every
// instruction it saves shortens the tensor pipe's wait for work).
__device__ __forceinline__ uint64_t desc_with_lo(uint32_t lo, uint32_t hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
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


__device__ __forceinline__ void flag_timeout(int *err, volatile int *abort_flag)
{
    *abort_flag = 1;
    atomicCAS(err, 0, kDevTimeout);
}


__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Packed fp32 pairs (two lanes of one 64-bit register) for the softmax.
__device__ __forceinline__ uint64_t pk2(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void unpk2(uint64_t r, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---- the two CTAs of a cluster (split units) ----
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float a)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(a) : "memory");
}

// Arrive on a barrier of another CTA of the cluster, releasing this thread's
// earlier writes to that CTA's shared memory.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// Bounded wait that acquires at cluster scope (sees the writes another CTA
// released before arriving).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    const uint64_t t0 = globaltimer();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok)
            return true;
        if (*abort_flag)
            return false;
        if (globaltimer() - t0 > kWaitNs)
            return false;
    }
}

// All threads of both CTAs of the cluster (a launch without clusters is a
// cluster of one CTA).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Geometry of one work unit, computed identically by every role.
struct Unit {
    DevReq rq;
    int b;              // request index
    int l, h, lh;
    int row0[2];        // first packed row of tiles A and B in the request
    int n_t[2];         // K/V tiles each query tile needs (0: tile has no rows)
    int n_tiles;        // max of the two
    int n_valid;        // rows of the (layer, kv-head) block that hold data
    int m_rows;         // packed query rows of the request
    int64_t kv_row0;    // first cache row of the block
    int q_row0;         // first row of tile A in the packed rotated Q
};

// Units are numbered request by request in the table's (schedule) order, and
// inside a request (layer, kv-head)-major, so that the 256-row blocks of one
// (layer, kv-head) are neighbours: in the persistent loop they run at the
// same time on neighbouring SMs and read the same K/V tiles (the second read
// hits L2).  With the longest requests first, every round of units is of
// even length and the last, partial round holds the shortest.
// The geometry of unit u of request `rq` (table index b).
__device__ __forceinline__ Unit unit_geometry(const AttnArgs &a, const DevReq &rq, int b, int u)
{
    Unit w;
    w.rq = rq;
    w.b = b;
    const int G = a.n_q_heads / a.n_kv_heads;
    const int nb = (G * w.rq.q_len + 2 * kTileM - 1) / (2 * kTileM);   // 256-row blocks of the request
    const int local = u - w.rq.unit0;
    const int lh_i = local / nb;           // within the kernel's (layer, kv-head) slice
    const int mb = local - lh_i * nb;
    w.lh = a.lh_base + lh_i;
    w.l = w.lh / a.n_kv_heads;
    w.h = w.lh - w.l * a.n_kv_heads;
    w.m_rows = G * w.rq.q_len;
    const int base = mb * 2 * kTileM;
    w.row0[0] = base;
    w.row0[1] = base + kTileM;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        if (w.row0[x] >= w.m_rows) {
            w.n_t[x] = 0;
        } else {
            const int t_max = min(w.rq.q_len - 1, (w.row0[x] + kTileM - 1) / G);
            w.n_t[x] = (w.rq.prefix + t_max + 1 + kTileN - 1) / kTileN;
        }
    }
    w.n_tiles = max(w.n_t[0], w.n_t[1]);
    w.n_valid = w.rq.prefix + w.rq.q_len;
    w.kv_row0 = w.rq.cache_row0 + (int64_t)w.lh * w.rq.cap;
    w.q_row0 = (w.lh * a.total_q + w.rq.q_off) * G + base;
    return w;
}

__device__ __forceinline__ Unit unit_at(const AttnArgs &a, const DevReq *reqs, int n_blocks, int u)
{
    (void)n_blocks;
    int lo = 0, hi = a.n_reqs - 1;
    while (lo < hi) {   // the last request whose first unit is <= u
        const int mid = (lo + hi + 1) >> 1;
        if (reqs[mid].unit0 <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return unit_geometry(a, reqs[lo], lo, u);
}

// The request table of a batch of up to 64 requests held in a warp's
// registers (lane i: requests i and 32 + i), so that the producer warp finds a
// unit's request with a ballot and shuffles instead of a chain of dependent
// loads (kernel parameters or global memory, whose lines the K/V stream keeps
// evicting: about 2 us per item otherwise).
struct ReqRegs {
    DevReq r[2];
    bool ok;            // the batch has at most 64 requests (else: table lookups)

    __device__ __forceinline__ void load(const AttnArgs &a, const DevReq *reqs, int lane)
    {
        ok = a.n_reqs <= 64;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = lane + 32 * k;
            r[k] = {};
            if (ok && i < a.n_reqs)
                r[k] = reqs[i];
        }
    }
};

__device__ __forceinline__ Unit unit_at_warp(const AttnArgs &a, const ReqRegs &rr, int u, int lane)
{
    const unsigned lo = __ballot_sync(0xffffffffu, lane < a.n_reqs && rr.r[0].unit0 <= u);
    const unsigned hi = __ballot_sync(0xffffffffu, lane + 32 < a.n_reqs && rr.r[1].unit0 <= u);
    const int b = hi ? 32 + 31 - __clz(hi) : 31 - __clz(lo);   // the last request whose first unit is <= u
    const int k = b >> 5, src = b & 31;
    DevReq rq;
    rq.cache_row0 = __shfl_sync(0xffffffffu, k ? rr.r[1].cache_row0 : rr.r[0].cache_row0, src);
    rq.cap = __shfl_sync(0xffffffffu, k ? rr.r[1].cap : rr.r[0].cap, src);
    rq.prefix = __shfl_sync(0xffffffffu, k ? rr.r[1].prefix : rr.r[0].prefix, src);
    rq.q_off = __shfl_sync(0xffffffffu, k ? rr.r[1].q_off : rr.r[0].q_off, src);
    rq.q_len = __shfl_sync(0xffffffffu, k ? rr.r[1].q_len : rr.r[0].q_len, src);
    rq.unit0 = __shfl_sync(0xffffffffu, k ? rr.r[1].unit0 : rr.r[0].unit0, src);
    rq.span0 = __shfl_sync(0xffffffffu, k ? rr.r[1].span0 : rr.r[0].span0, src);
    rq.span_end = __shfl_sync(0xffffffffu, k ? rr.r[1].span_end : rr.r[0].span_end, src);
    rq.flags = __shfl_sync(0xffffffffu, k ? rr.r[1].flags : rr.r[0].flags, src);
    rq.pad_[0] = rq.pad_[1] = 0;
    return unit_geometry(a, rq, b, u);
}

// Work item `it` of the persistent loop: units 0..n_full-1 whole, then two
// halves of each remaining unit (key tiles [0, h) and [h, n), h = ceil(n/2)).
struct Item {
    Unit w;
    int half;           // -1: the whole unit
    int jb, je;         // key tiles of the item
};

// The producer warp computes each item's geometry once and publishes it in
// shared memory; the other roles read it there.  (Computed by every role, its
// request-table and argument reads -- kernel parameters or global memory,
// whose lines the K/V stream evicts from the caches -- held each role 2-4 us
// at every item boundary, all waiting on the same lines.)
// What the consumer roles read of an item.
struct Geo {
    int jb, je, half, n_tiles;
    int n_t[2], row0[2];
    int m_rows, q_len, prefix, q_off;
    int l, h, n_valid, cap;
    int span0, span_end;   // the request's spans (values-gathering variant)
    int tma_v, pad2_;      // prefix value tiles through TMA (values-gathering variant)
    int64_t kv_row0;
};
static_assert(sizeof(Geo) <= kGeoBytes, "geometry slot");

// (the span range and value mode only for the values-gathering variant: in
// the stitched one those request fields stay dead and cost no registers)
template <bool kV>
__device__ __forceinline__ void geo_of(const Item &t, Geo &o)
{
    o.jb = t.jb;
    o.je = t.je;
    o.half = t.half;
    o.n_tiles = t.w.n_tiles;
    o.n_t[0] = t.w.n_t[0];
    o.n_t[1] = t.w.n_t[1];
    o.row0[0] = t.w.row0[0];
    o.row0[1] = t.w.row0[1];
    o.m_rows = t.w.m_rows;
    o.q_len = t.w.rq.q_len;
    o.prefix = t.w.rq.prefix;
    o.q_off = t.w.rq.q_off;
    o.l = t.w.l;
    o.h = t.w.h;
    o.n_valid = t.w.n_valid;
    o.cap = t.w.rq.cap;
    if constexpr (kV) {
        o.span0 = t.w.rq.span0;
        o.span_end = t.w.rq.span_end;
        o.tma_v = (t.w.rq.flags & kReqValuesTma) != 0;
    }
    o.kv_row0 = t.w.kv_row0;
}
// the kernel's variants: K and V from the stitched cache; or K from the cache
// and the prefix values gathered from the pool; or the same for calls whose
// spans may also name request-local sources (the gather warps' row lookup
// then has a second kind of source)
constexpr int kModeStitched = 0, kModeGatherV = 1, kModeGatherVLocal = 2;
// softmax 8, MMA 1, and the two gather warps (values-gathering variants)
template <int kM>
constexpr uint32_t geo_consumer_warps() { return kM != kModeStitched ? 11u : 9u; }

// The value tile j of a values-gathering item that the gather warps fill: a
// tile that reaches past the cache block (into rows this variant does not
// write); and a tile with prefix rows -- every one for a request of short
// spans, only the one that also holds the first query rows for a request of
// long spans (`tma_v`: its other prefix tiles come from the pool through TMA
// box loads, whose runs of 32 consecutive pool rows move a tile in a few
// instructions).
__device__ __forceinline__ bool v_gathered(int j, int prefix, int cap, bool tma_v)
{
    const bool has_prefix = j * kTileN < prefix;
    return (j + 1) * kTileN > cap || (has_prefix && (!tma_v || prefix < (j + 1) * kTileN));
}

// `rr`: the producer warp's register copy of the request table (all 32
// lanes call with the same `it`), or NULL.
__device__ __forceinline__ Item item_at(const AttnArgs &a, const DevReq *reqs, int n_blocks, int it,
                                        const ReqRegs *rr = nullptr, int lane = 0)
{
    Item t;
    const int u = it < a.n_full ? it : a.n_full + ((it - a.n_full) >> 1);
    t.half = it < a.n_full ? -1 : ((it - a.n_full) & 1);
    t.w = (rr && rr->ok) ? unit_at_warp(a, *rr, u, lane) : unit_at(a, reqs, n_blocks, u);
    const int hs = (t.w.n_tiles + 1) >> 1;
    t.jb = t.half == 1 ? hs : 0;
    t.je = t.half == 0 ? hs : t.w.n_tiles;
    return t;
}

}  // namespace

template <int kM>
__global__ void __launch_bounds__(kThreads, 1)
    k_attention_tc(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ AttnArgs a,
                   const __grid_constant__ ReqTable rt, const int n_blocks,
                   const __grid_constant__ CUtensorMap tmpv, const __grid_constant__ CUtensorMap tmbv,
                   const __grid_constant__ GatherArgs g, const __grid_constant__ SpanTable st,
                   const __grid_constant__ CUtensorMap tmo)
{
    constexpr bool kV = kM != kModeStitched;
    constexpr bool kLocals = kM == kModeGatherVLocal;
    const DevReq *reqs = a.reqs ? a.reqs : rt.reqs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kOffBar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemAddr);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_units = n_blocks * (a.lh_count > 0 ? a.lh_count : a.n_layers * a.n_kv_heads);
    const int n_items = 2 * n_units - a.n_full;

    // geometry of this CTA's k-th item: slot k & 1 of the shared-memory ring
    auto geo_slot = [&](int k) { return reinterpret_cast<Geo *>(smem + kOffGeo + (k & 1) * kGeoBytes); };
    // consumer warps: wait for item k's geometry (then read its fields and
    // release the slot with geo_done)
    auto geo_wait = [&](int k) -> const Geo * {
        if (!mbar_wait(bar(kBarGeoFull + (k & 1)), (uint32_t)(k >> 1) & 1u, abort_flag))
            return nullptr;
        return geo_slot(k);
    };
    auto geo_done = [&](int k) {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar(kBarGeoEmpty + (k & 1)));
    };
    // producer (one thread): publish item k's geometry once its slot is free
    auto geo_put = [&](int k, const Item &gm) -> bool {
        if (k >= 2 && !mbar_wait(bar(kBarGeoEmpty + (k & 1)), (uint32_t)((k >> 1) - 1) & 1u, abort_flag))
            return false;
        geo_of<kV>(gm, *geo_slot(k));
        mbar_arrive(bar(kBarGeoFull + (k & 1)));   // release: the record is visible to the waiters
        return true;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool wg = (i >= kBarPFull && i < kBarPFull + 2) || (i >= kBarOEmpty && i < kBarOEmpty + 2) ||
                            i == kBarPeerData;
            const bool geo_empty = i >= kBarGeoEmpty && i < kBarGeoEmpty + 2;
            const bool gathered = i >= kBarGathered && i < kBarGathered + 2;
            mbar_init(bar(i), wg ? 128u : geo_empty ? geo_consumer_warps<kM>() : gathered ? 2u : 1u);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 9)
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    if (warp == 8 && lane == 0) {   // descriptors only: nothing the previous kernel writes
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        if constexpr (kV) {
            if (g.tma_pool) {
                prefetch_tmap(&tmpv);
                prefetch_tmap(&tmbv);
            }
        }
        if (a.out_tma)
            prefetch_tmap(&tmo);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();   // the partner CTA's barriers are initialised before any remote arrive
    const uint32_t tmem = *tmem_slot;
    // each role's branch starts by setting its warp's register count, for
    // whole warpgroups (0-1: softmax; 2: producer, MMA, patch or idle warps)
    auto regs_softmax = [] { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmaxS)); };
    auto regs_other = [] { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOtherS)); };
    // setup above overlaps the previous kernel's tail; its outputs (the
    // stitched cache, the rotated queries) are read only from here on
    pdl_wait_prerequisites();

    if (warp < 8) {
        regs_softmax();
        // =================== softmax / epilogue warpgroup of tile x ===================
        const int x = warp >> 2;
        const int r = threadIdx.x & 127;           // row of the tile = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float sc = a.scale_log2;
        const int G = a.n_q_heads / a.n_kv_heads;
        int s_cnt = 0, o_cnt = 0, gk = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++gk) {
            const Geo *gp = geo_wait(gk);
            if (!gp) {
                ok = false;
                break;
            }
            // the fields the key-tile loop needs; the epilogue reads the rest
            // from the slot afterwards (held until then: fewer live registers)
            const int jb = gp->jb;
            const int nx = min(gp->je, gp->n_t[x]);   // this tile's key tiles in the item: [jb, nx)
            if (jb >= nx) {
                geo_done(gk);
                continue;
            }
            const int rr = gp->row0[x] + r;        // packed row in the request
            const bool row_ok = rr < gp->m_rows;
            const int t = row_ok ? rr / G : gp->q_len - 1;
            const int g = row_ok ? rr - (rr / G) * G : 0;
            const int pos = gp->prefix + t;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = jb; j < nx; ++j) {
                if (!mbar_wait(bar(kBarSFull + x), s_cnt & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                ++s_cnt;
                tc_fence_after();
                float s[kTileN];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tmem_ld32(lane_base + col_s(x) + 32 * q, s + 32 * q);
                tmem_wait_ld();
                // key 128j + c is visible to this row iff c < lim
                const int lim = pos + 1 - j * kTileN;
                if (lim < kTileN) {
#pragma unroll
                    for (int c = 0; c < kTileN; ++c)
                        s[c] = (c < lim) ? s[c] : -INFINITY;
                }
                float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int c = 4; c < kTileN; c += 8) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        m4[k] = max3(m4[k], s[c + 2 * k], s[c + 2 * k + 1]);
                }
                const float mx = max3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
                const float mxs = mx * sc;
                // lazy max: keep m_run unless this tile's max exceeds it by more than
                // the threshold; O_x and l are rescaled after P_x is written (S is dead)
                float corr = 1.f;
                if (j == jb) {
                    m_run = mxs;
                } else if (mxs > m_run + kRescaleThreshold) {
                    corr = ex2(m_run - mxs);
                    m_run = mxs;
                }
                // a row that sees no key of the item's first tile sees none of
                // the item (p = 0 throughout, m stays -inf)
                const float nm = m_run == -INFINITY ? 0.f : -m_run;
                const uint64_t sc2 = pk2(sc, sc), nm2 = pk2(nm, nm);
                uint64_t acc[2] = {pk2(0.f, 0.f), pk2(0.f, 0.f)};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float x0, x1;
                        unpk2(fma2(pk2(s[32 * q + 2 * i], s[32 * q + 2 * i + 1]), sc2, nm2), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        acc[i & 1] = add2(acc[i & 1], pk2(p0, p1));
                        pk[i] = pack_bf16(p0, p1);
                    }
                    tmem_st16(lane_base + col_s(x) + 16 * q, pk);
                }
                float sum;
                {
                    float a0, a1, b0, b1;
                    unpk2(acc[0], a0, a1);
                    unpk2(acc[1], b0, b1);
                    sum = (a0 + a1) + (b0 + b1);
                }
                l_run = l_run * corr + sum;
                if (corr != 1.f) {
                    // the commit that signalled S_x(j) covers PV_x(j-1): O_x is stable
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float o[32];
                        tmem_ld32(lane_base + col_o(x) + 32 * q, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] *= corr;
                        tmem_st32(lane_base + col_o(x) + 32 * q, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(kBarPFull + x));
            }
            if (!ok)
                break;
            const int half = gp->half, n_tiles = gp->n_tiles, ntx = gp->n_t[x], row0x = gp->row0[x];
            const int m_rows = gp->m_rows, q_off = gp->q_off, wl = gp->l, wh = gp->h;
            geo_done(gk);
            // epilogue: O / l -> bf16 -> out[l][q_off + t][h*G + g][:], read from
            // TMEM 64 columns at a time (a whole row of O in registers spills)
            if (!mbar_wait(bar(kBarOFull + x), o_cnt & 1, abort_flag)) {
                ok = false;
                break;
            }
            ++o_cnt;
            tc_fence_after();
            const uint32_t o_tm = lane_base + col_o(x);
            float l_fin = l_run;
            // a split unit whose second half reaches this tile: the two halves run
            // on the two CTAs of a cluster (half h on rank h), and rank x merges
            // tile x, half 0 first (one rounding order); the other CTA sends its
            // half of tile x through distributed shared memory, O as fp16 with a
            // power-of-two scale per row (exact to ~2^-12, below the output's bf16
            // rounding, at half the bytes of fp32).  Nothing of it touches L2.
            const bool split2 = half >= 0 && (n_tiles + 1) / 2 < ntx;
            const bool merger = split2 && half == x;
            const uint32_t peer_o = sbase + kOffPeerO, peer_ml = sbase + kOffPeerML;
            if (split2 && !merger) {
                // the partner's ring and Q tiles are free once its MMAs are done
                if (!mbar_wait_cluster(bar(kBarPeerFree), 0, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t peer = (uint32_t)x;
                float amax = 0.f;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float f[64];
                    tmem_ld32(o_tm + 64 * hh, f);
                    tmem_ld32(o_tm + 64 * hh + 32, f + 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        amax = fmaxf(amax, fabsf(f[e]));
                }
                // scale 2^k with amax / 2^k in [2^14, 2^15): no fp16 overflow
                const int be = (__float_as_int(amax) >> 23) & 0xff;
                const int se = be >= 15 ? be - 14 : 1;
                const float scale = __int_as_float(se << 23), inv_scale = __int_as_float((254 - se) << 23);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float f[64];
                    tmem_ld32(o_tm + 64 * hh, f);
                    tmem_ld32(o_tm + 64 * hh + 32, f + 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t hw[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const __half2 h2 = __floats2half2_rn(f[8 * c + 2 * q] * inv_scale, f[8 * c + 2 * q + 1] * inv_scale);
                            hw[q] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        st_cluster_v4(mapa_rank(peer_o + (uint32_t)(((8 * hh + c) * kTileM + r) * 16), peer),
                                      __uint_as_float(hw[0]), __uint_as_float(hw[1]), __uint_as_float(hw[2]),
                                      __uint_as_float(hw[3]));
                    }
                }
                st_cluster_f32(mapa_rank(peer_ml + (uint32_t)r * 4, peer), m_run);
                st_cluster_f32(mapa_rank(peer_ml + (uint32_t)(kTileM + r) * 4, peer), l_run);
                st_cluster_f32(mapa_rank(peer_ml + (uint32_t)(2 * kTileM + r) * 4, peer), scale);
                mbar_arrive_remote(mapa_rank(bar(kBarPeerData), peer));
                tc_fence_before();
                mbar_arrive(bar(kBarOEmpty + x));
                continue;
            }
            float w0 = 1.f, w1 = 0.f, p_scale = 0.f;
            if (merger) {
                if (!mbar_wait_cluster(bar(kBarPeerData), 0, abort_flag)) {
                    ok = false;
                    break;
                }
                const float mp = ld_shared_f32(peer_ml + (uint32_t)r * 4);
                const float lp = ld_shared_f32(peer_ml + (uint32_t)(kTileM + r) * 4);
                p_scale = ld_shared_f32(peer_ml + (uint32_t)(2 * kTileM + r) * 4);
                const float m0 = x == 0 ? m_run : mp, m1 = x == 0 ? mp : m_run;   // halves 0 and 1
                const float M = fmaxf(m0, m1);     // m0 is finite: every row sees key 0
                w0 = ex2(m0 - M);
                w1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
                l_fin = __fmaf_rn(x == 0 ? lp : l_run, w1, __fmul_rn(x == 0 ? l_run : lp, w0));
            }
            const float inv = row_ok ? 1.f / l_fin : 0.f;
            // a NaN or infinity among the row's query or key elements leaves no
            // finite positive denominator: report it (the row is written as computed)
            if (row_ok && !(l_fin > 0.f && l_fin < INFINITY))
                atomicCAS(a.err, kDevOk, kDevBadInput);
            // this warp's 32 rows are whole tokens of the request: one TMA store
            // per 64-column half, and the warp does not wait for global memory
            const int wrow0 = row0x + (warp & 3) * 32;
            const bool tma_out = a.out_tma && wrow0 + 31 < m_rows;
            // TMA stores: the box's (head, token) coordinates; otherwise this
            // row's output element offset (-1: no row)
            const int64_t orow = tma_out ? (((int64_t)(wh * G) << 32) | (uint32_t)(wl * a.total_q + q_off + wrow0 / G))
                                 : row_ok ? (((int64_t)wl * a.total_q + q_off + t) * a.n_q_heads + wh * G + g) * kD
                                          : -1;
            __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
            const uint32_t stg = sbase + kOffStage + (uint32_t)warp * 32 * 128;
            const int wr = r & 31;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float f[64];
                tmem_ld32(o_tm + 64 * hh, f);
                tmem_ld32(o_tm + 64 * hh + 32, f + 32);
                tmem_wait_ld();
                if (a.out_tma) {   // the staging is free once the last TMA store has read it
                    if (lane == 0)
                        bulk_wait_read();
                    __syncwarp();
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        v[e] = f[8 * c + e];
                    if (merger) {
                        // half-0 value times w0 plus half-1 value times w1
                        const uint4 u = ld_shared_v4(peer_o + (uint32_t)(((8 * hh + c) * kTileM + r) * 16));
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 pv = __half22float2(*reinterpret_cast<const __half2 *>(&uw[q]));
                            const float p0 = pv.x * p_scale, p1 = pv.y * p_scale;
                            if (x == 0) {
                                v[2 * q] = __fmaf_rn(p0, w1, __fmul_rn(v[2 * q], w0));
                                v[2 * q + 1] = __fmaf_rn(p1, w1, __fmul_rn(v[2 * q + 1], w0));
                            } else {
                                v[2 * q] = __fmaf_rn(v[2 * q], w1, __fmul_rn(p0, w0));
                                v[2 * q + 1] = __fmaf_rn(v[2 * q + 1], w1, __fmul_rn(p1, w0));
                            }
                        }
                    }
                    st_shared_v4(stg + wr * 128 + ((c ^ (wr & 7)) << 4), pack_bf16(v[0] * inv, v[1] * inv),
                                 pack_bf16(v[2] * inv, v[3] * inv), pack_bf16(v[4] * inv, v[5] * inv),
                                 pack_bf16(v[6] * inv, v[7] * inv));
                }
                if (tma_out) {
                    // the staging is the box's 128B-swizzled layout: rows t * G + g
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tmo, stg, 64 * hh, (int)(orow >> 32), (int)(uint32_t)orow);
                        bulk_commit();
                    }
                } else {
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int row = 4 * i + (lane >> 3), c = lane & 7;
                        const int64_t base = __shfl_sync(0xffffffffu, orow, row);
                        const uint4 v = ld_shared_v4(stg + row * 128 + ((c ^ (row & 7)) << 4));
                        if (base >= 0)
                            *reinterpret_cast<uint4 *>(out + base + 64 * hh + 8 * c) = v;
                    }
                    __syncwarp();
                }
            }
            // the output is staged and stored: O_x and the shared memory may
            // take the next item's MMAs
            tc_fence_before();
            mbar_arrive(bar(kBarOEmpty + x));
        }
        if (a.out_tma && lane == 0)
            bulk_wait_all();   // every output store has landed before the CTA ends
        if (!ok)
            flag_timeout(a.err, abort_flag);
    } else if (warp == 8) {
        regs_other();
        if constexpr (kV) {
            // ====== values-gathering producer: Q, the K tiles and the V tiles
            // past the prefix as in the stitched variant (lane 0); a request of
            // long spans has its other prefix value tiles loaded from the pool
            // here (lane i: rows 4i..4i+3, resolved through the span table; a
            // group of 8 lanes whose 32 rows are consecutive pool rows takes one
            // 32-row box load per panel, other lanes a gather4 each); a V tile
            // that the gather warps fill (v_gathered) is announced to them once
            // its ring slot is free ======
            int tt = 0, nq = 0, gk = 0;
            bool ok = true;
            const DevSpan *spans = g.spans ? g.spans : st.spans;
            const int64_t e_rows = (int64_t)a.n_layers * a.n_kv_heads * g.entry_len;   // pool rows per entry
            ReqRegs rr;
            rr.load(a, reqs, lane);
            Item nxt;
            if ((int)blockIdx.x < n_items) {
                nxt = item_at(a, reqs, n_blocks, blockIdx.x, &rr, lane);
                if (lane == 0)
                    ok = geo_put(0, nxt);
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++gk) {
                const Item itm = nxt;
                const Unit &w = itm.w;
                const bool more = it + (int)gridDim.x < n_items;
                if (more && gk > 0)
                    nxt = item_at(a, reqs, n_blocks, it + gridDim.x, &rr, lane);
                const bool tma_v = (w.rq.flags & kReqValuesTma) != 0;
                if (itm.je > itm.jb && !tma_v && lane == 0) {
                    // a request of short spans: lane 0 alone, as in the stitched variant
                    const int n_loads = 2 * (itm.je - itm.jb);
                    for (int i = 0; i <= n_loads && ok; ++i) {
                        if (i == 2) {
                            if (nq > 0 && !mbar_wait(bar(kBarQEmpty), (nq - 1) & 1, abort_flag)) {
                                ok = false;
                                break;
                            }
                            const int nqt = w.n_t[1] > 0 ? 2 : 1;
                            mbar_expect_tx(bar(kBarQFull), nqt * kTileBytes);
                            for (int x = 0; x < nqt; ++x) {
                                const uint32_t dst = sbase + kOffQ + x * kTileBytes;
                                tma_load_2d(dst, &tmq, 0, w.q_row0 + x * kTileM, bar(kBarQFull));
                                tma_load_2d(dst + kPanelBytes, &tmq, 64, w.q_row0 + x * kTileM, bar(kBarQFull));
                            }
                            ++nq;
                        }
                        if (i == n_loads)
                            break;
                        const int slot = tt % kSlots;
                        if (tt >= kSlots && !mbar_wait(bar(kBarEmpty + slot), ((tt / kSlots) - 1) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const int j = itm.jb + (i >> 1);
                        if ((i & 1) == 1 && v_gathered(j, w.rq.prefix, w.rq.cap, false)) {
                            mbar_arrive(bar(kBarFull + slot));
                            mbar_arrive(bar(kBarGatherJob + (slot >> 1)));
                        } else {
                            const uint32_t dst = sbase + kOffKV + slot * kTileBytes;
                            const CUtensorMap *map = (i & 1) ? &tmv : &tmk;
                            const int row = (int)(w.kv_row0 + (int64_t)j * kTileN);
                            mbar_expect_tx(bar(kBarFull + slot), kTileBytes);
                            tma_load_2d(dst, map, 0, row, bar(kBarFull + slot));
                            tma_load_2d(dst + kPanelBytes, map, 64, row, bar(kBarFull + slot));
                        }
                        ++tt;
                    }
                } else if (itm.je > itm.jb && tma_v) {
                    const int prefix = w.rq.prefix, cap = w.rq.cap, s_end = w.rq.span_end;
                    const int64_t lh_row = (int64_t)w.lh * g.entry_len;   // (layer, kv-head) block inside an entry
                    // the span holding the item's first row; each lane's cursor
                    // then only moves forward
                    int cur = w.rq.span0;
                    if (tma_v && itm.jb * kTileN < prefix) {
                        int lo = w.rq.span0, hi = s_end - 1;
                        while (lo < hi) {
                            const int mid = (lo + hi + 1) >> 1;
                            if (spans[mid].row <= itm.jb * kTileN)
                                lo = mid;
                            else
                                hi = mid - 1;
                        }
                        cur = lo;
                    }
                    const int n_loads = 2 * (itm.je - itm.jb);
                    int rows[4] = {0, 0, 0, 0};
                    bool run32 = false;   // this lane's 32-row group is 32 consecutive pool rows
                    for (int i = 0; i <= n_loads; ++i) {
                        if (i == 2 && lane == 0) {   // Q after K_0 and V_0, as in the stitched variant
                            if (nq > 0 && !mbar_wait(bar(kBarQEmpty), (nq - 1) & 1, abort_flag)) {
                                ok = false;
                            } else {
                                const int nqt = w.n_t[1] > 0 ? 2 : 1;
                                mbar_expect_tx(bar(kBarQFull), nqt * kTileBytes);
                                for (int x = 0; x < nqt; ++x) {
                                    const uint32_t dst = sbase + kOffQ + x * kTileBytes;
                                    tma_load_2d(dst, &tmq, 0, w.q_row0 + x * kTileM, bar(kBarQFull));
                                    tma_load_2d(dst + kPanelBytes, &tmq, 64, w.q_row0 + x * kTileM, bar(kBarQFull));
                                }
                            }
                        }
                        if (i == 2)
                            ++nq;
                        if (i == n_loads)
                            break;
                        const int slot = tt % kSlots;
                        if (lane == 0 && ok && tt >= kSlots &&
                            !mbar_wait(bar(kBarEmpty + slot), ((tt / kSlots) - 1) & 1, abort_flag))
                            ok = false;
                        if (!(ok = __shfl_sync(0xffffffffu, ok, 0)))
                            break;
                        const int j = itm.jb + (i >> 1);
                        const uint32_t dst = sbase + kOffKV + slot * kTileBytes;
                        const bool v = (i & 1) == 1;
                        if (v && v_gathered(j, prefix, cap, tma_v)) {
                            // the slot's full barrier still completes a phase for this
                            // load (its parity then stays the load count's), with no bytes
                            if (lane == 0) {
                                mbar_arrive(bar(kBarFull + slot));
                                mbar_arrive(bar(kBarGatherJob + (slot >> 1)));
                            }
                        } else if (v && j * kTileN < prefix) {
                            // a long-span request's prefix value tile, from the pool
                            if (lane == 0)
                                mbar_expect_tx(bar(kBarFull + slot), kTileBytes);
                            __syncwarp();
                            const uint32_t d4 = dst + (uint32_t)(4 * lane) * 128u;
                            if (run32) {
                                if ((lane & 7) == 0) {
                                    tma_load_2d(d4, &tmbv, 0, rows[0], bar(kBarFull + slot));
                                    tma_load_2d(d4 + kPanelBytes, &tmbv, 64, rows[0], bar(kBarFull + slot));
                                }
                            } else {
                                tma_gather4(d4, &tmpv, 0, rows, bar(kBarFull + slot));
                                tma_gather4(d4 + kPanelBytes, &tmpv, 64, rows, bar(kBarFull + slot));
                            }
                        } else if (lane == 0) {
                            // a K tile, or a V tile past the prefix: the cache block's rows
                            const CUtensorMap *map = v ? &tmv : &tmk;
                            const int row = (int)(w.kv_row0 + (int64_t)j * kTileN);
                            mbar_expect_tx(bar(kBarFull + slot), kTileBytes);
                            tma_load_2d(dst, map, 0, row, bar(kBarFull + slot));
                            tma_load_2d(dst + kPanelBytes, map, 64, row, bar(kBarFull + slot));
                        }
                        // after K tile j: the pool rows of V tile j, if the producer loads it
                        if (!v && tma_v && j * kTileN < prefix && !v_gathered(j, prefix, cap, tma_v)) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int r = j * kTileN + 4 * lane + k;
                                while (cur + 1 < s_end && spans[cur].row + spans[cur].len <= r)
                                    ++cur;
                                const DevSpan &sp = spans[cur];
                                rows[k] = (int)((int64_t)sp.src * e_rows + lh_row + sp.start + (r - sp.row));
                            }
                            const int last = __shfl_up_sync(0xffffffffu, rows[3], 1);
                            const bool mine = rows[1] == rows[0] + 1 && rows[2] == rows[0] + 2 &&
                                              rows[3] == rows[0] + 3 && ((lane & 7) == 0 || rows[0] == last + 1);
                            const unsigned ball = __ballot_sync(0xffffffffu, mine);
                            run32 = ((ball >> (lane & ~7)) & 0xffu) == 0xffu;
                        }
                        ++tt;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                tt = __shfl_sync(0xffffffffu, tt, 0);
                nq = __shfl_sync(0xffffffffu, nq, 0);
                // the next item's geometry, published for the other roles; its Q
                // brought into L2 ahead of its load
                if (ok && more) {
                    if (gk == 0)
                        nxt = item_at(a, reqs, n_blocks, it + gridDim.x, &rr, lane);
                    if (lane == 0) {
                        ok = geo_put(gk + 1, nxt);
                        if (ok && nxt.je > nxt.jb)
                            for (int x = 0; x < (nxt.w.n_t[1] > 0 ? 2 : 1); ++x) {
                                tma_prefetch_2d(&tmq, 0, nxt.w.q_row0 + x * kTileM);
                                tma_prefetch_2d(&tmq, 64, nxt.w.q_row0 + x * kTileM);
                            }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                }
            }
            if (lane == 0) {
                if (!ok)
                    flag_timeout(a.err, abort_flag);
                // drain: every issued copy lands before the CTA leaves
                const uint64_t t0 = globaltimer();
                for (int k = (tt > kSlots ? tt - kSlots : 0); k < tt; ++k)
                    while (!mbar_try_wait(bar(kBarFull + k % kSlots), (k / kSlots) & 1) &&
                           globaltimer() - t0 < kWaitNs) {
                    }
                if (nq > 0)
                    while (!mbar_try_wait(bar(kBarQFull), (nq - 1) & 1) && globaltimer() - t0 < kWaitNs) {
                    }
            }
        } else {
            // ====== stitched producer: the whole warp computes each item's
            // geometry (request table in registers), lane 0 waits and issues ======
            int tt = 0, nq = 0, gk = 0;
            bool ok = true;
            ReqRegs rr;
            rr.load(a, reqs, lane);
            Item nxt;
            if ((int)blockIdx.x < n_items) {
                nxt = item_at(a, reqs, n_blocks, blockIdx.x, &rr, lane);
                if (lane == 0)
                    ok = geo_put(0, nxt);
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++gk) {
                const Item itm = nxt;
                const Unit &w = itm.w;
                // the next item's geometry now, while this item's first loads wait
                // for ring slots -- except on the first item, whose loads go
                // first (nothing else can start before them)
                const bool more = it + (int)gridDim.x < n_items;
                if (more && gk > 0)
                    nxt = item_at(a, reqs, n_blocks, it + gridDim.x, &rr, lane);
                if (itm.je > itm.jb && lane == 0) {
                    // K_0 and V_0 first (their ring slots free up a tile before the
                    // previous item ends), then Q (its buffer frees only once the
                    // previous item's last S MMAs are done), then the other tiles
                    const int n_loads = 2 * (itm.je - itm.jb);
                    for (int i = 0; i <= n_loads && ok; ++i) {
                        if (i == 2) {
                            if (nq > 0 && !mbar_wait(bar(kBarQEmpty), (nq - 1) & 1, abort_flag)) {
                                ok = false;
                                break;
                            }
                            const int nqt = w.n_t[1] > 0 ? 2 : 1;
                            mbar_expect_tx(bar(kBarQFull), nqt * kTileBytes);
                            for (int x = 0; x < nqt; ++x) {
                                const uint32_t dst = sbase + kOffQ + x * kTileBytes;
                                tma_load_2d(dst, &tmq, 0, w.q_row0 + x * kTileM, bar(kBarQFull));
                                tma_load_2d(dst + kPanelBytes, &tmq, 64, w.q_row0 + x * kTileM, bar(kBarQFull));
                            }
                            ++nq;
                        }
                        if (i == n_loads)
                            break;
                        const int slot = tt % kSlots;
                        if (tt >= kSlots && !mbar_wait(bar(kBarEmpty + slot), ((tt / kSlots) - 1) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = sbase + kOffKV + slot * kTileBytes;
                        const CUtensorMap *map = (i & 1) ? &tmv : &tmk;
                        const int row = (int)(w.kv_row0 + (int64_t)(itm.jb + (i >> 1)) * kTileN);
                        mbar_expect_tx(bar(kBarFull + slot), kTileBytes);
                        tma_load_2d(dst, map, 0, row, bar(kBarFull + slot));
                        tma_load_2d(dst + kPanelBytes, map, 64, row, bar(kBarFull + slot));
                        ++tt;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                tt = __shfl_sync(0xffffffffu, tt, 0);
                nq = __shfl_sync(0xffffffffu, nq, 0);
                // the next item's geometry, published for the other roles; its Q
                // and its first K and V tiles brought into L2 ahead of their loads
                // (the whole grid reaches its item boundaries at about the same
                // time, and those loads would queue together; the other K/V tiles
                // are not prefetched: their loads are issued a tile ahead anyway,
                // and a prefetch costs the SM's TMA unit as much time as the load
                // that follows it)
                if (ok && more) {
                    if (gk == 0)
                        nxt = item_at(a, reqs, n_blocks, it + gridDim.x, &rr, lane);
                    if (lane == 0) {
                        ok = geo_put(gk + 1, nxt);
                        if (ok && nxt.je > nxt.jb)
                            for (int x = 0; x < (nxt.w.n_t[1] > 0 ? 2 : 1); ++x) {
                                tma_prefetch_2d(&tmq, 0, nxt.w.q_row0 + x * kTileM);
                                tma_prefetch_2d(&tmq, 64, nxt.w.q_row0 + x * kTileM);
                            }
                        if (ok && nxt.je > nxt.jb) {
                            const int krow = (int)(nxt.w.kv_row0 + (int64_t)nxt.jb * kTileN);
                            tma_prefetch_2d(&tmk, 0, krow);
                            tma_prefetch_2d(&tmk, 64, krow);
                            tma_prefetch_2d(&tmv, 0, krow);
                            tma_prefetch_2d(&tmv, 64, krow);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                }
            }
            if (lane == 0) {
                if (!ok)
                    flag_timeout(a.err, abort_flag);
                // drain: every issued copy lands before the CTA leaves
                const uint64_t t0 = globaltimer();
                for (int k = (tt > kSlots ? tt - kSlots : 0); k < tt; ++k)
                    while (!mbar_try_wait(bar(kBarFull + k % kSlots), (k / kSlots) & 1) &&
                           globaltimer() - t0 < kWaitNs) {
                    }
                if (nq > 0)
                    while (!mbar_try_wait(bar(kBarQFull), (nq - 1) & 1) && globaltimer() - t0 < kWaitNs) {
                    }
            }
        }
    } else if (warp == 9) {
        regs_other();
        // =================== MMA issuer ===================
        {
            const uint32_t lead = elect_one();
            int tt = 0, nq = 0;
            int p_cnt[2] = {0, 0}, oe_cnt[2] = {0, 0};
            bool o_used[2] = {false, false};
            int peer_wait = -1;   // the last item is half h of a split unit whose tile h the other half reaches
            bool ok = true;
            // descriptors: K-major 128B-swizzled tiles (Q, K) and the MN-major V tile
            const uint64_t d_k_major = sdesc(sbase, 16, 1024);
            const uint64_t d_mn_major = sdesc(sbase, kPanelBytes, 1024);
            const uint32_t lo_k = (uint32_t)d_k_major, hi_k = (uint32_t)(d_k_major >> 32);
            const uint32_t lo_v = (uint32_t)d_mn_major, hi_v = (uint32_t)(d_mn_major >> 32);
            // S_x = Q_x K^T with K in ring slot `slot`
            auto issue_s = [&](int x, int slot) {
                const uint32_t qa = lo_k + ((kOffQ + x * kTileBytes) >> 4);
                const uint32_t kb = lo_k + ((kOffKV + slot * kTileBytes) >> 4);
                const uint32_t d = tmem + col_s(x);
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t off = ((k >> 2) * kPanelBytes + (k & 3) * 32) >> 4;
                    if (k == 0)
                        mma_ss<false>(lead, d, desc_with_lo(qa + off, hi_k), desc_with_lo(kb + off, hi_k), kIdescS);
                    else
                        mma_ss<true>(lead, d, desc_with_lo(qa + off, hi_k), desc_with_lo(kb + off, hi_k), kIdescS);
                }
                umma_commit(lead, bar(kBarSFull + x));
            };
            auto wait_kv = [&](int k) -> bool {
                if (!mbar_wait(bar(kBarFull + k % kSlots), (k / kSlots) & 1, abort_flag))
                    return false;
                tc_fence_after();
                return true;
            };
            // values-gathering variant: a gathered V tile is complete once both
            // gather warps have released it
            int np[2] = {0, 0}, prefix_v = 0, cap_v = 0;
            bool tma_v = false;
            auto wait_v = [&](int k, int j) -> bool {
                if constexpr (kV) {
                    if (v_gathered(j, prefix_v, cap_v, tma_v)) {
                        const int b = (k % kSlots) >> 1;   // V tiles sit in slots 1 and 3
                        if (!mbar_wait(bar(kBarGathered + b), np[b] & 1, abort_flag))
                            return false;
                        ++np[b];
                        tc_fence_after();
                        return true;
                    }
                }
                return wait_kv(k);
            };
            int gk = 0;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++gk) {
                const Geo *gp = geo_wait(gk);
                if (!gp) {
                    ok = false;
                    break;
                }
                const int jb = gp->jb, je = gp->je, half = gp->half, n_tiles = gp->n_tiles;
                const int nt0 = gp->n_t[0], nt1 = gp->n_t[1];
                if constexpr (kV) {
                    prefix_v = gp->prefix;
                    cap_v = gp->cap;
                    tma_v = gp->tma_v != 0;
                }
                geo_done(gk);
                if (je <= jb)
                    continue;
                const int jx[2] = {min(je, nt0), min(je, nt1)};   // tile x's key tiles: [jb, jx[x])
                peer_wait = half >= 0 && (n_tiles + 1) / 2 < (half ? nt1 : nt0) ? half : -1;
                if (!mbar_wait(bar(kBarQFull), nq & 1, abort_flag) || !wait_kv(tt)) {
                    ok = false;
                    break;
                }
                ++nq;
                // a tile's first S of the item waits until the epilogue of its
                // previous item is done (O read, staged and stored): this MMA
                // reads both operands from shared memory, at the bandwidth the
                // epilogue's staging stores also need; its PV MMAs, which
                // overwrite O, come later still
                for (int x = 0; x < 2 && ok; ++x)
                    if (jb < jx[x]) {
                        if (o_used[x]) {
                            if (!mbar_wait(bar(kBarOEmpty + x), oe_cnt[x] & 1, abort_flag)) {
                                ok = false;
                                break;
                            }
                            ++oe_cnt[x];
                            o_used[x] = false;
                        }
                        issue_s(x, tt % kSlots);
                    }
                if (!ok)
                    break;
                if (je - jb == 1)
                    umma_commit(lead, bar(kBarQEmpty));
                umma_commit(lead, bar(kBarEmpty + tt % kSlots));
                for (int j = jb; j < je && ok; ++j) {
                    const int i = j - jb;
                    const int tv = tt + 2 * i + 1, tk = tt + 2 * i + 2;
                    const uint32_t vb = lo_v + ((kOffKV + (tv % kSlots) * kTileBytes) >> 4);
                    bool v_ready = false, k_ready = false;
                    for (int x = 0; x < 2; ++x) {
                        if (j >= jx[x])
                            continue;
                        if (!mbar_wait(bar(kBarPFull + x), p_cnt[x] & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        ++p_cnt[x];
                        if (!v_ready && !(v_ready = wait_v(tv, j))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d = tmem + col_o(x), pa = tmem + col_s(x);
                        const uint32_t acc0 = j > jb;
#pragma unroll
                        for (int k = 0; k < kTileN / 16; ++k)
                            mma_ts(lead, d, pa + 8 * k, desc_with_lo(vb + ((k * 2048) >> 4), hi_v), kIdescPV,
                                   k > 0 ? 1u : acc0);
                        if (j + 1 == jx[x]) {
                            umma_commit(lead, bar(kBarOFull + x));
                            o_used[x] = true;
                        } else {
                            if (!k_ready && !(k_ready = wait_kv(tk))) {
                                ok = false;
                                break;
                            }
                            issue_s(x, tk % kSlots);
                        }
                    }
                    if (!ok)
                        break;
                    if (k_ready && j + 2 == je)
                        umma_commit(lead, bar(kBarQEmpty));   // the item's last S MMAs are issued
                    umma_commit(lead, bar(kBarEmpty + tv % kSlots));
                    if (k_ready)
                        umma_commit(lead, bar(kBarEmpty + tk % kSlots));
                }
                tt += 2 * (je - jb);
            }
            if (!ok)
                flag_timeout(a.err, abort_flag);
            // drain: all issued MMAs complete before TMEM is released
            umma_commit(lead, bar(kBarDrain));
            const uint64_t t0 = globaltimer();
            bool drained = false;
            while (!(drained = mbar_try_wait(bar(kBarDrain), 0)) && globaltimer() - t0 < kWaitNs) {
            }
            // a split unit whose tile (this CTA's rank) the partner's half reaches:
            // the partner may now write its half over this CTA's K/V ring and Q tiles
            if (ok && drained && peer_wait >= 0 && lane == 0)
                mbar_arrive_remote(mapa_rank(bar(kBarPeerFree), (uint32_t)(1 - peer_wait)));
        }
    } else if (kV && warp >= 10) {
        regs_other();
        // ========== gather (values-gathering variant, warps 10-11) ==========
        // Each V tile that v_gathered names (for a request of short spans every
        // tile with prefix rows; for one of long spans the tile that also holds
        // the first query rows; and any tile that reaches past its cache block,
        // whose value rows this variant does not write) is filled here with
        // 16-byte asynchronous copies: prefix rows from the pool
        // (resolved through the span table), query rows from the cache block
        // (the query prologue appended them there), zeros past the request's
        // keys (a masked key has weight 0, but 0 x NaN is NaN).  Warp 10 takes
        // rows 0-63 of the tile, warp 11 rows 64-127; lane l resolves rows
        // 2l and 2l + 1 of its warp's half, and in copy i the warp moves rows
        // 2i and 2i + 1 (lanes 0-15 and 16-31, one 16-byte chunk each of the
        // two 64-column panels' 8).  A tile's copies are one group; the tile
        // is released to the MMA warp once the next tile's copies are issued
        // and its own have landed, or before waiting for any tile but the
        // very next one.
        const int rb = 64 * (warp - 10);
        const int q16 = lane & 15, half_sel = lane >> 4;
        const uint32_t chunk_off = (uint32_t)((q16 >> 3) * kPanelBytes);
        const int c8 = q16 & 7;
        const DevSpan *spans = g.spans ? g.spans : st.spans;
        const __nv_bfloat16 *pv = static_cast<const __nv_bfloat16 *>(g.pool_v);
        const __nv_bfloat16 *cv = static_cast<const __nv_bfloat16 *>(a.cache_v);
        int tt = 0, gk = 0, nj[2] = {0, 0}, prev_b = -1, prev_j = -1;
        bool ok = true;
        // release the tile whose copies were issued last (all of this thread's
        // copies land first, then the async proxy sees them)
        auto release = [&](int wait_all) {
            if (prev_b < 0)
                return;
            if (wait_all)
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            else
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(kBarGathered + prev_b));
            prev_b = -1;
        };
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++gk) {
            int jb, je, prefix, n_valid, cap, l, h, s0, s_end;
            bool tma_v;
            int64_t kv_row0;
            {
                const Geo *gp = geo_wait(gk);
                if (!gp) {
                    ok = false;
                    break;
                }
                jb = gp->jb;
                je = gp->je;
                prefix = gp->prefix;
                n_valid = gp->n_valid;
                cap = gp->cap;
                kv_row0 = gp->kv_row0;
                l = gp->l;
                h = gp->h;
                s0 = gp->span0;
                s_end = gp->span_end;
                tma_v = gp->tma_v != 0;
                geo_done(gk);
            }
            // this lane's span cursor: the span holding its first prefix row of
            // the item (a request's spans are in stitched-row order)
            int cur = s0;
            {
                const int r0 = jb * kTileN + rb + 2 * lane;
                if (r0 < prefix) {
                    int lo = s0, hi = s_end - 1;
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (spans[mid].row <= r0)
                            lo = mid;
                        else
                            hi = mid - 1;
                    }
                    cur = lo;
                }
            }
            for (int j = jb; j < je && ok; ++j, tt += 2) {
                if (!v_gathered(j, prefix, cap, tma_v))
                    continue;
                // the source of this lane's two rows (0: zeros)
                const __nv_bfloat16 *src[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int r = j * kTileN + rb + 2 * lane + k;
                    src[k] = nullptr;
                    if (r < prefix) {
                        while (cur + 1 < s_end && spans[cur].row + spans[cur].len <= r)
                            ++cur;
                        const DevSpan &sp = spans[cur];
                        const int64_t tok = sp.start + (r - sp.row);
                        if (kLocals && (sp.src & KVR_SRC_LOCAL)) {   // a request-local source
                            const DevLocal &lc = g.locals[sp.src & ~KVR_SRC_LOCAL];
                            src[k] = static_cast<const __nv_bfloat16 *>(lc.v) + l * lc.s_layer + h * lc.s_head +
                                     tok * lc.s_tok;
                        } else {
                            src[k] = pv + sp.src * g.ps_entry + l * g.ps_layer + h * g.ps_head + tok * g.ps_tok;
                        }
                    } else if (r < n_valid) {
                        src[k] = cv + (kv_row0 + r) * kD;
                    }
                }
                const int sv = (tt + 1) % kSlots, b = sv >> 1;
                // a tile held back that is not the one just before this: the MMAs
                // reach this tile's slot only after consuming it (and the tiles
                // the producer loads in between), so release it first
                if (prev_b >= 0 && j != prev_j + 1)
                    release(1);
                if (!mbar_wait(bar(kBarGatherJob + b), nj[b] & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                ++nj[b];
                const uint32_t vb = sbase + kOffKV + sv * kTileBytes + chunk_off;
#pragma unroll 4
                for (int i = 0; i < 32; ++i) {
                    const __nv_bfloat16 *s_lo = (const __nv_bfloat16 *)__shfl_sync(0xffffffffu, (uintptr_t)src[0], i);
                    const __nv_bfloat16 *s_hi = (const __nv_bfloat16 *)__shfl_sync(0xffffffffu, (uintptr_t)src[1], i);
                    const __nv_bfloat16 *sp = half_sel ? s_hi : s_lo;
                    const int r = rb + 2 * i + half_sel;   // row of the tile
                    cp_async16_zfill(vb + r * 128 + ((c8 ^ (r & 7)) << 4),
                                     sp ? sp + (q16 >> 3) * 64 + 8 * c8 : cv, sp ? 16 : 0);
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                release(0);
                prev_b = b;
                prev_j = j;
            }
            release(1);
        }
        release(1);
        if (!ok)
            flag_timeout(a.err, abort_flag);
    } else {
        regs_other();   // warps 10-11 (stitched) or 11 (values gathered): no role
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no CTA leaves while its partner may still touch its shared memory
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

bool attention_tc_supported(int dtype, int head_dim) { return dtype == KVR_DTYPE_BF16 && head_dim == kD; }

template <int kM>
static cudaError_t set_smem_attr()
{
    // the shared-memory opt-in is per device and per kernel (callers on
    // several host threads may both set it: the same value)
    static std::atomic<bool> attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
        {
            // the register split (setmaxnreg) must fit what the CTA is launched
            // with, or the softmax warpgroups' increase would wait forever
            cudaFuncAttributes fa{};
            if ((e = cudaFuncGetAttributes(&fa, k_attention_tc<kM>)) != cudaSuccess)
                return e;
            if (fa.numRegs != kRegsLaunchS)
                return cudaErrorInvalidConfiguration;
        }
        e = cudaFuncSetAttribute(k_attention_tc<kM>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            attr_set[dev].store(true, std::memory_order_release);
    }
    return cudaSuccess;
}

template <int kM>
static bool pairs_fit(int n_sms)
{
    static std::atomic<int> fit[64] = {};   // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64 || (n_sms & 1))
        return false;
    if (fit[dev].load(std::memory_order_acquire) == 0) {
        if (set_smem_attr<kM>() != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n_sms);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k_attention_tc<kM>, &cfg);
        if (e != cudaSuccess)
            cudaGetLastError();
        fit[dev].store((e == cudaSuccess && 2 * n >= n_sms) ? 1 : 2, std::memory_order_release);
    }
    return fit[dev].load(std::memory_order_acquire) == 1;
}

// (the values-gathering variant has the same block and shared memory)
bool attention_tc_pairs_fit(int n_sms) { return pairs_fit<kModeStitched>(n_sms); }

template <int kM>
static cudaError_t launch_variant(const TcAttnArgs &ta, int grid, bool pdl, bool pairs, cudaStream_t s)
{
    constexpr bool kV = kM != kModeStitched;
    cudaError_t e = set_smem_attr<kM>();
    if (e != cudaSuccess)
        return e;
    static const CUtensorMap no_map{};
    static const GatherArgs no_gather{};
    static const SpanTable no_spans{};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n_attr = 0;
    if (pdl) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    if (pairs) {   // split units: half 0 on the even CTA of a cluster, half 1 on the odd one
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = 2;
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    return cudaLaunchKernelEx(&cfg, k_attention_tc<kM>, *static_cast<const CUtensorMap *>(ta.tmap_q),
                              *static_cast<const CUtensorMap *>(ta.tmap_k),
                              *static_cast<const CUtensorMap *>(ta.tmap_v), ta.base, *ta.rt, ta.n_m_blocks,
                              kV ? *static_cast<const CUtensorMap *>(ta.tmap_pv) : no_map,
                              kV ? *static_cast<const CUtensorMap *>(ta.tmap_bv) : no_map,
                              kV ? ta.g : no_gather, kV && ta.st ? *ta.st : no_spans,
                              ta.base.out_tma ? *static_cast<const CUtensorMap *>(ta.tmap_out) : no_map);
}

cudaError_t launch_attention_tc(const TcAttnArgs &ta, bool pdl, cudaStream_t s)
{
    if (ta.n_m_blocks == 0)
        return cudaSuccess;
    const int64_t units = (int64_t)ta.n_m_blocks *
                          (ta.base.lh_count > 0 ? ta.base.lh_count : ta.base.n_layers * ta.base.n_kv_heads);
    if (units > 0x7fffffff)
        return cudaErrorInvalidValue;
    const int64_t items = 2 * units - ta.base.n_full;
    const int grid = (int)(items < ta.n_sms ? items : ta.n_sms);
    const bool pairs = ta.base.n_full < units;
    // the two halves of split unit i are items n_full + 2i and n_full + 2i + 1:
    // CTAs 2i and 2i + 1 of the last round when n_full is a multiple of the grid
    if (pairs && ((grid & 1) || ta.base.n_full % grid != 0))
        return cudaErrorInvalidValue;
    if (!ta.gather_v)
        return launch_variant<kModeStitched>(ta, grid, pdl, pairs, s);
    return ta.g.locals ? launch_variant<kModeGatherVLocal>(ta, grid, pdl, pairs, s)
                       : launch_variant<kModeGatherV>(ta, grid, pdl, pairs, s);
}

}  // namespace kvr
