// kvr_decode_common.cuh -- pieces of the decode-step kernel: tile geometry,
// bounded mbarrier waits, TMA loads, and the warp-level bf16 MMA (mma.sync
// m16n8k16 with ldmatrix operands) it streams tiles through.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "kvr_internal.cuh"

namespace kvr {
namespace dec {

constexpr int kDecThreads = 128;
constexpr int kDecStages = 3;
constexpr int kDecTile = 128;                       // keys per tile
constexpr int kDecD = 128;                          // head dim
constexpr int kDecTileBytes = kDecTile * kDecD * 2; // 32 KB
constexpr int kDecPanel = kDecTileBytes / 2;        // 16 KB: 128 rows x 64 columns
constexpr int kDecStageBytes = 2 * kDecTileBytes;   // K tile, then V tile
constexpr unsigned long long kDecWaitNs = 2000000000ull;
// the four warps' final states: m, l [4][16] and O [4][16][128] fp32
constexpr int kDecMergeBytes = 4 * 16 * 4 * 2 + 4 * 16 * kDecD * 4;

__device__ __forceinline__ uint64_t dec_globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t dec_smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void dec_mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void dec_mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void dec_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bounded wait on a barrier phase; false after 2 s (the caller records a timeout).
__device__ __forceinline__ bool dec_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = dec_globaltimer();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok)
            return true;
        if (dec_globaltimer() - t0 > kDecWaitNs)
            return false;
    }
}

__device__ __forceinline__ void dec_tma_load(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// d += a (16x16, row) * b (16x8, col), bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float *d, const uint32_t *a, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float dec_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of 16-byte chunk `c` (0..15) of row `r` in a tile stored as two
// 128B-swizzled panels of 64 columns.
__device__ __forceinline__ uint32_t sw_off(int r, int c)
{
    return (uint32_t)((c >> 3) * kDecPanel + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}


}  // namespace dec
}  // namespace kvr
