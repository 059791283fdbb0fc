// kvr_selftest.cu -- the bounded-wait error path, made to run out on purpose.
//
// Every wait in the library's kernels (TMA copies, MMA completions, the
// partner CTA of a cluster) gives up after a time limit, records
// KVR_ERR_TIMEOUT in the pool's error word and lets the kernel end, so that a
// lost signal surfaces as a status from kvr_check instead of a hung GPU.  This
// kernel waits, the same way, on an mbarrier that nothing ever completes, so
// that the reporting path can be tested without breaking a hot-path kernel.
#include "kvr_internal.cuh"

namespace kvr {

__global__ void k_wait_selftest(int *err, unsigned long long limit_ns)
{
    __shared__ alignas(8) unsigned long long bar;
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t0));
    uint32_t done = 0;
    do {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(b)
            : "memory");
        asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    } while (!done && t - t0 < limit_ns);
    if (!done && threadIdx.x == 0 && err)
        atomicCAS(err, kDevOk, kDevTimeout);
}

cudaError_t launch_wait_selftest(int *err, unsigned long long limit_ns, cudaStream_t s)
{
    k_wait_selftest<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace kvr
