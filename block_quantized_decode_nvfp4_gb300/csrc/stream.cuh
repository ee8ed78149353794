// stream.cuh -- bulk-copy (TMA) weight streaming into a shared-memory ring,
// with mbarrier hand-off between one producer warp and consumer warps
// (sm_90+ PTX, used on sm_103a). Every wait is bounded: a wait that runs out
// records an error in the library's device error word and the waiter gives
// up instead of hanging the GPU.
#pragma once

#include <cstdint>

namespace bqd {

// Error bit set in a kernel's device error word when a wait runs out.
constexpr unsigned int kErrWaitTimeout = 1u;
// 2^31 SM cycles (about one second): far beyond any legitimate wait
// (microseconds), short enough to give the GPU back.
constexpr long long kWaitCycles = 1ll << 31;

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false if it ran out,
// after setting kErrWaitTimeout in *err. try_wait itself suspends the thread
// until the phase completes or a short hardware time limit passes, so the
// loop needs no sleep of its own (a sleep only delays the wake-up).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err,
                                          long long limit = kWaitCycles)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    do {
        if (mbar_try_wait(bar, parity)) return true;
    } while (clock64() - t0 < limit);
    atomicOr(err, kErrWaitTimeout);
    return false;
}

// The same wait for a whole (converged) warp: lane 0 polls, the other lanes
// wait at the warp barrier, which also orders their later memory accesses
// after lane 0's acquire. Keeps polling traffic to one thread per warp.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, unsigned int* err)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err);
    __syncwarp();
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

// 1-D bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned); completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Named barrier `id` (not 0, which __syncthreads uses) over `threads` threads.
__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace bqd
