// moe_noalloc.cu -- the routed MoE layer for callers that cannot allocate
// device memory.
//
// Some callers have no way to call cudaMalloc: plug-ins inside a host
// program that owns every device allocation and hands its plug-ins no
// allocator, or latency-critical loops that are forbidden to allocate once
// they have started. moe_grouped_gemv needs a scratch workspace from its
// caller; moe_grouped_gemv_noalloc instead runs the same kernels on a
// scratch array that lives in this file as a static device variable, so
// the caller passes only inputs and outputs.
//
// The array (kScratchBytes) exists on every GPU that loads the library, for
// the life of the process. Host code cannot use the array's name as a
// device address, so on the first call on a device (with that device
// current) the address is looked up with cudaGetSymbolAddress and cached.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "bqd.h"
#include "gemv.h"

namespace {

// Largest workspace the shared scratch can hold: moe_workspace_bytes(T, topk,
// H, I) must not exceed it (T = 16, top-8, H = 2048, I = 512 needs 1.31 MiB).
constexpr size_t kScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_moe_scratch[kScratchBytes];

struct DeviceScratch {
    bool ready = false;
    bool sm103 = false;
    void* addr = nullptr;
};

// Per-device set-up, once: architecture check and the device address of the
// scratch array (the device must be current).
bqd_status scratch_for_current_device(void** out)
{
    static std::mutex mu;
    static DeviceScratch cache[64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return BQD_ERR_ARCH;
    }
    std::lock_guard<std::mutex> g(mu);
    DeviceScratch& c = cache[dev];
    if (!c.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return BQD_ERR_ARCH;
        }
        c.sm103 = major == 10 && minor == 3;
        if (c.sm103) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_moe_scratch) != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return BQD_ERR_LAUNCH;
            }
            c.addr = p;
        }
        c.ready = true;
    }
    if (!c.sm103) return BQD_ERR_ARCH;
    *out = c.addr;
    return BQD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" bqd_status moe_grouped_gemv_noalloc(const uint8_t* gu_codes, const uint8_t* gu_scales,
                                               const float* gu_ts, const uint8_t* dn_codes,
                                               const uint8_t* dn_scales, const float* dn_ts, const uint16_t* x,
                                               const int32_t* expert_offsets, const int32_t* pair_token,
                                               const float* pair_weight, const int32_t* pair_slot, float* y, int E,
                                               int H, int I, int T, int topk, cudaStream_t stream)
{
    if (T < 1 || E < 1 || E > bqd::kMoeMaxExperts || topk < 1 || topk > E || topk > bqd::kMoeMaxTopk ||
        static_cast<int64_t>(T) * topk > bqd::kMoeMaxPairs || H < 32 || H > 8192 || H % 32 != 0 || I < 32 ||
        I > 4096 || I % 32 != 0)
        return BQD_ERR_SHAPE;
    const void* ptrs[] = {gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts,
                          x,        expert_offsets, pair_token, pair_weight, pair_slot, y};
    for (const void* p : ptrs)
        if (!p) return BQD_ERR_NULL;
    for (const void* p : ptrs)
        if (!aligned16(p)) return BQD_ERR_ALIGN;
    if (bqd::moe_workspace_size(T, topk, H, I) > kScratchBytes) return BQD_ERR_WORKSPACE;
    void* scratch = nullptr;
    const bqd_status st = scratch_for_current_device(&scratch);
    if (st != BQD_OK) return st;
    // The launcher clears the status word, and the first kernel clears the
    // per-(token, slot) counters and weights, so the previous call's contents
    // of the shared array do not leak into this one.
    const bqd::MoeWorkspace ws = bqd::moe_workspace_carve(scratch, T, topk, H, I);
    const cudaError_t e = bqd::launch_moe_grouped(gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x,
                                                  expert_offsets, pair_token, pair_weight, pair_slot, y, ws, E, H,
                                                  I, T, topk, stream);
    return e == cudaSuccess ? BQD_OK : BQD_ERR_LAUNCH;
}
