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
// device address, so the address is looked up with cudaGetSymbolAddress, with
// the device current, on the first call in each CUDA context, and cached
// under that context's id. A device reset (cudaDeviceReset) destroys the
// context and the module with it; the next call sees a new context id and
// looks the address up again instead of using the freed one.
#include <cuda.h>
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

// Driver entry points for the current context and its id, taken through the
// runtime so that the library does not link the driver library itself.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns()
{
    static DriverFns fns = [] {
        DriverFns f;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
        return f;
    }();
    return fns;
}

// Id of the calling thread's current context; 0 if there is none yet (the
// runtime makes the device's primary context current lazily).
unsigned long long current_context_id()
{
    const DriverFns& f = driver_fns();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!f.get_current || !f.get_id || f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

struct DeviceScratch {
    bool arch_known = false;
    bool sm103 = false;
    unsigned long long ctx_id = 0;  // context the cached address belongs to (0: none)
    void* addr = nullptr;
};

// Per-device set-up: architecture check (once) and the device address of the
// scratch array in the current context (once per context). The device must
// be current. CUDA failures are recorded for bqd_last_cuda_error().
bqd_status scratch_for_current_device(void** out)
{
    static std::mutex mu;
    static DeviceScratch cache[64];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        bqd::record_cuda_error(e);
        cudaGetLastError();
        return BQD_ERR_ARCH;
    }
    std::lock_guard<std::mutex> g(mu);
    DeviceScratch& c = cache[dev];
    if (!c.arch_known) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) {
            bqd::record_cuda_error(e);
            cudaGetLastError();
            return BQD_ERR_ARCH;
        }
        c.sm103 = major == 10 && minor == 3;
        c.arch_known = true;
    }
    if (!c.sm103) return BQD_ERR_ARCH;
    const unsigned long long id = current_context_id();
    if (id == 0 || id != c.ctx_id) {
        // First call in this context (or no context current yet: the lookup
        // below makes the device's primary context current).
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_moe_scratch)) != cudaSuccess || p == nullptr) {
            bqd::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            cudaGetLastError();
            return BQD_ERR_LAUNCH;
        }
        c.addr = p;
        c.ctx_id = current_context_id();
    }
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
    if (e == cudaSuccess) return BQD_OK;
    bqd::record_cuda_error(e);
    return BQD_ERR_LAUNCH;
}
