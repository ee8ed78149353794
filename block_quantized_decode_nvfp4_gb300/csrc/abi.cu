// abi.cu -- the extern "C" entry points declared in include/bqd.h: argument
// validation (host only, before any CUDA call), the device architecture
// check, and dispatch to the kernels' launchers.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "bqd.h"
#include "gemm.h"
#include "gemv.h"
#include "host_util.h"
#include "q4_1.cuh"

namespace {

constexpr int kMaxN = 16;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The current device must be compute capability 10.3 (sm_103a code only).
bqd_status check_arch()
{
    static std::mutex mu;
    static int state[64] = {0};  // 0 unknown, 1 ok, 2 wrong
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return BQD_ERR_ARCH;
    }
    if (dev >= 64) return BQD_ERR_ARCH;
    std::lock_guard<std::mutex> g(mu);
    if (state[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return BQD_ERR_ARCH;
        }
        state[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return state[dev] == 1 ? BQD_OK : BQD_ERR_ARCH;
}

thread_local const char* t_last_cuda_error = "cudaSuccess";

bqd_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return BQD_OK;
    bqd::record_cuda_error(e);
    return BQD_ERR_LAUNCH;
}

bqd_status zero_output(float* y, int64_t count, cudaStream_t s)
{
    if (count == 0) return BQD_OK;
    return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(count) * sizeof(float), s));
}

// Common shape rules of the dense GEMV / dequant calls.
bqd_status check_dense(const void* a, const void* b, const void* x, const void* y, int64_t M, int64_t K, int N,
                       int kdiv, bool has_x)
{
    if (M < 0 || K < 0 || K % kdiv != 0) return BQD_ERR_SHAPE;
    if (has_x && (N < 1 || N > kMaxN)) return BQD_ERR_SHAPE;
    if (M > 0 && K > 0 && M > (int64_t(1) << 62) / K) return BQD_ERR_SHAPE;
    if (M == 0) return BQD_OK;
    if (!y) return BQD_ERR_NULL;
    if (!aligned16(y)) return BQD_ERR_ALIGN;
    if (K == 0) return BQD_OK;
    if (!a || !b || (has_x && !x)) return BQD_ERR_NULL;
    if (!aligned16(a) || !aligned16(b) || (has_x && !aligned16(x))) return BQD_ERR_ALIGN;
    return BQD_OK;
}

}  // namespace

void bqd::record_cuda_error(cudaError_t e)
{
    if (e != cudaSuccess) t_last_cuda_error = cudaGetErrorName(e);
}

extern "C" {

const char* bqd_status_string(bqd_status s)
{
    switch (s) {
        case BQD_OK: return "ok";
        case BQD_ERR_NULL: return "a required pointer is NULL";
        case BQD_ERR_SHAPE: return "a size is out of range or breaks a divisibility rule";
        case BQD_ERR_ALIGN: return "a base pointer is not 16-byte aligned";
        case BQD_ERR_ARCH: return "no current CUDA device, or it is not compute capability 10.3";
        case BQD_ERR_LAUNCH: return "CUDA launch failed";
        case BQD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case BQD_ERR_PATH: return "unknown compute path, or it does not support these arguments";
        case BQD_ERR_DEVICE: return "device-side status bits set (malformed MoE list)";
        default: return "unknown status";
    }
}

int bqd_version(void) { return 100; }

const char* bqd_last_cuda_error(void) { return t_last_cuda_error; }

unsigned int bqd_set_launch_flags(unsigned int flags)
{
    return bqd::launch_flags_ref().exchange(flags & BQD_LAUNCH_PDL);
}

unsigned int bqd_get_launch_flags(void) { return bqd::launch_flags(); }

bqd_status nvfp4_gemv_path(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x,
                           float* y, int64_t M, int64_t K, int N, int path, cudaStream_t stream)
{
    if (path != BQD_PATH_AUTO && path != BQD_PATH_CUDA_CORE && path != BQD_PATH_STREAM && path != BQD_PATH_MMA &&
        path != BQD_PATH_DIRECT && path != BQD_PATH_TILES)
        return BQD_ERR_PATH;
    bqd_status st = check_dense(codes, scales, x, y, M, K, N, 16, true);
    if (st != BQD_OK || M == 0) return st;
    if (path == BQD_PATH_STREAM && !bqd::stream_gemv_supported(M, K, N)) return BQD_ERR_PATH;
    if (path == BQD_PATH_MMA && !bqd::mma_gemv_supported(M, K, N)) return BQD_ERR_PATH;
    if (path == BQD_PATH_DIRECT && !bqd::direct_gemv_supported(M, K, N)) return BQD_ERR_PATH;
    if (path == BQD_PATH_TILES && !bqd::tiles_gemv_supported(M, K, N)) return BQD_ERR_PATH;
    if ((st = check_arch()) != BQD_OK) return st;
    if (K == 0) return zero_output(y, M * N, stream);
    const bool use_tiles = path == BQD_PATH_TILES;
    const bool use_direct = path == BQD_PATH_DIRECT || (path == BQD_PATH_AUTO && bqd::direct_gemv_supported(M, K, N));
    const bool use_stream = path == BQD_PATH_STREAM || (path == BQD_PATH_AUTO && bqd::stream_gemv_supported(M, K, N));
    const bool use_mma = path == BQD_PATH_MMA || (path == BQD_PATH_AUTO && N >= 2 && bqd::mma_gemv_supported(M, K, N));
    if (use_direct)
        return from_cuda(bqd::launch_nvfp4_gemv_direct(codes, scales, tensor_scale, x, y, M, K, stream));
    if (use_stream)
        return from_cuda(bqd::launch_nvfp4_gemv_stream(codes, scales, tensor_scale, x, y, M, K, stream));
    if (use_tiles)
        return from_cuda(bqd::launch_nvfp4_gemv_tiles(codes, scales, tensor_scale, x, y, M, K, N, stream));
    if (use_mma) return from_cuda(bqd::launch_nvfp4_gemv_mma(codes, scales, tensor_scale, x, y, M, K, N, stream));
    return from_cuda(bqd::launch_nvfp4_gemv_cuda_core(codes, scales, tensor_scale, x, y, M, K, N, stream));
}

bqd_status nvfp4_gemv(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x, float* y,
                      int64_t M, int64_t K, int N, cudaStream_t stream)
{
    return nvfp4_gemv_path(codes, scales, tensor_scale, x, y, M, K, N, BQD_PATH_AUTO, stream);
}

bqd_status q8_0_gemv_path(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M, int64_t K,
                          int N, int path, cudaStream_t stream)
{
    if (path != BQD_PATH_AUTO && path != BQD_PATH_CUDA_CORE && path != BQD_PATH_STREAM && path != BQD_PATH_DIRECT)
        return BQD_ERR_PATH;
    bqd_status st = check_dense(q, d, x, y, M, K, N, 32, true);
    if (st != BQD_OK || M == 0) return st;
    if (path == BQD_PATH_STREAM && !bqd::stream_gemv_supported(M, K, N)) return BQD_ERR_PATH;
    if (path == BQD_PATH_DIRECT && !bqd::direct_gemv_supported(M, K, N)) return BQD_ERR_PATH;
    if ((st = check_arch()) != BQD_OK) return st;
    if (K == 0) return zero_output(y, M * N, stream);
    if (path == BQD_PATH_DIRECT || (path == BQD_PATH_AUTO && bqd::direct_gemv_supported(M, K, N)))
        return from_cuda(bqd::launch_q8_0_gemv_direct(q, d, x, y, M, K, stream));
    if (path != BQD_PATH_CUDA_CORE && bqd::stream_gemv_supported(M, K, N))
        return from_cuda(bqd::launch_q8_0_gemv_stream(q, d, x, y, M, K, stream));
    return from_cuda(bqd::launch_q8_0_gemv_cuda_core(q, d, x, y, M, K, N, stream));
}

bqd_status q8_0_gemv(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M, int64_t K, int N,
                     cudaStream_t stream)
{
    return q8_0_gemv_path(q, d, x, y, M, K, N, BQD_PATH_AUTO, stream);
}

bqd_status q4_0_gemv_path(const uint8_t* codes, const uint16_t* d, const uint16_t* x, float* y, int64_t M,
                          int64_t K, int N, int path, cudaStream_t stream)
{
    if (path != BQD_PATH_AUTO && path != BQD_PATH_CUDA_CORE && path != BQD_PATH_DIRECT) return BQD_ERR_PATH;
    bqd_status st = check_dense(codes, d, x, y, M, K, N, 32, true);
    if (st != BQD_OK || M == 0) return st;
    if (path == BQD_PATH_DIRECT && !bqd::direct_gemv_supported(M, K, N)) return BQD_ERR_PATH;
    if ((st = check_arch()) != BQD_OK) return st;
    if (K == 0) return zero_output(y, M * N, stream);
    if (path == BQD_PATH_DIRECT || (path == BQD_PATH_AUTO && bqd::direct_gemv_supported(M, K, N)))
        return from_cuda(bqd::launch_q4_0_gemv_direct(codes, d, x, y, M, K, stream));
    return from_cuda(bqd::launch_q4_0_gemv_cuda_core(codes, d, x, y, M, K, N, stream));
}

bqd_status q4_0_gemv(const uint8_t* codes, const uint16_t* d, const uint16_t* x, float* y, int64_t M, int64_t K,
                     int N, cudaStream_t stream)
{
    return q4_0_gemv_path(codes, d, x, y, M, K, N, BQD_PATH_AUTO, stream);
}

bqd_status q4_1_gemv(const uint8_t* codes, const uint16_t* dm, const uint16_t* x, float* y, int64_t M, int64_t K,
                     int N, cudaStream_t stream)
{
    bqd_status st = check_dense(codes, dm, x, y, M, K, N, 32, true);
    if (st != BQD_OK || M == 0) return st;
    if ((st = check_arch()) != BQD_OK) return st;
    if (K == 0) return zero_output(y, M * N, stream);
    return from_cuda(bqd::launch_q4_1_gemv_cuda_core(codes, dm, x, y, M, K, N, stream));
}

bqd_status q4_1_dequant(const uint8_t* codes, const uint16_t* dm, float* w, int64_t M, int64_t K, cudaStream_t stream)
{
    bqd_status st = check_dense(codes, dm, nullptr, w, M, K, 1, 32, false);
    if (st != BQD_OK || M == 0 || K == 0) return st;
    if ((st = check_arch()) != BQD_OK) return st;
    return from_cuda(bqd::launch_q4_1_dequant(codes, dm, w, M, K, stream));
}

bqd_status fp8_b128_gemv_path(const uint8_t* codes, const float* scales, const uint16_t* x, float* y, int64_t M,
                              int64_t K, int N, int path, cudaStream_t stream)
{
    if (path != BQD_PATH_AUTO && path != BQD_PATH_CUDA_CORE && path != BQD_PATH_DIRECT) return BQD_ERR_PATH;
    bqd_status st = check_dense(codes, scales, x, y, M, K, N, 32, true);
    if (st != BQD_OK || M == 0) return st;
    if (path == BQD_PATH_DIRECT && !bqd::direct_gemv_supported(M, K, N)) return BQD_ERR_PATH;
    if ((st = check_arch()) != BQD_OK) return st;
    if (K == 0) return zero_output(y, M * N, stream);
    if (path == BQD_PATH_DIRECT || (path == BQD_PATH_AUTO && bqd::direct_gemv_supported(M, K, N)))
        return from_cuda(bqd::launch_fp8_b128_gemv_direct(codes, scales, x, y, M, K, stream));
    return from_cuda(bqd::launch_fp8_b128_gemv_cuda_core(codes, scales, x, y, M, K, N, stream));
}

bqd_status fp8_b128_gemv(const uint8_t* codes, const float* scales, const uint16_t* x, float* y, int64_t M,
                         int64_t K, int N, cudaStream_t stream)
{
    return fp8_b128_gemv_path(codes, scales, x, y, M, K, N, BQD_PATH_AUTO, stream);
}

// ---------------------------------------------------------------- prefill GEMM
bqd_status nvfp4_gemm(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x, float* y,
                      int64_t M, int64_t K, int64_t T, cudaStream_t stream)
{
    if (M < 0 || K < 0 || T < 0 || K % 64 != 0) return BQD_ERR_SHAPE;
    if (M > 0 && K > 0 && M > (int64_t(1) << 62) / K) return BQD_ERR_SHAPE;
    if (M == 0 || T == 0) return BQD_OK;
    if (!y) return BQD_ERR_NULL;
    if (!aligned16(y)) return BQD_ERR_ALIGN;
    bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    if (K == 0) return zero_output(y, M * T, stream);
    if (!codes || !scales || !x) return BQD_ERR_NULL;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(x)) return BQD_ERR_ALIGN;
    if (!bqd::gemm_supported(M, K, T)) return BQD_ERR_SHAPE;
    return from_cuda(bqd::launch_nvfp4_gemm(codes, scales, tensor_scale, x, y, M, K, T, stream));
}

bqd_status nvfp4_gemm_grouped(const uint8_t* codes, const uint8_t* scales, const float* tensor_scales,
                              const uint16_t* x, const int32_t* expert_offsets, float* y, int E, int64_t M, int64_t K,
                              int64_t P, cudaStream_t stream)
{
    if (E < 1 || M < 0 || K < 0 || P < 0 || K % 64 != 0) return BQD_ERR_SHAPE;
    if (M > 0 && K > 0 && static_cast<int64_t>(E) * M > (int64_t(1) << 62) / K) return BQD_ERR_SHAPE;
    if (M == 0 || P == 0) return BQD_OK;
    if (!y) return BQD_ERR_NULL;
    if (!aligned16(y)) return BQD_ERR_ALIGN;
    bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    if (K == 0) return zero_output(y, M * P, stream);
    if (!codes || !scales || !tensor_scales || !x || !expert_offsets) return BQD_ERR_NULL;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) ||
        (reinterpret_cast<uintptr_t>(tensor_scales) & 3u) != 0 || (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) != 0)
        return BQD_ERR_ALIGN;
    if (!bqd::gemm_grouped_supported(E, M, K, P)) return BQD_ERR_SHAPE;
    return from_cuda(
        bqd::launch_nvfp4_gemm_grouped(codes, scales, tensor_scales, expert_offsets, E, x, y, M, K, P, stream));
}

size_t moe_prefill_workspace_bytes(int T, int topk, int H, int I, int E)
{
    if (T < 1 || topk < 1 || H < 1 || I < 1 || E < 1) return 0;
    return bqd::moe_prefill_workspace_size(T, topk, H, I, E);
}

bqd_status moe_prefill_layer(const float* logits, const uint8_t* gu_codes, const uint8_t* gu_scales,
                             const float* gu_ts, const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts,
                             const uint16_t* x, float* y, void* workspace, size_t workspace_bytes, int E, int H, int I,
                             int T, int topk, cudaStream_t stream)
{
    if (T < 1 || E < 1 || E > bqd::kMoeMaxExperts || topk < 1 || topk > E || topk > bqd::kMoeMaxTopk ||
        static_cast<int64_t>(T) * topk > bqd::kMoeMaxPairs || H < 64 || H % 64 != 0 || I < 64 || I % 64 != 0 ||
        H > (1 << 16) || I > (1 << 16))
        return BQD_ERR_SHAPE;
    if (!logits || !gu_codes || !gu_scales || !gu_ts || !dn_codes || !dn_scales || !dn_ts || !x || !y)
        return BQD_ERR_NULL;
    if (!workspace || workspace_bytes < bqd::moe_prefill_workspace_size(T, topk, H, I, E)) return BQD_ERR_WORKSPACE;
    for (const void* p : {static_cast<const void*>(logits), static_cast<const void*>(gu_codes),
                          static_cast<const void*>(gu_scales), static_cast<const void*>(dn_codes),
                          static_cast<const void*>(dn_scales), static_cast<const void*>(x), static_cast<const void*>(y),
                          static_cast<const void*>(workspace)})
        if (!aligned16(p)) return BQD_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(gu_ts) & 3u) != 0 || (reinterpret_cast<uintptr_t>(dn_ts) & 3u) != 0)
        return BQD_ERR_ALIGN;
    const bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    return from_cuda(bqd::launch_moe_prefill_layer(logits, gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x,
                                                   y, workspace, E, H, I, T, topk, stream));
}

// ---------------------------------------------------------------- encoders
bqd_status nvfp4_encode(const uint16_t* w, float tensor_scale, uint8_t* codes, uint8_t* scales, int64_t M, int64_t K,
                        cudaStream_t stream)
{
    if (M < 0 || K < 0 || K % 16 != 0 || (M > 0 && K > 0 && M > (int64_t(1) << 62) / K)) return BQD_ERR_SHAPE;
    if (!(tensor_scale >= 0x1p-100f && tensor_scale <= 0x1p100f)) return BQD_ERR_SHAPE;  // also rejects NaN
    if (M == 0 || K == 0) return BQD_OK;
    if (!w || !codes || !scales) return BQD_ERR_NULL;
    if (!aligned16(w) || !aligned16(codes)) return BQD_ERR_ALIGN;
    const bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    return from_cuda(bqd::launch_nvfp4_encode(w, tensor_scale, codes, scales, M, K, stream));
}

bqd_status q8_0_encode(const uint16_t* w, int8_t* q, uint16_t* d, int64_t M, int64_t K, cudaStream_t stream)
{
    if (M < 0 || K < 0 || K % 32 != 0 || (M > 0 && K > 0 && M > (int64_t(1) << 62) / K)) return BQD_ERR_SHAPE;
    if (M == 0 || K == 0) return BQD_OK;
    if (!w || !q || !d) return BQD_ERR_NULL;
    if (!aligned16(w) || !aligned16(q) || (reinterpret_cast<uintptr_t>(d) & 1u) != 0) return BQD_ERR_ALIGN;
    const bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    return from_cuda(bqd::launch_q8_0_encode(w, q, d, M, K, stream));
}

// ---------------------------------------------------------------- decode-path epilogues
namespace {

// The fused-epilogue GEMVs run the direct kernel: N == 1, M >= 1, K a
// multiple of 1024 with K / 1024 in {1, 2, 3, 4, 6, 8, 12, 16}.
bqd_status check_epilogue(const void* a, const void* b, const void* x, const void* out, const float* r, bool has_r,
                          int64_t rows, int64_t K, int N, int kdiv)
{
    bqd_status st = check_dense(a, b, x, out, rows, K, N, kdiv, true);
    if (st != BQD_OK) return st;
    if (N != 1 || rows < 1 || !bqd::direct_gemv_supported(rows, K, 1)) return BQD_ERR_SHAPE;
    if (has_r && !r) return BQD_ERR_NULL;
    if (has_r && !aligned16(r)) return BQD_ERR_ALIGN;
    return check_arch();
}

}  // namespace

bqd_status nvfp4_gemv_add(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x,
                          const float* residual, float* y, int64_t M, int64_t K, int N, cudaStream_t stream)
{
    const bqd_status st = check_epilogue(codes, scales, x, y, residual, true, M, K, N, 16);
    if (st != BQD_OK) return st;
    return from_cuda(bqd::launch_nvfp4_gemv_direct_add(codes, scales, tensor_scale, x, residual, y, M, K, stream));
}

bqd_status q8_0_gemv_add(const int8_t* q, const uint16_t* d, const uint16_t* x, const float* residual, float* y,
                         int64_t M, int64_t K, int N, cudaStream_t stream)
{
    const bqd_status st = check_epilogue(q, d, x, y, residual, true, M, K, N, 32);
    if (st != BQD_OK) return st;
    return from_cuda(bqd::launch_q8_0_gemv_direct_add(q, d, x, residual, y, M, K, stream));
}

bqd_status nvfp4_gemv_silu_mul(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x,
                               float* h, int64_t I, int64_t K, int N, cudaStream_t stream)
{
    if (I < 1 || I > (int64_t(1) << 38)) return BQD_ERR_SHAPE;
    const bqd_status st = check_epilogue(codes, scales, x, h, nullptr, false, 2 * I, K, N, 16);
    if (st != BQD_OK) return st;
    return from_cuda(bqd::launch_nvfp4_gemv_direct_silu_mul(codes, scales, tensor_scale, x, h, I, K, stream));
}

bqd_status q8_0_gemv_silu_mul(const int8_t* q, const uint16_t* d, const uint16_t* x, float* h, int64_t I, int64_t K,
                              int N, cudaStream_t stream)
{
    if (I < 1 || I > (int64_t(1) << 38)) return BQD_ERR_SHAPE;
    const bqd_status st = check_epilogue(q, d, x, h, nullptr, false, 2 * I, K, N, 32);
    if (st != BQD_OK) return st;
    return from_cuda(bqd::launch_q8_0_gemv_direct_silu_mul(q, d, x, h, I, K, stream));
}

bqd_status bqd_device_error(unsigned int* bits_out)
{
    if (!bits_out) return BQD_ERR_NULL;
    bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    unsigned int v = 0, w = 0, m = 0, n = 0, g = 0;
    if (bqd::read_and_clear_stream_error(&v) != cudaSuccess || bqd::read_and_clear_mma_error(&w) != cudaSuccess ||
        bqd::read_and_clear_moe_stream_error(&m) != cudaSuccess ||
        bqd::read_and_clear_moe_small_error(&n) != cudaSuccess || bqd::read_and_clear_gemm_error(&g) != cudaSuccess)
        return BQD_ERR_LAUNCH;
    v |= w | m | n | g;
    *bits_out = v;
    return v ? BQD_ERR_DEVICE : BQD_OK;
}

bqd_status bqd_debug_stream_fault(int withhold_last_stage, long long wait_limit_cycles)
{
    if (wait_limit_cycles < 0) return BQD_ERR_SHAPE;
    bqd::set_stream_fault(withhold_last_stage, wait_limit_cycles);
    return BQD_OK;
}

bqd_status nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float tensor_scale, float* w, int64_t M,
                         int64_t K, cudaStream_t stream)
{
    bqd_status st = check_dense(codes, scales, nullptr, w, M, K, 1, 16, false);
    if (st != BQD_OK || M == 0 || K == 0) return st;
    if ((st = check_arch()) != BQD_OK) return st;
    return from_cuda(bqd::launch_nvfp4_dequant(codes, scales, tensor_scale, w, M, K, stream));
}

bqd_status q8_0_dequant(const int8_t* q, const uint16_t* d, float* w, int64_t M, int64_t K, cudaStream_t stream)
{
    bqd_status st = check_dense(q, d, nullptr, w, M, K, 1, 32, false);
    if (st != BQD_OK || M == 0 || K == 0) return st;
    if ((st = check_arch()) != BQD_OK) return st;
    return from_cuda(bqd::launch_q8_0_dequant(q, d, w, M, K, stream));
}

bqd_status q4_0_dequant(const uint8_t* codes, const uint16_t* d, float* w, int64_t M, int64_t K, cudaStream_t stream)
{
    bqd_status st = check_dense(codes, d, nullptr, w, M, K, 1, 32, false);
    if (st != BQD_OK || M == 0 || K == 0) return st;
    if ((st = check_arch()) != BQD_OK) return st;
    return from_cuda(bqd::launch_q4_0_dequant(codes, d, w, M, K, stream));
}

bqd_status fp8_b128_dequant(const uint8_t* codes, const float* scales, float* w, int64_t M, int64_t K,
                            cudaStream_t stream)
{
    bqd_status st = check_dense(codes, scales, nullptr, w, M, K, 1, 32, false);
    if (st != BQD_OK || M == 0 || K == 0) return st;
    if ((st = check_arch()) != BQD_OK) return st;
    return from_cuda(bqd::launch_fp8_b128_dequant(codes, scales, w, M, K, stream));
}

bqd_status moe_route_topk(const float* logits, int T, int E, int topk, int32_t* expert_offsets, int32_t* pair_token,
                          float* pair_weight, int32_t* pair_slot, cudaStream_t stream)
{
    if (T < 1 || E < 1 || E > bqd::kMoeMaxExperts || topk < 1 || topk > E || topk > bqd::kMoeMaxTopk ||
        static_cast<int64_t>(T) * topk > bqd::kMoeMaxPairs)
        return BQD_ERR_SHAPE;
    if (!logits || !expert_offsets || !pair_token || !pair_weight || !pair_slot) return BQD_ERR_NULL;
    if (!aligned16(logits) || !aligned16(expert_offsets) || !aligned16(pair_token) || !aligned16(pair_weight) ||
        !aligned16(pair_slot))
        return BQD_ERR_ALIGN;
    bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    return from_cuda(
        bqd::launch_moe_route(logits, T, E, topk, expert_offsets, pair_token, pair_weight, pair_slot, stream));
}

size_t moe_workspace_bytes(int T, int topk, int H, int I)
{
    if (T < 1 || topk < 1 || H < 1 || I < 1) return 0;
    return bqd::moe_workspace_size(T, topk, H, I);
}

bqd_status moe_grouped_gemv(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                            const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts, const uint16_t* x,
                            const int32_t* expert_offsets, const int32_t* pair_token, const float* pair_weight,
                            const int32_t* pair_slot, float* y, void* workspace, size_t workspace_bytes, int E,
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
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        workspace_bytes < bqd::moe_workspace_size(T, topk, H, I))
        return BQD_ERR_WORKSPACE;
    bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    const bqd::MoeWorkspace ws = bqd::moe_workspace_carve(workspace, T, topk, H, I);
    return from_cuda(bqd::launch_moe_grouped(gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x,
                                             expert_offsets, pair_token, pair_weight, pair_slot, y, ws, E, H, I, T,
                                             topk, stream));
}

static size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

size_t moe_layer_workspace_bytes(int T, int topk, int H, int I, int E)
{
    if (T < 1 || topk < 1 || H < 1 || I < 1 || E < 1) return 0;
    const size_t P = static_cast<size_t>(T) * topk;
    return bqd::moe_workspace_size(T, topk, H, I) + align256((static_cast<size_t>(E) + 1) * 4) + 3 * align256(P * 4);
}

bqd_status moe_layer(const float* logits, const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                     const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts, const uint16_t* x,
                     float* y, void* workspace, size_t workspace_bytes, int E, int H, int I, int T, int topk,
                     cudaStream_t stream)
{
    if (T < 1 || E < 1 || E > bqd::kMoeMaxExperts || topk < 1 || topk > E || topk > bqd::kMoeMaxTopk ||
        static_cast<int64_t>(T) * topk > bqd::kMoeMaxPairs || H < 32 || H > 8192 || H % 32 != 0 || I < 32 ||
        I > 4096 || I % 32 != 0)
        return BQD_ERR_SHAPE;
    const void* ptrs[] = {logits, gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x, y};
    for (const void* p : ptrs)
        if (!p) return BQD_ERR_NULL;
    for (const void* p : ptrs)
        if (!aligned16(p)) return BQD_ERR_ALIGN;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        workspace_bytes < moe_layer_workspace_bytes(T, topk, H, I, E))
        return BQD_ERR_WORKSPACE;
    bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    const bqd::MoeWorkspace ws = bqd::moe_workspace_carve(workspace, T, topk, H, I);
    if (bqd::moe_small_supported(E, H, I, T, topk))
        return from_cuda(bqd::launch_moe_small_layer(logits, gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts,
                                                     x, nullptr, nullptr, nullptr, nullptr, y, ws, E, H, I, T, topk,
                                                     stream));
    // the list after the layer's own workspace
    const size_t P = static_cast<size_t>(T) * topk;
    char* lp = static_cast<char*>(workspace) + bqd::moe_workspace_size(T, topk, H, I);
    int32_t* offsets = reinterpret_cast<int32_t*>(lp);
    lp += align256((static_cast<size_t>(E) + 1) * 4);
    int32_t* pair_token = reinterpret_cast<int32_t*>(lp);
    lp += align256(P * 4);
    float* pair_weight = reinterpret_cast<float*>(lp);
    lp += align256(P * 4);
    int32_t* pair_slot = reinterpret_cast<int32_t*>(lp);
    st = from_cuda(
        bqd::launch_moe_route(logits, T, E, topk, offsets, pair_token, pair_weight, pair_slot, stream));
    if (st != BQD_OK) return st;
    return from_cuda(bqd::launch_moe_grouped(gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x, offsets,
                                             pair_token, pair_weight, pair_slot, y, ws, E, H, I, T, topk, stream));
}

bqd_status bqd_moe_read_status(const void* workspace, int32_t* status_out, cudaStream_t stream)
{
    if (!workspace || !status_out) return BQD_ERR_NULL;
    bqd_status st = check_arch();
    if (st != BQD_OK) return st;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return BQD_ERR_LAUNCH;
    *status_out = v;
    return v ? BQD_ERR_DEVICE : BQD_OK;
}

}  // extern "C"
