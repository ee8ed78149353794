// gemv.cu -- CUDA-core block-quantized GEMV for sm_103a, N = 1..16 columns,
// plus the exact dequantisation kernels used to check the decode bit by bit.
//
// Y[n][m] = ts * sum_b scale[m][b] * sum_{k in block b} elem[m][k] * X[n][k]
// for NVFP4 (E2M1 elements, E4M3 scale per 16 k, FP32 tensor scale ts), and
// Y[n][m] = sum_b d[m][b] * sum_{k in block b} q[m][k] * X[n][k] for Q8_0
// (int8 elements, fp16 scale per 32 k). X is bf16 [N][K], Y fp32 [N][M].
// ("robertbfuentes7-cloud/bw24" README, NVFP4 (W4) decode path and
// speculative verify of K+1 tokens; "avifenesh/memra" README, Decode kernels.)
//
// Design: every weight byte is read once from HBM with 16-byte streaming
// loads; the activations are staged once per CTA in shared memory as fp32;
// elements are decoded in registers (E2M1 -> f16x2 by the hardware convert,
// int8 -> fp32 by a byte-permute trick); products accumulate in fp32 with
// packed f32x2 FMAs; each warp reduces its rows with xor shuffles. Rows are
// split evenly over a grid sized to fill every SM once.
#include "gemv.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "host_util.h"
#include "q4_1.cuh"

namespace bqd {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
// Shared memory for the fp32 activations of one segment of K.
constexpr int kXsBudgetBytes = 96 * 1024;

// One launch computes NC columns for groups of RPW rows, keeping D chunks of
// each row in flight. When NC * K fp32 activations fit in shared memory
// (seg_len == K) every warp owns a contiguous, balanced range of rows; it
// issues its first weight loads before the CTA stages the activations, and
// never synchronises afterwards. Otherwise K is processed in segments of
// seg_len elements: the CTA owns a balanced row range, walks it in batches of
// kWarps * RPW rows and restages the activations for each segment.
// Row pointers of the group starting at r0 (rows past r_end repeat r0).
template <class F, int RPW>
__device__ __forceinline__ void group_rows(const uint8_t* codes, const uint8_t* scales, int64_t cpitch, int64_t K,
                                           int64_t r0, int64_t r_end, const uint8_t* (&crow)[RPW],
                                           const uint8_t* (&srow)[RPW])
{
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int64_t m = r0 + r < r_end ? r0 + r : r0;
        crow[r] = codes + m * cpitch;
        srow[r] = scales + RowPitch<F>::srow(m, K);
    }
}

template <class F, int RPW, int NC, int D>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const uint8_t* __restrict__ codes,
                                                        const uint8_t* __restrict__ scales, float ts,
                                                        const uint16_t* __restrict__ x, float* __restrict__ y,
                                                        int64_t M, int64_t K, int seg_len)
{
    extern __shared__ __align__(16) float xs[];
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int64_t cpitch = RowPitch<F>::codes(K);
    const int chunks = static_cast<int>(K / F::kElems);
    RowStream<F, RPW, D> rs;

    if (seg_len == K) {
        const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
        const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
        const int64_t r_lo = M * gw / nw, r_hi = M * (gw + 1) / nw;
        const uint8_t* crow[RPW];
        const uint8_t* srow[RPW];
        group_rows<F>(codes, scales, cpitch, K, r_lo, r_hi, crow, srow);
        if (r_lo < r_hi) rs.start(crow, srow, 0, chunks, lane);
        stage_x_bf16<F>(x, K, NC, 0, static_cast<int>(K), xs);
        __syncthreads();
        for (int64_t r0 = r_lo; r0 < r_hi; r0 += RPW) {
            if (r0 != r_lo) {
                group_rows<F>(codes, scales, cpitch, K, r0, r_hi, crow, srow);
                rs.start(crow, srow, 0, chunks, lane);
            }
            const int nrows = static_cast<int>(r_hi - r0 < RPW ? r_hi - r0 : RPW);
            float2 acc[RPW][NC];
#pragma unroll
            for (int r = 0; r < RPW; ++r)
#pragma unroll
                for (int n = 0; n < NC; ++n) acc[r][n] = make_float2(0.f, 0.f);
            rs.template run<NC>(xs, static_cast<int>(K), acc);
#pragma unroll
            for (int r = 0; r < RPW; ++r)
#pragma unroll
                for (int n = 0; n < NC; ++n) {
                    const float v = warp_sum(acc[r][n].x + acc[r][n].y);
                    if (lane == 0 && r < nrows) y[n * M + r0 + r] = v * ts;
                }
        }
        return;
    }

    // Segmented K.
    const int64_t b_lo = M * blockIdx.x / gridDim.x, b_hi = M * (blockIdx.x + 1) / gridDim.x;
    const int seg_chunks = seg_len / F::kElems;
    for (int64_t batch = b_lo; batch < b_hi; batch += static_cast<int64_t>(kWarps) * RPW) {
        const int64_t r0 = batch + static_cast<int64_t>(warp) * RPW;
        const int64_t left = b_hi - r0;
        const int nrows = left <= 0 ? 0 : static_cast<int>(left < RPW ? left : RPW);
        const uint8_t* crow[RPW];
        const uint8_t* srow[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int64_t m = nrows > 0 ? r0 + (r < nrows ? r : 0) : 0;
            crow[r] = codes + m * cpitch;
            srow[r] = scales + RowPitch<F>::srow(m, K);
        }
        float2 acc[RPW][NC];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[r][n] = make_float2(0.f, 0.f);
        for (int c0 = 0; c0 < chunks; c0 += seg_chunks) {
            const int c1 = c0 + seg_chunks < chunks ? c0 + seg_chunks : chunks;
            const int len = (c1 - c0) * F::kElems;
            if (nrows > 0) rs.start(crow, srow, c0, c1, lane);
            __syncthreads();
            stage_x_bf16<F>(x, K, NC, c0 * F::kElems, len, xs);
            __syncthreads();
            if (nrows > 0) rs.template run<NC>(xs, len, acc);
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float v = warp_sum(acc[r][n].x + acc[r][n].y);
                if (lane == 0 && r < nrows) y[n * M + r0 + r] = v * ts;
            }
    }
}

// ------------------------------------------------------------------ dequant
// w[m][k] = e2m1 * e4m3 * ts in fp32: e2m1 * e4m3 is exact in fp32, the
// multiply by ts rounds once to nearest.
__global__ void nvfp4_dequant_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                     float ts, float* __restrict__ w, int64_t M, int64_t K)
{
    const int64_t nbytes = M * (K / 2);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nbytes;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / (K / 2), kk = 2 * (i - m * (K / 2));
        const float s = e4m3_to_float(scales[m * (K / 16) + kk / 16]);
        uint32_t h[4];
        e2m1x8_to_f16x2(codes[i], h);  // only the first byte is used
        const float2 v = f16x2_to_float2(h[0]);
        w[m * K + kk] = (v.x * s) * ts;
        w[m * K + kk + 1] = (v.y * s) * ts;
    }
}

// w[m][k] = fp16(d) * q in fp32 (exact).
__global__ void q8_0_dequant_kernel(const int8_t* __restrict__ q, const uint16_t* __restrict__ d,
                                    float* __restrict__ w, int64_t M, int64_t K)
{
    const int64_t n = M * K;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / K, k = i - m * K;
        w[i] = fp16_to_float(d[m * (K / 32) + k / 32]) * static_cast<float>(q[i]);
    }
}

// w[m][k] = fp16(d) * (q - 8) in fp32 (exact), q from the GGUF Q4_0 block
// order (element j of a 32-block: low nibble of byte j for j < 16, high
// nibble of byte j - 16 otherwise). One thread per code byte.
__global__ void q4_0_dequant_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ d,
                                    float* __restrict__ w, int64_t M, int64_t K)
{
    const int64_t nbytes = M * (K / 2);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nbytes;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / (K / 2), bi = i - m * (K / 2);  // byte index within the row
        const int64_t k0 = (bi / 16) * 32 + bi % 16;          // element of the low nibble
        const float s = fp16_to_float(d[m * (K / 32) + k0 / 32]);
        const int c = codes[i];
        w[m * K + k0] = s * static_cast<float>((c & 15) - 8);
        w[m * K + k0 + 16] = s * static_cast<float>((c >> 4) - 8);
    }
}

// w[m][k] = fp16(d) * q + fp16(m) in fp32 (the exact value rounded once:
// one fused multiply-add), q in the Q4_0 block order. One thread per code
// byte (elements k0 and k0 + 16 of a block).
__global__ void q4_1_dequant_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ dm,
                                    float* __restrict__ w, int64_t M, int64_t K)
{
    const int64_t nbytes = M * (K / 2);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nbytes;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / (K / 2), bi = i - m * (K / 2);  // byte index within the row
        const int64_t k0 = (bi / 16) * 32 + bi % 16;          // element of the low nibble
        const uint16_t* f = dm + (m * (K / 32) + k0 / 32) * 2;
        const float d = fp16_to_float(f[0]), mn = fp16_to_float(f[1]);
        const int c = codes[i];
        w[m * K + k0] = fmaf(d, static_cast<float>(c & 15), mn);
        w[m * K + k0 + 16] = fmaf(d, static_cast<float>(c >> 4), mn);
    }
}

// w[m][k] = e4m3(code) * the fp32 scale of the 128 x 128 tile holding
// (m, k), in fp32: the E4M3 value is exact in fp32 and the one multiply
// rounds the exact product once to nearest. One thread per pair of codes
// (K is even, so a pair never straddles two rows).
__global__ void fp8_b128_dequant_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ scales,
                                        float* __restrict__ w, int64_t M, int64_t K)
{
    const int64_t npairs = M * K / 2, kt = (K + 127) / 128;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < npairs;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = (2 * i) / K, k = 2 * i - m * K;
        const float2 v = e4m3x2_to_float2(codes[2 * i] | (static_cast<uint32_t>(codes[2 * i + 1]) << 8));
        w[2 * i] = v.x * scales[(m / 128) * kt + k / 128];
        w[2 * i + 1] = v.y * scales[(m / 128) * kt + (k + 1) / 128];
    }
}

// ------------------------------------------------------------------ host
// Launch one (RPW, D) instantiation over a balanced grid filling every SM.
template <class F, int RPW, int NC, int D>
cudaError_t launch_cfg(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x, float* y, int64_t M,
                       int64_t K, int seg, cudaStream_t stream, int dev, int64_t* grid_out, bool dry)
{
    auto kern = gemv_kernel<F, RPW, NC, D>;
    static OccCache occ;
    const size_t smem = static_cast<size_t>(NC) * seg * sizeof(float);
    const int bps = blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kThreads, smem);
    int64_t grid = static_cast<int64_t>(dev_info(dev).sms) * bps;
    const int64_t need = (seg == K) ? (M + kWarps - 1) / kWarps : (M + kWarps * RPW - 1) / (kWarps * RPW);
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    *grid_out = grid;
    if (dry) return cudaSuccess;
    kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(codes, scales, ts, x, y, M, K, seg);
    return cudaGetLastError();
}

template <class F, int NC>
cudaError_t launch_nc(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x, float* y,
                      int64_t M, int64_t K, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int64_t budget = kXsBudgetBytes / 4 / NC;  // fp32 elements per column
    int seg = static_cast<int>(K);
    if (K > budget) seg = static_cast<int>(budget / F::kElems) * F::kElems;
    int64_t grid = 0;
    if constexpr (NC == 1) {
        // Rows per warp decide the group size: fewer rows -> smaller groups
        // with a deeper per-row prefetch, so no warp loads duplicate rows.
        launch_cfg<F, 4, 1, 2>(codes, scales, ts, x, y, M, K, seg, stream, dev, &grid, true);
        const int64_t rows_per_warp = M / (grid * kWarps);
        if (rows_per_warp >= 4 || seg != K)
            return launch_cfg<F, 4, 1, 2>(codes, scales, ts, x, y, M, K, seg, stream, dev, &grid, false);
        if (rows_per_warp >= 2)
            return launch_cfg<F, 2, 1, 4>(codes, scales, ts, x, y, M, K, seg, stream, dev, &grid, false);
        return launch_cfg<F, 1, 1, 8>(codes, scales, ts, x, y, M, K, seg, stream, dev, &grid, false);
    } else {
        constexpr int RPW = NC <= 4 ? 4 : 2;
        return launch_cfg<F, RPW, NC, 2>(codes, scales, ts, x, y, M, K, seg, stream, dev, &grid, false);
    }
}

template <class F>
cudaError_t launch_gemv(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x, float* y,
                        int64_t M, int64_t K, int N, cudaStream_t s)
{
    switch (N) {
#define BQD_CASE(n) \
    case n: return launch_nc<F, n>(codes, scales, ts, x, y, M, K, s);
        BQD_CASE(1) BQD_CASE(2) BQD_CASE(3) BQD_CASE(4) BQD_CASE(5) BQD_CASE(6) BQD_CASE(7) BQD_CASE(8)
        BQD_CASE(9) BQD_CASE(10) BQD_CASE(11) BQD_CASE(12) BQD_CASE(13) BQD_CASE(14) BQD_CASE(15) BQD_CASE(16)
#undef BQD_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_nvfp4_gemv_cuda_core(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                        float* y, int64_t M, int64_t K, int N, cudaStream_t s)
{
    if (K % 32 == 0) return launch_gemv<Nvfp4Vec>(codes, scales, ts, x, y, M, K, N, s);
    return launch_gemv<Nvfp4Narrow>(codes, scales, ts, x, y, M, K, N, s);
}

cudaError_t launch_q8_0_gemv_cuda_core(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M,
                                       int64_t K, int N, cudaStream_t s)
{
    return launch_gemv<Q8_0Fmt>(reinterpret_cast<const uint8_t*>(q), reinterpret_cast<const uint8_t*>(d), 1.0f, x,
                                y, M, K, N, s);
}

cudaError_t launch_q4_0_gemv_cuda_core(const uint8_t* codes, const uint16_t* d, const uint16_t* x, float* y,
                                       int64_t M, int64_t K, int N, cudaStream_t s)
{
    return launch_gemv<Q4_0Fmt>(codes, reinterpret_cast<const uint8_t*>(d), 1.0f, x, y, M, K, N, s);
}

cudaError_t launch_q4_1_gemv_cuda_core(const uint8_t* codes, const uint16_t* dm, const uint16_t* x, float* y,
                                       int64_t M, int64_t K, int N, cudaStream_t s)
{
    return launch_gemv<Q4_1Fmt>(codes, reinterpret_cast<const uint8_t*>(dm), 1.0f, x, y, M, K, N, s);
}

cudaError_t launch_fp8_b128_gemv_cuda_core(const uint8_t* codes, const float* scales, const uint16_t* x, float* y,
                                           int64_t M, int64_t K, int N, cudaStream_t s)
{
    return launch_gemv<Fp8B128Fmt>(codes, reinterpret_cast<const uint8_t*>(scales), 1.0f, x, y, M, K, N, s);
}

static unsigned dequant_grid(int64_t work)
{
    int64_t g = (work + 255) / 256;
    if (g > 152 * 16) g = 152 * 16;
    if (g < 1) g = 1;
    return static_cast<unsigned>(g);
}

cudaError_t launch_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float ts, float* w, int64_t M,
                                 int64_t K, cudaStream_t s)
{
    nvfp4_dequant_kernel<<<dequant_grid(M * K / 2), 256, 0, s>>>(codes, scales, ts, w, M, K);
    return cudaGetLastError();
}

cudaError_t launch_q8_0_dequant(const int8_t* q, const uint16_t* d, float* w, int64_t M, int64_t K, cudaStream_t s)
{
    q8_0_dequant_kernel<<<dequant_grid(M * K), 256, 0, s>>>(q, d, w, M, K);
    return cudaGetLastError();
}

cudaError_t launch_q4_0_dequant(const uint8_t* codes, const uint16_t* d, float* w, int64_t M, int64_t K,
                                cudaStream_t s)
{
    q4_0_dequant_kernel<<<dequant_grid(M * K / 2), 256, 0, s>>>(codes, d, w, M, K);
    return cudaGetLastError();
}

cudaError_t launch_q4_1_dequant(const uint8_t* codes, const uint16_t* dm, float* w, int64_t M, int64_t K,
                                cudaStream_t s)
{
    q4_1_dequant_kernel<<<dequant_grid(M * K / 2), 256, 0, s>>>(codes, dm, w, M, K);
    return cudaGetLastError();
}

cudaError_t launch_fp8_b128_dequant(const uint8_t* codes, const float* scales, float* w, int64_t M, int64_t K,
                                    cudaStream_t s)
{
    fp8_b128_dequant_kernel<<<dequant_grid(M * K / 2), 256, 0, s>>>(codes, scales, w, M, K);
    return cudaGetLastError();
}

}  // namespace bqd
