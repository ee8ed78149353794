// encode.cu -- bf16 weights to NVFP4 or Q8_0 on the GPU: re-encoding large
// tensors at load ("robertbfuentes7-cloud/bw24" README, safetensors loader
// bullet: FP8 and large BF16 tensors re-encode to Q8_0 / NVFP4 at load).
//
// NVFP4, per 16-element block of a row: s = E4M3(amax / 6 / ts) and each
// element's code = E2M1(w / (e4m3(s) * ts)); Q8_0, per 32-element block:
// d = fp16(amax / 127) and q = rint(w / d) clamped to [-127, 127]. Every
// value is an IEEE fp32 operation rounded to nearest even (explicit _rn
// intrinsics), and the conversions are the hardware's round-to-nearest-even
// ones that saturate (E4M3 at 448, E2M1 at 6), so the integer codes are a
// function of the input bits alone. A zero scale gives zero codes.
//
// One thread per block: it reads the block's 32 (NVFP4) or 64 (Q8_0)
// contiguous bytes with 16-byte loads, consecutive threads take consecutive
// blocks, so a warp reads 1 or 2 KiB and writes its codes contiguously.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "gemv.h"
#include "host_util.h"

namespace bqd {

namespace {

constexpr int kThE = 256;

// Two fp32 values to a byte of two E2M1 codes (lo in the low nibble).
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// An fp32 value to an E4M3 byte.
__device__ __forceinline__ uint32_t e4m3_rn(float v)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}

__global__ void __launch_bounds__(kThE)
    nvfp4_encode_kernel(const uint16_t* __restrict__ w, float ts, uint8_t* __restrict__ codes,
                        uint8_t* __restrict__ scales, int64_t nblk)
{
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * kThE + threadIdx.x; b < nblk;
         b += static_cast<int64_t>(gridDim.x) * kThE) {
        const uint4 p0 = reinterpret_cast<const uint4*>(w)[2 * b];
        const uint4 p1 = reinterpret_cast<const uint4*>(w)[2 * b + 1];
        const uint32_t wd[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        float f[16];
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            f[2 * j] = bf16_lo(wd[j]);
            f[2 * j + 1] = bf16_hi(wd[j]);
            amax = fmaxf(amax, fmaxf(fabsf(f[2 * j]), fabsf(f[2 * j + 1])));
        }
        const uint32_t sc = e4m3_rn(__fdiv_rn(__fdiv_rn(amax, 6.0f), ts));
        const float sdec = e4m3_to_float(sc);
        const float den = __fmul_rn(sdec, ts);
        uint32_t out[2] = {0u, 0u};
        if (sdec != 0.f) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t byte = e2m1x2_rn(__fdiv_rn(f[2 * j], den), __fdiv_rn(f[2 * j + 1], den));
                out[j / 4] |= byte << (8 * (j % 4));
            }
        }
        reinterpret_cast<uint2*>(codes)[b] = make_uint2(out[0], out[1]);
        scales[b] = static_cast<uint8_t>(sc);
    }
}

__global__ void __launch_bounds__(kThE)
    q8_0_encode_kernel(const uint16_t* __restrict__ w, int8_t* __restrict__ q, uint16_t* __restrict__ d,
                       int64_t nblk)
{
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * kThE + threadIdx.x; b < nblk;
         b += static_cast<int64_t>(gridDim.x) * kThE) {
        uint32_t wd[16];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint4 v = reinterpret_cast<const uint4*>(w)[4 * b + p];
            wd[4 * p] = v.x;
            wd[4 * p + 1] = v.y;
            wd[4 * p + 2] = v.z;
            wd[4 * p + 3] = v.w;
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(wd[j])), fabsf(bf16_hi(wd[j]))));
        const __half d16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
        const float d32 = __half2float(d16);
        uint32_t out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t word = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t pair = wd[2 * j + e / 2];
                const float x = (e & 1) ? bf16_hi(pair) : bf16_lo(pair);
                const float r = d32 != 0.f ? fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(x, d32)))) : 0.f;
                word |= (static_cast<uint32_t>(static_cast<int32_t>(r)) & 0xFFu) << (8 * e);
            }
            out[j] = word;
        }
        reinterpret_cast<uint4*>(q)[2 * b] = make_uint4(out[0], out[1], out[2], out[3]);
        reinterpret_cast<uint4*>(q)[2 * b + 1] = make_uint4(out[4], out[5], out[6], out[7]);
        d[b] = __half_as_ushort(d16);
    }
}

int encode_grid(int64_t nblk)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const int64_t want = (nblk + kThE - 1) / kThE, cap = static_cast<int64_t>(dev_info(dev).sms) * 8;
    return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_nvfp4_encode(const uint16_t* w, float ts, uint8_t* codes, uint8_t* scales, int64_t M, int64_t K,
                                cudaStream_t s)
{
    const int64_t nblk = M * (K / 16);
    nvfp4_encode_kernel<<<encode_grid(nblk), kThE, 0, s>>>(w, ts, codes, scales, nblk);
    return cudaGetLastError();
}

cudaError_t launch_q8_0_encode(const uint16_t* w, int8_t* q, uint16_t* d, int64_t M, int64_t K, cudaStream_t s)
{
    const int64_t nblk = M * (K / 32);
    q8_0_encode_kernel<<<encode_grid(nblk), kThE, 0, s>>>(w, q, d, nblk);
    return cudaGetLastError();
}

}  // namespace bqd
