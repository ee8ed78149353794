// q4_1.cuh -- the Q4_1 block format on the CUDA-core GEMV path: GGUF's
// Q4_1 block ("robertbfuentes7-cloud/bw24" README, GGUF bullet: files mix
// BF16, Q8_0, Q4_0, Q4_1 and the K-quants), split into a code plane (16
// bytes per 32 elements, the Q4_0 nibble order: byte j holds element j in
// its low and element j + 16 in its high nibble) and a (d, m) plane (the
// block's two fp16 fields side by side); w = d * q + m.
//
// Per chunk (one block) and column: sum w x = d * sum q x + m * sum x. The
// codes decode exactly to fp32 q, q x is exact in fp32, and sum x of the
// chunk is taken once per column, not per row.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace bqd {

// Four bytes holding 4-bit codes q (0..15) to fp32 q, exactly: the byte is
// the low mantissa byte of 2^23, so the float reads 2^23 + q.
__device__ __forceinline__ void u4x4_to_float_q(uint32_t w, float2& lo, float2& hi)
{
    const float2 a = make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540)),
                                 __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541)));
    const float2 b = make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542)),
                                 __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543)));
    lo = __fadd2_rn(a, make_float2(-8388608.0f, -8388608.0f));
    hi = __fadd2_rn(b, make_float2(-8388608.0f, -8388608.0f));
}

struct Q4_1Fmt {
    static constexpr int kElems = 32;
    __device__ static __forceinline__ int swz(int c) { return c & 7; }
    struct Chunk {
        uint4 c;
        uint32_t dm;  // d in the low half, m in the high half (fp16 bits)
    };
    __device__ static __forceinline__ Chunk load(const uint8_t* codes_row, const uint8_t* dm_row, int c)
    {
        Chunk ch;
        ch.c = ld_stream_v4(codes_row + 16 * c);
        ch.dm = ld_stream_u32(dm_row + 4 * c);
        return ch;
    }
    template <int RPW, int NC>
    __device__ static __forceinline__ void dot(const Chunk (&ch)[RPW], const float* xs, int xstride, int sw,
                                               float2 (&acc)[RPW][NC])
    {
        float2 part[RPW][NC];
        float2 sx[NC];
#pragma unroll
        for (int n = 0; n < NC; ++n) {
            sx[n] = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < RPW; ++r) part[r][n] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // code word j: elements 4j .. 4j+3 (low nibbles), 16+4j .. (high)
            float2 l01[RPW], l23[RPW], h01[RPW], h23[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const uint32_t words[4] = {ch[r].c.x, ch[r].c.y, ch[r].c.z, ch[r].c.w};
                u4x4_to_float_q(words[j] & 0x0F0F0F0Fu, l01[r], l23[r]);
                u4x4_to_float_q((words[j] >> 4) & 0x0F0F0F0Fu, h01[r], h23[r]);
            }
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float4 xl = *reinterpret_cast<const float4*>(xs + n * xstride + ((j ^ sw) << 2));
                const float4 xh = *reinterpret_cast<const float4*>(xs + n * xstride + (((4 + j) ^ sw) << 2));
                sx[n] = __fadd2_rn(sx[n], __fadd2_rn(make_float2(xl.x, xl.y), make_float2(xl.z, xl.w)));
                sx[n] = __fadd2_rn(sx[n], __fadd2_rn(make_float2(xh.x, xh.y), make_float2(xh.z, xh.w)));
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    part[r][n] = __ffma2_rn(l01[r], make_float2(xl.x, xl.y), part[r][n]);
                    part[r][n] = __ffma2_rn(l23[r], make_float2(xl.z, xl.w), part[r][n]);
                    part[r][n] = __ffma2_rn(h01[r], make_float2(xh.x, xh.y), part[r][n]);
                    part[r][n] = __ffma2_rn(h23[r], make_float2(xh.z, xh.w), part[r][n]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float d = fp16_to_float(ch[r].dm & 0xFFFFu), m = fp16_to_float(ch[r].dm >> 16);
#pragma unroll
            for (int n = 0; n < NC; ++n)
                acc[r][n].x = fmaf(d, part[r][n].x + part[r][n].y, fmaf(m, sx[n].x + sx[n].y, acc[r][n].x));
        }
    }
};

template <>
struct RowPitch<Q4_1Fmt> {
    __host__ __device__ static int64_t codes(int64_t K) { return K / 2; }
    __host__ __device__ static int64_t scales(int64_t K) { return (K / 32) * 4; }
    __host__ __device__ static int64_t srow(int64_t m, int64_t K) { return m * scales(K); }
};

// Q4_1 on the CUDA-core path (any M, K % 32 == 0, 1 <= N <= 16) and its
// dequantisation (gemv.cu).
cudaError_t launch_q4_1_gemv_cuda_core(const uint8_t* codes, const uint16_t* dm, const uint16_t* x, float* y,
                                       int64_t M, int64_t K, int N, cudaStream_t s);
cudaError_t launch_q4_1_dequant(const uint8_t* codes, const uint16_t* dm, float* w, int64_t M, int64_t K,
                                cudaStream_t s);

}  // namespace bqd
