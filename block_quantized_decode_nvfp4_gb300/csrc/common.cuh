// common.cuh -- device building blocks of the block-quantized decode matvec
// (sm_103a): streaming weight loads, in-register element decode, per-chunk dot
// products with fp32 accumulation, warp-shuffle reductions.
//
// What is computed follows the pages' decode path: NVFP4 weights (4-bit E2M1
// elements, an E4M3 scale per 16 consecutive k, one FP32 tensor scale) and
// Q8_0 weights (int8 with an fp16 scale per 32 k) multiplied into bf16
// activations with fp32 accumulation ("robertbfuentes7-cloud/bw24" README,
// NVFP4 (W4) decode path; "avifenesh/memra" README, Decode kernels;
// "Vemloir/LumenLLM" README, Kernels: warp-shuffle GEMVs).
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

namespace bqd {

constexpr int kWarp = 32;

// ------------------------------------------------------------------ loads
// Weights are read exactly once per call: bypass L1 allocation so the
// streamed bytes do not evict the activations staged next to them.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p)
{
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p)
{
    uint16_t r;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p)
{
    uint32_t r;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u8(const void* p)
{
    uint16_t r;
    asm("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return r & 0xFFu;
}

// ------------------------------------------------------------------ decode
// Four bytes of packed E2M1 codes (8 elements, low nibble = lower k) to four
// f16x2 pairs with the hardware FP4 -> f16x2 conversion (exact: every E2M1
// value is an f16). Pair j holds elements 2j (low half) and 2j+1 (high half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4])
{
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// Two E4M3 bytes (low byte first) to f32 (exact: E4M3 values are f16 values).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_bytes)
{
    uint32_t h;
    uint16_t b = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(b));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte)
{
    return e4m3x2_to_float2(byte & 0xFFu).x;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h)
{
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

__device__ __forceinline__ float fp16_to_float(uint32_t bits)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// Four int8 (one 32-bit word) to fp32 without the int->float conversion
// unit: flip the sign bit to get q + 128 in [1, 255], place it in the low
// mantissa byte of 2^23 (the float 2^23 + q + 128), subtract 2^23 + 128.
// Exact for every int8 value.
__device__ __forceinline__ void s8x4_to_float(uint32_t w, float2& lo, float2& hi)
{
    const uint32_t u = w ^ 0x80808080u;
    const float2 bias = make_float2(8388736.0f, 8388736.0f);  // 2^23 + 128
    float2 a = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)),
                           __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)));
    float2 b = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)),
                           __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)));
    lo = __fadd2_rn(a, make_float2(-bias.x, -bias.y));
    hi = __fadd2_rn(b, make_float2(-bias.x, -bias.y));
}

// Four bytes holding 4-bit codes q (0..15) to fp32 q - 8, exactly: the byte
// is the low mantissa byte of 2^23, so the float reads 2^23 + q.
__device__ __forceinline__ void u4x4_to_float(uint32_t w, float2& lo, float2& hi)
{
    const float2 bias = make_float2(8388616.0f, 8388616.0f);  // 2^23 + 8
    float2 a = make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540)),
                           __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7541)));
    float2 b = make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7542)),
                           __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7543)));
    lo = __fadd2_rn(a, make_float2(-bias.x, -bias.y));
    hi = __fadd2_rn(b, make_float2(-bias.x, -bias.y));
}

// ------------------------------------------------------------------ formats
// A "chunk" is the unit one lane loads and multiplies per row: a run of
// consecutive k of one weight row, with its block scales.
//
//   Nvfp4Vec:    32 elements = 16 code bytes + 2 scale bytes (needs K % 32 == 0)
//   Nvfp4Narrow: 16 elements =  8 code bytes + 1 scale byte
//   Q8_0Fmt:     32 elements = 32 int8 + 1 fp16 scale
//
// dot<RPW, NC>() adds, for RPW rows (one chunk each, same k range) and NC
// activation columns held in shared memory as fp32 (column n at
// xs + n * xstride), the partial sums  sum_k w[r][k] * x[n][k]  with block
// scales applied and the tensor scale not, into acc[r][n] (an even/odd pair
// of fp32 partial sums; the row total is .x + .y). Each activation value is
// read from shared memory once per chunk for all RPW rows.

// E2M1 x E4M3 products have at most 6 significant bits and lie in
// [2^-10, 2688], so scaling the decoded f16 elements by the f16 block scale
// is exact.
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b)
{
    __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// Two E4M3 bytes to f16x2 (bits), low byte in the low half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes)
{
    uint32_t h;
    uint16_t b = static_cast<uint16_t>(two_bytes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(b));
    return h;
}

// One word of E2M1 codes (8 elements) of each row times NC columns.
// With kScaled the block scale is already folded into the elements.
template <int RPW, int NC>
__device__ __forceinline__ void nvfp4_word(const uint32_t (&w)[RPW], const uint32_t (&s2)[RPW], const float* xs,
                                           int xstride, int piece, int sw, float2 (&acc)[RPW][NC])
{
    float2 wf[RPW][4];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        uint32_t h[4];
        e2m1x8_to_f16x2(w[r], h);
#pragma unroll
        for (int q = 0; q < 4; ++q) wf[r][q] = f16x2_to_float2(hmul2_bits(h[q], s2[r]));
    }
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        const float4 xa = *reinterpret_cast<const float4*>(xs + n * xstride + ((piece ^ sw) << 2));
        const float4 xb = *reinterpret_cast<const float4*>(xs + n * xstride + (((piece + 1) ^ sw) << 2));
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            acc[r][n] = __ffma2_rn(wf[r][0], make_float2(xa.x, xa.y), acc[r][n]);
            acc[r][n] = __ffma2_rn(wf[r][1], make_float2(xa.z, xa.w), acc[r][n]);
            acc[r][n] = __ffma2_rn(wf[r][2], make_float2(xb.x, xb.y), acc[r][n]);
            acc[r][n] = __ffma2_rn(wf[r][3], make_float2(xb.z, xb.w), acc[r][n]);
        }
    }
}

// One 16-element block of each row, one column, scale applied per block
// (cheaper than scaling every element when there is a single column).
template <int RPW>
__device__ __forceinline__ void nvfp4_block_n1(const uint32_t (&w0)[RPW], const uint32_t (&w1)[RPW],
                                               const float (&s)[RPW], const float* xs, int piece, int sw,
                                               float2 (&acc)[RPW][1])
{
    float2 part[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) part[r] = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float4 xa = *reinterpret_cast<const float4*>(xs + (((piece + 2 * j) ^ sw) << 2));
        const float4 xb = *reinterpret_cast<const float4*>(xs + (((piece + 2 * j + 1) ^ sw) << 2));
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            uint32_t h[4];
            e2m1x8_to_f16x2(j ? w1[r] : w0[r], h);
            part[r] = __ffma2_rn(f16x2_to_float2(h[0]), make_float2(xa.x, xa.y), part[r]);
            part[r] = __ffma2_rn(f16x2_to_float2(h[1]), make_float2(xa.z, xa.w), part[r]);
            part[r] = __ffma2_rn(f16x2_to_float2(h[2]), make_float2(xb.x, xb.y), part[r]);
            part[r] = __ffma2_rn(f16x2_to_float2(h[3]), make_float2(xb.z, xb.w), part[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) acc[r][0].x = fmaf(s[r], part[r].x + part[r].y, acc[r][0].x);
}

// Activations are staged in shared memory chunk by chunk (kElems fp32 per
// chunk), the 16-byte pieces of chunk c permuted by XOR with swz(c), so that
// the 32 lanes of a warp, which read the same piece of 32 consecutive
// chunks, hit distinct banks.
struct Nvfp4Vec {
    static constexpr int kElems = 32;
    __device__ static __forceinline__ int swz(int c) { return c & 7; }
    struct Chunk {
        uint4 c;
        uint32_t s;
    };
    __device__ static __forceinline__ Chunk load(const uint8_t* codes_row, const uint8_t* scales_row, int c)
    {
        Chunk ch;
        ch.c = ld_stream_v4(codes_row + 16 * c);
        ch.s = ld_stream_u16(scales_row + 2 * c);
        return ch;
    }
    template <int RPW, int NC>
    __device__ static __forceinline__ void dot(const Chunk (&ch)[RPW], const float* xs, int xstride, int sw,
                                               float2 (&acc)[RPW][NC])
    {
        if constexpr (NC == 1) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                uint32_t w0[RPW], w1[RPW];
                float s[RPW];
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    const uint32_t words[4] = {ch[r].c.x, ch[r].c.y, ch[r].c.z, ch[r].c.w};
                    w0[r] = words[2 * b];
                    w1[r] = words[2 * b + 1];
                    const float2 sc = e4m3x2_to_float2(ch[r].s);
                    s[r] = b ? sc.y : sc.x;
                }
                nvfp4_block_n1<RPW>(w0, w1, s, xs, 4 * b, sw, acc);
            }
        } else {
            uint32_t sb[2][RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const uint32_t s2 = e4m3x2_to_f16x2(ch[r].s);
                sb[0][r] = __byte_perm(s2, 0, 0x1010);  // block 0 scale in both halves
                sb[1][r] = __byte_perm(s2, 0, 0x3232);  // block 1 scale in both halves
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t w[RPW];
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    const uint32_t words[4] = {ch[r].c.x, ch[r].c.y, ch[r].c.z, ch[r].c.w};
                    w[r] = words[j];
                }
                nvfp4_word<RPW, NC>(w, sb[j / 2], xs, xstride, 2 * j, sw, acc);
            }
        }
    }
};

struct Nvfp4Narrow {
    static constexpr int kElems = 16;
    __device__ static __forceinline__ int swz(int c) { return (c >> 1) & 3; }
    struct Chunk {
        uint2 c;
        uint32_t s;
    };
    __device__ static __forceinline__ Chunk load(const uint8_t* codes_row, const uint8_t* scales_row, int c)
    {
        Chunk ch;
        ch.c = ld_stream_v2(codes_row + 8 * c);
        ch.s = ld_stream_u8(scales_row + c);
        return ch;
    }
    template <int RPW, int NC>
    __device__ static __forceinline__ void dot(const Chunk (&ch)[RPW], const float* xs, int xstride, int sw,
                                               float2 (&acc)[RPW][NC])
    {
        uint32_t sb[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) sb[r] = __byte_perm(e4m3x2_to_f16x2(ch[r].s), 0, 0x1010);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t w[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) w[r] = j ? ch[r].c.y : ch[r].c.x;
            nvfp4_word<RPW, NC>(w, sb, xs, xstride, 2 * j, sw, acc);
        }
    }
};

struct Q8_0Fmt {
    static constexpr int kElems = 32;
    __device__ static __forceinline__ int swz(int c) { return c & 7; }
    struct Chunk {
        uint4 a, b;
        uint32_t d;
    };
    // For Q8_0 "codes_row" is the int8 row and "scales_row" the fp16 row.
    __device__ static __forceinline__ Chunk load(const uint8_t* q_row, const uint8_t* d_row, int c)
    {
        Chunk ch;
        ch.a = ld_stream_v4(q_row + 32 * c);
        ch.b = ld_stream_v4(q_row + 32 * c + 16);
        ch.d = ld_stream_u16(d_row + 2 * c);
        return ch;
    }
    template <int RPW, int NC>
    __device__ static __forceinline__ void dot(const Chunk (&ch)[RPW], const float* xs, int xstride, int sw,
                                               float2 (&acc)[RPW][NC])
    {
        float2 part[RPW][NC];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) part[r][n] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float2 lo[RPW], hi[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const uint32_t words[8] = {ch[r].a.x, ch[r].a.y, ch[r].a.z, ch[r].a.w,
                                           ch[r].b.x, ch[r].b.y, ch[r].b.z, ch[r].b.w};
                s8x4_to_float(words[j], lo[r], hi[r]);
            }
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float4 xv = *reinterpret_cast<const float4*>(xs + n * xstride + ((j ^ sw) << 2));
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    part[r][n] = __ffma2_rn(lo[r], make_float2(xv.x, xv.y), part[r][n]);
                    part[r][n] = __ffma2_rn(hi[r], make_float2(xv.z, xv.w), part[r][n]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float d = fp16_to_float(ch[r].d);
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[r][n].x = fmaf(d, part[r][n].x + part[r][n].y, acc[r][n].x);
        }
    }
};

// Q4_0: a 32-element chunk is one block, 16 code bytes (byte j: element j
// in the low nibble, element j + 16 in the high nibble, the GGUF block
// order) and one fp16 scale; element = d * (q - 8).
struct Q4_0Fmt {
    static constexpr int kElems = 32;
    __device__ static __forceinline__ int swz(int c) { return c & 7; }
    struct Chunk {
        uint4 c;
        uint32_t d;
    };
    __device__ static __forceinline__ Chunk load(const uint8_t* codes_row, const uint8_t* d_row, int c)
    {
        Chunk ch;
        ch.c = ld_stream_v4(codes_row + 16 * c);
        ch.d = ld_stream_u16(d_row + 2 * c);
        return ch;
    }
    template <int RPW, int NC>
    __device__ static __forceinline__ void dot(const Chunk (&ch)[RPW], const float* xs, int xstride, int sw,
                                               float2 (&acc)[RPW][NC])
    {
        float2 part[RPW][NC];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) part[r][n] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // code word j: elements 4j .. 4j+3 (low nibbles), 16+4j .. (high)
            float2 l01[RPW], l23[RPW], h01[RPW], h23[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const uint32_t words[4] = {ch[r].c.x, ch[r].c.y, ch[r].c.z, ch[r].c.w};
                u4x4_to_float(words[j] & 0x0F0F0F0Fu, l01[r], l23[r]);
                u4x4_to_float((words[j] >> 4) & 0x0F0F0F0Fu, h01[r], h23[r]);
            }
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float4 xl = *reinterpret_cast<const float4*>(xs + n * xstride + ((j ^ sw) << 2));
                const float4 xh = *reinterpret_cast<const float4*>(xs + n * xstride + (((4 + j) ^ sw) << 2));
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
            const float d = fp16_to_float(ch[r].d);
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[r][n].x = fmaf(d, part[r][n].x + part[r][n].y, acc[r][n].x);
        }
    }
};

// FP8 block-128: a 32-element chunk is 32 E4M3 bytes in element order; its
// fp32 scale is the one of the 128-element k tile holding it (four chunks
// share it), and 128 consecutive rows share one row of scales.
struct Fp8B128Fmt {
    static constexpr int kElems = 32;
    __device__ static __forceinline__ int swz(int c) { return c & 7; }
    struct Chunk {
        uint4 a, b;
        uint32_t s;
    };
    __device__ static __forceinline__ Chunk load(const uint8_t* codes_row, const uint8_t* scales_row, int c)
    {
        Chunk ch;
        ch.a = ld_stream_v4(codes_row + 32 * c);
        ch.b = ld_stream_v4(codes_row + 32 * c + 16);
        ch.s = ld_stream_u32(scales_row + 4 * (c >> 2));
        return ch;
    }
    template <int RPW, int NC>
    __device__ static __forceinline__ void dot(const Chunk (&ch)[RPW], const float* xs, int xstride, int sw,
                                               float2 (&acc)[RPW][NC])
    {
        float2 part[RPW][NC];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) part[r][n] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {  // word j: elements 4j .. 4j + 3
            float2 lo[RPW], hi[RPW];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const uint32_t words[8] = {ch[r].a.x, ch[r].a.y, ch[r].a.z, ch[r].a.w,
                                           ch[r].b.x, ch[r].b.y, ch[r].b.z, ch[r].b.w};
                lo[r] = e4m3x2_to_float2(words[j]);
                hi[r] = e4m3x2_to_float2(words[j] >> 16);
            }
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float4 xv = *reinterpret_cast<const float4*>(xs + n * xstride + ((j ^ sw) << 2));
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    part[r][n] = __ffma2_rn(lo[r], make_float2(xv.x, xv.y), part[r][n]);
                    part[r][n] = __ffma2_rn(hi[r], make_float2(xv.z, xv.w), part[r][n]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float s = __uint_as_float(ch[r].s);
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[r][n].x = fmaf(s, part[r][n].x + part[r][n].y, acc[r][n].x);
        }
    }
};

// Bytes of the codes plane per weight row; bytes of one row of the scales
// plane; and the byte offset of weight row m's scales (rows share a scale
// row only in the FP8 block-128 format).
template <class F>
struct RowPitch;
template <>
struct RowPitch<Nvfp4Vec> {
    __host__ __device__ static int64_t codes(int64_t K) { return K / 2; }
    __host__ __device__ static int64_t scales(int64_t K) { return K / 16; }
    __host__ __device__ static int64_t srow(int64_t m, int64_t K) { return m * scales(K); }
};
template <>
struct RowPitch<Nvfp4Narrow> {
    __host__ __device__ static int64_t codes(int64_t K) { return K / 2; }
    __host__ __device__ static int64_t scales(int64_t K) { return K / 16; }
    __host__ __device__ static int64_t srow(int64_t m, int64_t K) { return m * scales(K); }
};
template <>
struct RowPitch<Q8_0Fmt> {
    __host__ __device__ static int64_t codes(int64_t K) { return K; }
    __host__ __device__ static int64_t scales(int64_t K) { return (K / 32) * 2; }
    __host__ __device__ static int64_t srow(int64_t m, int64_t K) { return m * scales(K); }
};
template <>
struct RowPitch<Q4_0Fmt> {
    __host__ __device__ static int64_t codes(int64_t K) { return K / 2; }
    __host__ __device__ static int64_t scales(int64_t K) { return (K / 32) * 2; }
    __host__ __device__ static int64_t srow(int64_t m, int64_t K) { return m * scales(K); }
};
template <>
struct RowPitch<Fp8B128Fmt> {
    __host__ __device__ static int64_t codes(int64_t K) { return K; }
    __host__ __device__ static int64_t scales(int64_t K) { return (K + 127) / 128 * 4; }
    __host__ __device__ static int64_t srow(int64_t m, int64_t K) { return (m >> 7) * scales(K); }
};

// ------------------------------------------------------------------ rows
// A stream of chunk loads for RPW weight rows over chunks [c_begin, c_end),
// spread over a group of LG lanes (lane g of the group takes chunks
// c_begin + g, c_begin + g + LG, ...), keeping D chunks of every row in
// flight in a register ring. start() issues the first D loads and may be
// called long before run() (e.g. before the activations are staged), so
// the HBM latency of the first loads overlaps that work.
// Every row pointer must address a valid row (callers repeat a valid row for
// the unused slots of a partial group).
template <class F, int RPW, int D, int LG = kWarp>
struct RowStream {
    using Chunk = typename F::Chunk;
    Chunk buf[D][RPW];
    const uint8_t* crow[RPW];
    const uint8_t* srow[RPW];
    int c0, c_end, g;

    __device__ __forceinline__ void start(const uint8_t* const (&codes_row)[RPW],
                                          const uint8_t* const (&scales_row)[RPW], int c_begin, int c_stop,
                                          int lane_in_group)
    {
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            crow[r] = codes_row[r];
            srow[r] = scales_row[r];
        }
        c0 = c_begin;
        c_end = c_stop;
        g = lane_in_group;
#pragma unroll
        for (int i = 0; i < D; ++i) {
            const int c = c0 + g + i * LG;
            if (c < c_end) {
#pragma unroll
                for (int r = 0; r < RPW; ++r) buf[i][r] = F::load(crow[r], srow[r], c);
            }
        }
    }

    // acc[r][n] += this lane's partial sums over its chunks; xs points at the
    // activation of chunk c_begin (column n at xs + n * xstride).
    template <int NC>
    __device__ __forceinline__ void run(const float* xs, int xstride, float2 (&acc)[RPW][NC])
    {
        for (int base = c0 + g; base < c_end; base += D * LG) {
#pragma unroll
            for (int i = 0; i < D; ++i) {
                const int c = base + i * LG;
                if (c < c_end) {
                    const int cn = c + D * LG;
                    Chunk nxt[RPW];
                    if (cn < c_end) {
#pragma unroll
                        for (int r = 0; r < RPW; ++r) nxt[r] = F::load(crow[r], srow[r], cn);
                    }
                    F::template dot<RPW, NC>(buf[i], xs + (c - c0) * F::kElems, xstride, F::swz(c - c0), acc);
                    if (cn < c_end) {
#pragma unroll
                        for (int r = 0; r < RPW; ++r) buf[i][r] = nxt[r];
                    }
                }
            }
        }
    }
};

// Sum over aligned groups of LG lanes (every lane of the group gets the sum).
template <int LG = kWarp>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = LG / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_sum(float v) { return group_sum<kWarp>(v); }

// Stage ncols bf16 activation columns x[n][k0 .. k0+len) (row pitch K) into
// shared memory as fp32 in the swizzled chunk layout of format F, column n
// at xs + n * len. Needs len % F::kElems == 0, k0 % 4 == 0, K % 4 == 0 and
// an 8-byte aligned x.
template <class F>
__device__ __forceinline__ void stage_x_bf16(const uint16_t* x, int64_t K, int ncols, int k0, int len, float* xs)
{
    constexpr int P = F::kElems / 4;  // 16-byte pieces per chunk
    const int pieces = len / 4;
    const int total = ncols * pieces;
#pragma unroll 4
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int n = i / pieces, q = i - n * pieces;
        const uint2 u = *reinterpret_cast<const uint2*>(x + n * K + k0 + 4 * q);
        const int c = q / P, j = q % P;
        *reinterpret_cast<float4*>(xs + n * len + c * F::kElems + ((j ^ F::swz(c)) << 2)) =
            make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    }
}

// Put one 16-byte piece (4 fp32, global piece index q of a column) at its
// swizzled place in the chunk layout of format F.
template <class F>
__device__ __forceinline__ void put_piece(float* col, int q, float4 v)
{
    constexpr int P = F::kElems / 4;
    const int c = q / P, j = q % P;
    *reinterpret_cast<float4*>(col + c * F::kElems + ((j ^ F::swz(c)) << 2)) = v;
}

}  // namespace bqd
