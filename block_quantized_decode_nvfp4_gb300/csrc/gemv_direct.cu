// gemv_direct.cu -- GEMV for one token (N = 1), NVFP4 and Q8_0, streaming
// the weights straight from HBM into registers.
//
// y[m] = ts * sum_b scale[m][b] * sum_{k in b} elem[m][k] * x[k]
// ("robertbfuentes7-cloud/bw24" README, NVFP4 (W4) decode path;
// "avifenesh/memra" README, Decode kernels: NVFP4, Q4_0 and Q8_0 matvecs;
// "Vemloir/LumenLLM" README, Kernels: warp-shuffle GEMVs).
//
// Every warp owns a contiguous, balanced range of rows and reads each row
// with fully coalesced 16-byte loads: lane l takes the 32-element chunks
// l, l + 32, ... of the row (16 code bytes and 2 scale bytes each for NVFP4,
// 16 code bytes and one fp16 scale for Q4_0, 32 int8 and one fp16 scale for
// Q8_0). K is a multiple of 1024, so a row is
// CPL = K / 1024 such chunks per lane, a compile-time constant: the loop
// over a row is unrolled and every load offset and every activation offset
// is an immediate. D chunks per lane stay in flight in registers (a ring
// indexed at compile time). The first D are requested before the kernel
// waits for the previous kernel in the stream (programmatic dependent
// launch), so they overlap its tail.
//
// Activations are staged once per CTA in shared memory as f16 after an exact
// power-of-two prescale (chosen from their largest exponent; f16 then holds
// every bf16 value exactly when all nonzero magnitudes lie within 31
// binades of the largest) and multiplied in by the mixed-precision FMA
// (f16 x f16 products are exact in fp32; sums fp32). Outside that range, or
// with subnormal, inf or NaN activations, the CTA keeps the bf16 values and
// uses fp32 FMAs (exact products as well). Block scales multiply 16-element
// partial sums; the tensor scale and the prescale's inverse multiply the
// warp-shuffle row sum. Results are deterministic.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "common.cuh"
#include "gemv.h"
#include "host_util.h"

namespace bqd {

namespace {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Two fp32 accumulators += (lo, hi) f16 halves of w2 times those of x2.
__device__ __forceinline__ void fma_f16x2(uint32_t w2, uint32_t x2, float& a0, float& a1)
{
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(w2), "r"(x2));
}

// Four int8 (one word) to two f16x2 pairs, exactly: the byte q + 128 is the
// low mantissa byte of the f16 0x6400 (= 1024), so the pair reads 1024 +
// q + 128; subtracting 1152 leaves q.
__device__ __forceinline__ void s8x4_to_f16x2(uint32_t w, uint32_t& p01, uint32_t& p23)
{
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    p01 = *reinterpret_cast<uint32_t*>(&ha);
    p23 = *reinterpret_cast<uint32_t*>(&hb);
}

// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Activations: 32-element chunks of 64 bytes (f16, or the raw bf16 in exact
// mode); the 16-byte piece p of chunk c sits at slot p ^ ((c >> 1) & 3), so
// the 32 lanes, which read the same piece of 32 consecutive chunks, hit
// distinct banks. Lane l's chunks are l + 32 i: its swizzle depends on l
// only, and chunk l + 32 i starts 1024 i elements after chunk l.
__device__ __forceinline__ int x_index(int c, int p) { return c * 32 + ((p ^ ((c >> 1) & 3)) << 3); }

struct Nvfp4Item {  // 32 elements of one row: 16 code bytes, two E4M3 scales
    uint4 c;
    uint32_t s;
};
struct Q8Item {  // 32 elements of one row: 32 int8, one fp16 scale
    uint4 a, b;
    uint32_t d;
};

// Scale addressing of a format: weight row pr's scales start at
// srow(pr) * spitch(K) bytes, and lane l's chunk of each 1024-element step
// nc finds its scale at slane(l) + nc * kSChunk bytes from there. Here: one
// 2-byte scale per 32-element chunk and per row.
struct DirScale16 {
    static constexpr int kSChunk = 64;
    __host__ __device__ static constexpr int64_t spitch(int64_t K) { return K / 16; }
    __device__ static __forceinline__ int64_t srow(int64_t pr) { return pr; }
    __device__ static __forceinline__ int slane(int lane) { return lane * 2; }
};

struct DirNvfp4 : DirScale16 {
    using Item = Nvfp4Item;
    static constexpr int kCodeBytes = 16;  // per 32-element chunk
    __device__ static __forceinline__ Item load(const uint8_t* c, const uint8_t* s)
    {
        Item it;
        it.c = ld_stream_v4(c);
        it.s = ld_stream_u16(s);
        return it;
    }
    // xc: this lane's chunk in shared memory; sw: its swizzle
    template <bool FAST>
    __device__ static __forceinline__ void dot(const Item& it, const uint16_t* xc, int sw, float& acc)
    {
        const float2 sc = e4m3x2_to_float2(it.s);
        const uint32_t words[4] = {it.c.x, it.c.y, it.c.z, it.c.w};
#pragma unroll
        for (int b = 0; b < 2; ++b) {  // 16-element blocks
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int wi = 2 * b + j;  // elements 8 wi .. 8 wi + 7 = activation piece wi
                const uint4 xq = *reinterpret_cast<const uint4*>(xc + ((wi ^ sw) << 3));
                const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
                uint32_t h[4];
                e2m1x8_to_f16x2(words[wi], h);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (FAST) {
                        fma_f16x2(h[q], xp[q], a0, a1);
                    } else {
                        const float2 wf = f16x2_to_float2(h[q]);
                        a0 = fmaf(wf.x, bf16_lo(xp[q]), a0);
                        a1 = fmaf(wf.y, bf16_hi(xp[q]), a1);
                    }
                }
            }
            acc = fmaf(b ? sc.y : sc.x, a0 + a1, acc);
        }
    }
};

// Q4_0: the chunk is one block; code byte j holds element j (low nibble) and
// element j + 16 (high nibble), the GGUF order, so word w of the chunk holds
// elements 4w .. 4w + 3 and 16 + 4w .. 16 + 4w + 3: activation pieces w / 2
// and 2 + w / 2. q - 8 is exact in f16 (1024 + q from the byte's mantissa
// bits, minus 1032).
struct DirQ4 : DirScale16 {
    using Item = Nvfp4Item;  // 16 code bytes, the fp16 scale
    static constexpr int kCodeBytes = 16;
    __device__ static __forceinline__ Item load(const uint8_t* c, const uint8_t* s)
    {
        Item it;
        it.c = ld_stream_v4(c);
        it.s = ld_stream_u16(s);
        return it;
    }
    template <bool FAST>
    __device__ static __forceinline__ void dot(const Item& it, const uint16_t* xc, int sw, float& acc)
    {
        const uint32_t words[4] = {it.c.x, it.c.y, it.c.z, it.c.w};
        uint4 xq[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) xq[p] = *reinterpret_cast<const uint4*>(xc + ((p ^ sw) << 3));
        const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t nib[2] = {words[w] & 0x0F0F0F0Fu, (words[w] >> 4) & 0x0F0F0F0Fu};
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // h = 0: elements 4w.., piece w / 2; h = 1: 16 + 4w.., piece 2 + w / 2
                const uint4 xv = xq[2 * h + w / 2];
                const uint32_t xp[4] = {xv.x, xv.y, xv.z, xv.w};
                const uint32_t x01 = xp[(w % 2) * 2], x23 = xp[(w % 2) * 2 + 1];
                uint32_t p01 = __byte_perm(nib[h], 0x64646464u, 0x4140);
                uint32_t p23 = __byte_perm(nib[h], 0x64646464u, 0x4342);
                __half2 q01 = __hsub2(*reinterpret_cast<__half2*>(&p01), bias);
                __half2 q23 = __hsub2(*reinterpret_cast<__half2*>(&p23), bias);
                const uint32_t w01 = *reinterpret_cast<uint32_t*>(&q01), w23 = *reinterpret_cast<uint32_t*>(&q23);
                if constexpr (FAST) {
                    fma_f16x2(w01, x01, a0, a1);
                    fma_f16x2(w23, x23, a0, a1);
                } else {
                    const float2 f01 = f16x2_to_float2(w01), f23 = f16x2_to_float2(w23);
                    a0 = fmaf(f01.x, bf16_lo(x01), a0);
                    a1 = fmaf(f01.y, bf16_hi(x01), a1);
                    a0 = fmaf(f23.x, bf16_lo(x23), a0);
                    a1 = fmaf(f23.y, bf16_hi(x23), a1);
                }
            }
        }
        acc = fmaf(fp16_to_float(it.s), a0 + a1, acc);
    }
};

struct DirQ8 : DirScale16 {
    using Item = Q8Item;
    static constexpr int kCodeBytes = 32;
    __device__ static __forceinline__ Item load(const uint8_t* c, const uint8_t* s)
    {
        Item it;
        it.a = ld_stream_v4(c);
        it.b = ld_stream_v4(c + 16);
        it.d = ld_stream_u16(s);
        return it;
    }
    template <bool FAST>
    __device__ static __forceinline__ void dot(const Item& it, const uint16_t* xc, int sw, float& acc)
    {
        const uint32_t words[8] = {it.a.x, it.a.y, it.a.z, it.a.w, it.b.x, it.b.y, it.b.z, it.b.w};
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int p = 0; p < 4; ++p) {  // 8 elements = 2 int8 words = activation piece p
            const uint4 xq = *reinterpret_cast<const uint4*>(xc + ((p ^ sw) << 3));
            const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t w = words[2 * p + h];
                if constexpr (FAST) {
                    uint32_t q01, q23;
                    s8x4_to_f16x2(w, q01, q23);
                    fma_f16x2(q01, xp[2 * h], a0, a1);
                    fma_f16x2(q23, xp[2 * h + 1], a0, a1);
                } else {
                    float2 lo, hi;
                    s8x4_to_float(w, lo, hi);
                    a0 = fmaf(lo.x, bf16_lo(xp[2 * h]), a0);
                    a1 = fmaf(lo.y, bf16_hi(xp[2 * h]), a1);
                    a0 = fmaf(hi.x, bf16_lo(xp[2 * h + 1]), a0);
                    a1 = fmaf(hi.y, bf16_hi(xp[2 * h + 1]), a1);
                }
            }
        }
        acc = fmaf(fp16_to_float(it.d), a0 + a1, acc);
    }
};

// FP8 block-128: the chunk is 32 E4M3 bytes in element order (word w holds
// elements 4w .. 4w + 3, activation piece w / 2); lanes 4i .. 4i + 3 take
// the four chunks of one 128-element k tile and read its one fp32 scale, and
// 128 consecutive rows share a row of scales. E4M3 -> f16 is exact, and so
// is its product with an f16 activation in fp32.
struct DirFp8 {
    using Item = Q8Item;  // 32 code bytes, the fp32 scale's bits
    static constexpr int kCodeBytes = 32;
    static constexpr int kSChunk = 32;  // eight tile scales per 1024-element step
    __host__ __device__ static constexpr int64_t spitch(int64_t K) { return K / 32; }  // (K / 128) scales
    __device__ static __forceinline__ int64_t srow(int64_t pr) { return pr >> 7; }
    __device__ static __forceinline__ int slane(int lane) { return lane & ~3; }
    __device__ static __forceinline__ Item load(const uint8_t* c, const uint8_t* s)
    {
        Item it;
        it.a = ld_stream_v4(c);
        it.b = ld_stream_v4(c + 16);
        it.d = ld_stream_u32(s);
        return it;
    }
    template <bool FAST>
    __device__ static __forceinline__ void dot(const Item& it, const uint16_t* xc, int sw, float& acc)
    {
        const uint32_t words[8] = {it.a.x, it.a.y, it.a.z, it.a.w, it.b.x, it.b.y, it.b.z, it.b.w};
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int p = 0; p < 4; ++p) {  // 8 elements = 2 code words = activation piece p
            const uint4 xq = *reinterpret_cast<const uint4*>(xc + ((p ^ sw) << 3));
            const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t w = words[2 * p + h];
                const uint32_t q01 = e4m3x2_to_f16x2(w), q23 = e4m3x2_to_f16x2(w >> 16);
                if constexpr (FAST) {
                    fma_f16x2(q01, xp[2 * h], a0, a1);
                    fma_f16x2(q23, xp[2 * h + 1], a0, a1);
                } else {
                    const float2 lo = f16x2_to_float2(q01), hi = f16x2_to_float2(q23);
                    a0 = fmaf(lo.x, bf16_lo(xp[2 * h]), a0);
                    a1 = fmaf(lo.y, bf16_hi(xp[2 * h]), a1);
                    a0 = fmaf(hi.x, bf16_lo(xp[2 * h + 1]), a0);
                    a1 = fmaf(hi.y, bf16_hi(xp[2 * h + 1]), a1);
                }
            }
        }
        acc = fmaf(__uint_as_float(it.d), a0 + a1, acc);
    }
};

// Rows [r_lo, r_hi) of a warp. Item g of the stream (row g / CPL, chunk
// g % CPL) lives in buf[g % D]; D divides CPL or is a multiple of it, so
// with U = max(1, D / CPL) rows unrolled per body the slot, the chunk and
// the row offset of every item are compile-time constants.
// Epilogues of a row's dot product v (the row's output is ts * 2^sexp * v):
// kEpiPlain writes it; kEpiAdd adds the residual r[row] (y may be r);
// kEpiSiluMul takes the rows in pairs (virtual row 2i: gate row i, 2i + 1:
// up row half + i) and writes SiLU(g) * u to y[i].
constexpr int kEpiPlain = 0, kEpiAdd = 1, kEpiSiluMul = 2;

// Physical weight row of virtual row v.
template <int EPI>
__device__ __forceinline__ int64_t phys_row(int64_t v, int64_t half)
{
    if constexpr (EPI == kEpiSiluMul)
        return (v & 1) ? half + (v >> 1) : (v >> 1);
    else
        return v;
}

template <class F, int CPL, int D, bool FAST, int EPI>
__device__ __forceinline__ void direct_rows(typename F::Item (&buf)[D], const uint8_t* cp, const uint8_t* sp,
                                            int64_t cpitch, int64_t spitch, const uint16_t* xl, int sw, float* y,
                                            const float* r, int64_t half, int64_t r_lo, int64_t r_hi, float ts,
                                            int sexp, int lane)
{
    float gsave = 0.f;  // kEpiSiluMul: the gate row's output, until its up row is done
    static_assert(CPL % D == 0 || D % CPL == 0, "the ring depth must divide a row or be a multiple of one");
    constexpr int U = D > CPL ? D / CPL : 1;
    for (int64_t row0 = r_lo; row0 < r_hi; row0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (row0 + u < r_hi) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    const int g = u * CPL + i;
                    const typename F::Item cur = buf[g % D];
                    const int nr = (g + D) / CPL, nc = (g + D) % CPL;
                    if (row0 + nr < r_hi) {
                        const int64_t pr = phys_row<EPI>(row0 + nr, half);
                        buf[g % D] = F::load(cp + pr * cpitch + nc * 32 * F::kCodeBytes,
                                             sp + F::srow(pr) * spitch + nc * F::kSChunk);
                    }
                    F::template dot<FAST>(cur, xl + i * 1024, sw, acc);
                    // keep the next chunk's shared-memory loads after this chunk's arithmetic
                    asm volatile("" ::: "memory");
                }
                const float v = ldexpf(warp_sum(acc) * ts, sexp);
                const int64_t row = row0 + u;
                if constexpr (EPI == kEpiPlain) {
                    if (lane == 0) y[row] = v;
                } else if constexpr (EPI == kEpiAdd) {
                    if (lane == 0) y[row] = v + r[row];
                } else {
                    if (!(row & 1))
                        gsave = v;
                    else if (lane == 0)
                        y[row >> 1] = gsave / (1.0f + expf(-gsave)) * v;
                }
            }
        }
    }
}

// Dynamic shared memory: K f16 (or bf16) activations. M is the number of
// virtual rows (2 * half for kEpiSiluMul, whose warps take whole pairs).
template <class F, int CPL, int THREADS, int D, int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    gemv_direct_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, float ts,
                       const uint16_t* __restrict__ x, float* y, const float* r, int64_t M)
{
    const int64_t half = M / 2;
    constexpr int W = THREADS / kWarp;
    constexpr int64_t K = 1024 * CPL;
    constexpr int64_t cpitch = K / 32 * F::kCodeBytes, spitch = F::spitch(K);
    constexpr int NP = CPL * 128;                        // 16-byte activation pieces
    constexpr int PPT = (NP + THREADS - 1) / THREADS;    // pieces per thread
    extern __shared__ __align__(16) uint16_t xs[];
    __shared__ int s_emax, s_emin, s_flags;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    // this warp's rows: an even split of [0, M) over all warps of the grid
    const uint32_t gw = blockIdx.x * W + warp, nw = gridDim.x * W;
    int64_t r_lo, r_hi;
    const int64_t units = EPI == kEpiSiluMul ? half : M;  // rows, or row pairs
    if (units * nw < (int64_t(1) << 32)) {  // 32-bit division when it is exact
        const uint32_t m = static_cast<uint32_t>(units);
        r_lo = m * gw / nw;
        r_hi = m * (gw + 1) / nw;
    } else {
        r_lo = units * gw / nw;
        r_hi = units * (gw + 1) / nw;
    }
    if constexpr (EPI == kEpiSiluMul) {
        r_lo *= 2;
        r_hi *= 2;
    }
    const uint8_t* cp = codes + lane * F::kCodeBytes;
    const uint8_t* sp = scales + F::slane(lane);
    if (threadIdx.x == 0) {
        s_emax = 0;
        s_emin = INT_MAX;
        s_flags = 0;
    }
    // the first D chunks: weights only, before the wait for the previous kernel
    typename F::Item buf[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
        const int64_t row = r_lo + d / CPL;
        if (row < r_hi) {
            const int64_t pr = phys_row<EPI>(row, half);
            buf[d] = F::load(cp + pr * cpitch + (d % CPL) * 32 * F::kCodeBytes,
                             sp + F::srow(pr) * spitch + (d % CPL) * F::kSChunk);
        }
    }
    pdl_trigger();
    __syncthreads();
    pdl_wait();  // the activations may come from the previous kernel; y may be read by it

    // activations, one global read into registers: exponent range of the
    // nonzero values (bf16 biased exponents), then the prescaled f16 copy
    uint4 xv[PPT];
    int emax = 0, emin = INT_MAX, flags = 0;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int i = threadIdx.x + k * THREADS;
        if (i < NP) {
            xv[k] = reinterpret_cast<const uint4*>(x)[i];
            const uint32_t w[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t b = (w[q / 2] >> (16 * (q & 1))) & 0x7FFFu;
                const int e = static_cast<int>(b >> 7);
                if (b == 0) continue;
                if (e == 0 || e == 255) flags = 1;  // subnormal, inf or NaN
                emax = max(emax, e);
                emin = min(emin, e);
            }
        }
    }
    emax = __reduce_max_sync(0xFFFFFFFFu, emax);
    emin = __reduce_min_sync(0xFFFFFFFFu, emin);
    flags = __reduce_or_sync(0xFFFFFFFFu, flags);
    if (lane == 0) {
        if (flags) atomicOr(&s_flags, 1);
        atomicMax(&s_emax, emax);
        atomicMin(&s_emin, emin);
    }
    __syncthreads();
    // f16 holds x * 2^-sexp exactly when every nonzero |x| is within 31
    // binades of the largest; the largest lands in [2^14, 2^15).
    const bool fast = !s_flags && (s_emin == INT_MAX || s_emax - s_emin <= 31);
    const int sexp = fast && s_emin != INT_MAX ? s_emax - 127 - 14 : 0;
    // x * 2^-sexp as two exact multiplies by normal powers of two
    const int e1 = max(-126, min(127, -sexp));
    const float f1 = pow2f(e1), f2 = pow2f(max(-126, min(127, -sexp - e1)));
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int i = threadIdx.x + k * THREADS;
        if (i < NP) {
            uint4 u = xv[k];
            if (fast) {
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    __half2 hv = __floats2half2_rn(bf16_lo(w[q]) * f1 * f2, bf16_hi(w[q]) * f1 * f2);
                    o[q] = *reinterpret_cast<uint32_t*>(&hv);
                }
                u = make_uint4(o[0], o[1], o[2], o[3]);
            }
            *reinterpret_cast<uint4*>(xs + x_index(i / 4, i % 4)) = u;
        }
    }
    __syncthreads();
    const uint16_t* xl = xs + lane * 32;
    const int sw = (lane >> 1) & 3;
    if (fast)
        direct_rows<F, CPL, D, true, EPI>(buf, cp, sp, cpitch, spitch, xl, sw, y, r, half, r_lo, r_hi, ts, sexp,
                                          lane);
    else
        direct_rows<F, CPL, D, false, EPI>(buf, cp, sp, cpitch, spitch, xl, sw, y, r, half, r_lo, r_hi, ts, sexp,
                                           lane);
}

// Launch shape per format, from back-to-back timings of 12288 x 4096 and
// 4096 x 12288 calls over rotating weights (GB300): one CTA per SM; NVFP4
// with K = 4096 768 threads and four chunks in flight per lane (0.61 of the
// measured copy peak on 12288 x 4096; 1024 threads with two: 0.56; 512 with
// eight: 0.55), with K = 12288 512 threads and six (0.56 on 4096 x 12288;
// 896 threads with two: 0.52; 512 with twelve: 0.53), else 896 threads and
// two chunks; Q8_0 (twice the bytes per element) 896 threads and two chunks
// (0.81 on 12288 x 4096, 0.76 on 4096 x 12288). D must divide CPL or be a
// multiple of it.
template <class F>
struct DirCfg;
template <>
struct DirCfg<DirNvfp4> {
    template <int CPL>
    static constexpr int threads() { return CPL == 4 ? 768 : (CPL == 12 ? 512 : 896); }
    template <int CPL>
    static constexpr int depth() { return CPL == 4 ? 4 : (CPL == 12 ? 6 : (CPL == 3 ? 3 : 2)); }
};
template <>
struct DirCfg<DirQ4> : DirCfg<DirNvfp4> {};
template <>
struct DirCfg<DirQ8> {
    template <int CPL>
    static constexpr int threads() { return 896; }
    template <int CPL>
    static constexpr int depth() { return CPL == 3 ? 3 : 2; }
};
template <>
struct DirCfg<DirFp8> : DirCfg<DirQ8> {};  // the same bytes per element

template <class F, int CPL, int EPI>
cudaError_t launch_cpl(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x, float* y,
                       const float* r, int64_t M, cudaStream_t stream)
{
    constexpr int T = DirCfg<F>::template threads<CPL>();
    constexpr int D = DirCfg<F>::template depth<CPL>();
    auto kern = gemv_direct_kernel<F, CPL, T, D, EPI>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(CPL) * 1024 * 2;
    static OccCache occ;
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, T, smem);  // sets the shared-memory opt-in
    int64_t grid = dev_info(dev).sms;
    const int64_t need = (M + T / kWarp - 1) / (T / kWarp);
    if (grid > need) grid = need;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(T);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_flags() & kLaunchPdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, codes, scales, ts, x, y, r, M);
}

template <class F, int EPI>
cudaError_t launch_direct(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x, float* y,
                          const float* r, int64_t M, int64_t K, cudaStream_t s)
{
    switch (K / 1024) {
        case 1: return launch_cpl<F, 1, EPI>(codes, scales, ts, x, y, r, M, s);
        case 2: return launch_cpl<F, 2, EPI>(codes, scales, ts, x, y, r, M, s);
        case 3: return launch_cpl<F, 3, EPI>(codes, scales, ts, x, y, r, M, s);
        case 4: return launch_cpl<F, 4, EPI>(codes, scales, ts, x, y, r, M, s);
        case 6: return launch_cpl<F, 6, EPI>(codes, scales, ts, x, y, r, M, s);
        case 8: return launch_cpl<F, 8, EPI>(codes, scales, ts, x, y, r, M, s);
        case 12: return launch_cpl<F, 12, EPI>(codes, scales, ts, x, y, r, M, s);
        case 16: return launch_cpl<F, 16, EPI>(codes, scales, ts, x, y, r, M, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool direct_gemv_supported(int64_t M, int64_t K, int N)
{
    if (N != 1 || M < 1 || K < 1024 || K % 1024 != 0 || M > (int64_t(1) << 40)) return false;
    switch (K / 1024) {
        case 1: case 2: case 3: case 4: case 6: case 8: case 12: case 16: return true;
        default: return false;
    }
}

cudaError_t launch_nvfp4_gemv_direct(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                     float* y, int64_t M, int64_t K, cudaStream_t s)
{
    return launch_direct<DirNvfp4, kEpiPlain>(codes, scales, ts, x, y, nullptr, M, K, s);
}

cudaError_t launch_q4_0_gemv_direct(const uint8_t* codes, const uint16_t* d, const uint16_t* x, float* y,
                                    int64_t M, int64_t K, cudaStream_t s)
{
    return launch_direct<DirQ4, kEpiPlain>(codes, reinterpret_cast<const uint8_t*>(d), 1.0f, x, y, nullptr, M, K, s);
}

cudaError_t launch_fp8_b128_gemv_direct(const uint8_t* codes, const float* scales, const uint16_t* x, float* y,
                                        int64_t M, int64_t K, cudaStream_t s)
{
    return launch_direct<DirFp8, kEpiPlain>(codes, reinterpret_cast<const uint8_t*>(scales), 1.0f, x, y, nullptr, M,
                                            K, s);
}

cudaError_t launch_q8_0_gemv_direct(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M,
                                    int64_t K, cudaStream_t s)
{
    return launch_direct<DirQ8, kEpiPlain>(reinterpret_cast<const uint8_t*>(q), reinterpret_cast<const uint8_t*>(d),
                                           1.0f, x, y, nullptr, M, K, s);
}

cudaError_t launch_nvfp4_gemv_direct_add(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                         const float* r, float* y, int64_t M, int64_t K, cudaStream_t s)
{
    return launch_direct<DirNvfp4, kEpiAdd>(codes, scales, ts, x, y, r, M, K, s);
}

cudaError_t launch_q8_0_gemv_direct_add(const int8_t* q, const uint16_t* d, const uint16_t* x, const float* r,
                                        float* y, int64_t M, int64_t K, cudaStream_t s)
{
    return launch_direct<DirQ8, kEpiAdd>(reinterpret_cast<const uint8_t*>(q), reinterpret_cast<const uint8_t*>(d),
                                         1.0f, x, y, r, M, K, s);
}

cudaError_t launch_nvfp4_gemv_direct_silu_mul(const uint8_t* codes, const uint8_t* scales, float ts,
                                              const uint16_t* x, float* h, int64_t I, int64_t K, cudaStream_t s)
{
    return launch_direct<DirNvfp4, kEpiSiluMul>(codes, scales, ts, x, h, nullptr, 2 * I, K, s);
}

cudaError_t launch_q8_0_gemv_direct_silu_mul(const int8_t* q, const uint16_t* d, const uint16_t* x, float* h,
                                             int64_t I, int64_t K, cudaStream_t s)
{
    return launch_direct<DirQ8, kEpiSiluMul>(reinterpret_cast<const uint8_t*>(q), reinterpret_cast<const uint8_t*>(d),
                                             1.0f, x, h, nullptr, 2 * I, K, s);
}

}  // namespace bqd
