// gemv_tiles.cu -- NVFP4 GEMV for a few tokens (2 <= N <= 16) on the tensor
// cores in warp tiles, streaming the weights straight from HBM into
// registers.
//
// Y[n][m] = ts * sum_b scale[m][b] * sum_{k in b} e2m1[m][k] * X[n][k]: the
// multi-token form of the NVFP4 matvec that checks K+1 drafted tokens in one
// batched target forward ("robertbfuentes7-cloud/bw24" README, NVFP4 (W4)
// decode path and speculative decoding bullets).
//
// The tokens share every weight, so the work is a thin dense contraction;
// it is also bound by the weight stream, so the design is the N = 1 direct
// GEMV's (coalesced 16-byte loads into a compile-time register ring, the
// first chunks requested before the dependency wait) with the per-row dot
// products replaced by mma.sync m16n8k16 (f16 or bf16 operands, fp32
// accumulation):
//  * A warp tile is 8 weight rows x 16 token slots. The activations are the
//    A operand (token g and g + 8 as rows g and g + 8 of the 16 x 16
//    fragment; unused slots hold zeros) and the weights the B operand
//    (weight row g as column g). Lane (g, i) = (lane / 4, lane % 4) loads 16
//    code bytes (32 elements, k = 32 i .. 32 i + 31 of each 128-element
//    chunk) and the two block scales of weight row g, and the same k of
//    token g (and g + 8) from shared memory. The k order inside an mma is
//    free as long as A and B agree: step j of a chunk takes, for quad i,
//    elements 32 i + 4 j .. + 3 (logical k 2i, 2i+1, 2i+8, 2i+9).
//  * The activations (N K <= 32768) pass through registers once per CTA:
//    loaded, their per-token exponent range reduced, converted and stored
//    in a bank-conflict-free layout read with immediate offsets.
//  * Weights enter as w * s (E2M1 code times its E4M3 block scale), exact
//    in f16 and in bf16 (at most 6 significant bits, magnitudes in
//    [2^-10, 2688]). The activations are staged as f16 after an exact
//    power-of-two prescale per token (f16 holds every bf16 value exactly
//    when the token's nonzero magnitudes lie within 31 binades of its
//    largest); otherwise the CTA keeps the bf16 values and both operands
//    are bf16. Every product is exact; sums are fp32.
//  * Work split: each CTA owns a contiguous range of 8-row tiles; its 16
//    warps split the range's (tile, chunk) units evenly, so a tile may be
//    shared by consecutive warps. A warp that covers a whole tile writes Y
//    directly; partial sums of shared tiles meet in shared memory and are
//    added in warp order, so results are deterministic.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "common.cuh"
#include "gemv.h"
#include "host_util.h"

namespace bqd {

namespace {

constexpr int kThT = 512;  // 16 warps, one CTA per SM
constexpr int kWpT = kThT / kWarp;
constexpr int kDepthT = 8;        // 128-element chunks in flight per lane
constexpr int kRowsT = 8;         // weight rows per tile
constexpr int kMaxNT = 16;        // token slots of a tile
constexpr int kXP = 8;            // 16-byte activation pieces per thread (N * K <= 8 * 8 * kThT)

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 2^e for a normal exponent e (-126 .. 127).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// An f16 pair whose values are bf16 values, as a bf16 pair (exact).
__device__ __forceinline__ uint32_t f16x2_as_bf16x2(uint32_t h)
{
    const float2 f = f16x2_to_float2(h);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));
    return r;
}

// Staged activations: token n's row at byte n * xpitch (xpitch = 2K + 64);
// element k of it at byte 256 (k >> 7) + 64 ((k >> 3) & 3) + 16 ((k >> 5)
// & 3) + 2 (k & 7): the four quads' pieces of one chunk and word sit side
// by side, and the 64-byte pad shifts consecutive tokens by half a bank
// row, so the eight lanes of a shared-memory wavefront (two tokens x four
// quads) read 128 distinct bytes.
__device__ __forceinline__ int x_off(int k) { return ((k >> 7) << 8) + (((k >> 3) & 3) << 6) + (((k >> 5) & 3) << 4); }

struct Slot {
    uint4 c;     // 16 code bytes
    uint32_t s;  // two E4M3 block scales
};

// One 128-element chunk of a tile: xa, xb point at token slots g and g + 8
// of the chunk, quad i (the four word pieces 64 bytes apart). Steps
// alternate between two accumulators (two dependency chains).
template <bool FAST, bool HI>
__device__ __forceinline__ void tile_chunk(const Slot& cur, const char* xa, const char* xb, float (&acc0)[4],
                                           float (&acc1)[4])
{
    const uint32_t s2 = e4m3x2_to_f16x2(cur.s & 0xFFFFu);
    const uint32_t sl = __byte_perm(s2, 0, 0x1010), sh = __byte_perm(s2, 0, 0x3232);
    const uint32_t cw[4] = {cur.c.x, cur.c.y, cur.c.z, cur.c.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t wp[4];
        e2m1x8_to_f16x2(cw[w], wp);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            wp[q] = hmul2_bits(wp[q], w < 2 ? sl : sh);
            if constexpr (!FAST) wp[q] = f16x2_as_bf16x2(wp[q]);
        }
        const uint4 a = *reinterpret_cast<const uint4*>(xa + 64 * w);
        // without tokens 8..15 the upper fragment rows repeat the lower ones
        // (their outputs are dropped)
        const uint4 b = HI ? *reinterpret_cast<const uint4*>(xb + 64 * w) : a;
        if constexpr (FAST) {
            mma_f16(acc0, a.x, b.x, a.y, b.y, wp[0], wp[1]);
            mma_f16(acc1, a.z, b.z, a.w, b.w, wp[2], wp[3]);
        } else {
            mma_bf16(acc0, a.x, b.x, a.y, b.y, wp[0], wp[1]);
            mma_bf16(acc1, a.z, b.z, a.w, b.w, wp[2], wp[3]);
        }
    }
}

// The end of a segment (the units of one tile within a warp's range): the
// whole tile goes to Y, c = (token g | g + 8, row 2i | 2i + 1); a part of
// one to the warp's partial slot. Out of line, so that the chunk loop
// carries none of it.
__device__ __noinline__ void segment_out(float v0, float v1, float v2, float v3, bool whole, float* slot,
                                         float* __restrict__ y, const int* sexp, float ts, int64_t M, int N,
                                         int64_t row0, int lane)
{
    const int g = lane >> 2, i = lane & 3;
    const float v[4] = {v0, v1, v2, v3};
    if (whole) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int n = g + (c >> 1) * 8;
            const int64_t m = row0 + 2 * i + (c & 1);
            if (n < N && m < M) y[static_cast<int64_t>(n) * M + m] = ldexpf(v[c] * ts, sexp[n]);
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) slot[lane * 4 + c] = v[c];
    }
}

// The warp's (tile, chunk) units [u_lo, u_hi) of the CTA's tiles starting at
// tile t0; the ring holds units u_lo .. u_lo + kDepthT - 1 on entry. A
// segment that is the whole tile goes to Y; a first or last segment that is
// not goes to the warp's partial slots 0 or 1 (part, 128 floats each).
template <bool FAST, bool HI>
__device__ __forceinline__ void tile_units(Slot (&ring)[kDepthT], const uint8_t* __restrict__ codes,
                                           const uint8_t* __restrict__ scales, const char* xsb, int xpitch,
                                           const int* sexp, float ts, float* __restrict__ y, float* part, int64_t M,
                                           int K, int N, int64_t t0, int u_lo, int u_hi, int lane)
{
    const int KCH = K / 128;
    const int g = lane >> 2, i = lane & 3;
    const int64_t cpitch = K / 2, spitch = K / 16;
    // load cursor at the unit after the ring's last: its chunk and the row pointers
    const int ul = u_lo + kDepthT;
    int lkc = ul % KCH;
    const int64_t lrow = (t0 + ul / KCH) * kRowsT + g;
    const uint8_t* lc = codes + lrow * cpitch + i * 16 + lkc * 64;
    const uint8_t* ls = scales + lrow * spitch + i * 2 + lkc * 8;
    int64_t lrem = M - lrow;  // rows left below the load cursor's row, for the bounds check
    const int64_t cwrap = kRowsT * cpitch - static_cast<int64_t>(KCH) * 64;
    const int64_t swrap = kRowsT * spitch - static_cast<int64_t>(KCH) * 8;
    // token slots g, g + 8 (a slot past N reads token 0: its outputs are dropped)
    const char* xa = xsb + (g < N ? g : 0) * xpitch + i * 16;
    const char* xb = xsb + (g + 8 < N ? g + 8 : 0) * xpitch + i * 16;
    int ct = u_lo / KCH, ckc = u_lo % KCH, seg0 = ckc;  // compute cursor; seg0: first chunk of the segment
    bool first_seg = true;
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    for (int u0 = u_lo; u0 < u_hi; u0 += kDepthT) {
#pragma unroll
        for (int d = 0; d < kDepthT; ++d) {
            const int u = u0 + d;
            if (u < u_hi) {
                const Slot cur = ring[d];
                if (u + kDepthT < u_hi) {
                    Slot sl;
                    sl.c = make_uint4(0u, 0u, 0u, 0u);
                    sl.s = 0u;
                    if (lrem > 0) {
                        sl.c = ld_stream_v4(lc);
                        sl.s = ld_stream_u16(ls);
                    }
                    ring[d] = sl;
                    lc += 64;
                    ls += 8;
                    if (++lkc == KCH) {
                        lkc = 0;
                        lc += cwrap;
                        ls += swrap;
                        lrem -= kRowsT;
                    }
                }
                tile_chunk<FAST, HI>(cur, xa + ckc * 256, xb + ckc * 256, acc0, acc1);
                if (++ckc == KCH || u + 1 == u_hi) {  // the segment ends
                    segment_out(acc0[0] + acc1[0], acc0[1] + acc1[1], acc0[2] + acc1[2], acc0[3] + acc1[3],
                                seg0 == 0 && ckc == KCH, part + (first_seg ? 0 : 128), y, sexp, ts, M, N,
                                (t0 + ct) * kRowsT, lane);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        acc0[c] = 0.f;
                        acc1[c] = 0.f;
                    }
                    first_seg = false;
                    if (ckc == KCH) {
                        ckc = 0;
                        ++ct;
                    }
                    seg0 = ckc;
                }
                asm volatile("" ::: "memory");
            }
        }
    }
}

// Dynamic shared memory: the activations, N rows of 2K + 64 bytes.
__global__ void __launch_bounds__(kThT, 1)
    gemv_tiles_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, float ts,
                      const uint16_t* __restrict__ x, float* __restrict__ y, int64_t M, int K, int N)
{
    extern __shared__ __align__(16) char xsb[];
    __shared__ float s_part[kWpT][2][128];
    __shared__ int s_emax[kMaxNT], s_emin[kMaxNT], s_sexp[kMaxNT], s_flags;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int KCH = K / 128, xpitch = 2 * K + 64;
    const int64_t ntile = (M + kRowsT - 1) / kRowsT;
    const int64_t t0 = ntile * blockIdx.x / gridDim.x, t1 = ntile * (blockIdx.x + 1) / gridDim.x;
    const int U = static_cast<int>(t1 - t0) * KCH;  // (tile, chunk) units of the CTA
    const int u_lo = static_cast<int>(static_cast<int64_t>(U) * warp / kWpT);
    const int u_hi = static_cast<int>(static_cast<int64_t>(U) * (warp + 1) / kWpT);
    const int g = lane >> 2, i = lane & 3;

    if (threadIdx.x == 0) s_flags = 0;
    if (threadIdx.x < kMaxNT) {
        s_emax[threadIdx.x] = 0;
        s_emin[threadIdx.x] = INT_MAX;
    }
    // the first kDepthT units' weights, before the dependency wait
    Slot ring[kDepthT];
    {
        int kc = u_lo % KCH;
        int64_t row = (t0 + u_lo / KCH) * kRowsT + g;
#pragma unroll
        for (int d = 0; d < kDepthT; ++d) {
            ring[d].c = make_uint4(0u, 0u, 0u, 0u);
            ring[d].s = 0u;
            if (u_lo + d < u_hi && row < M) {
                ring[d].c = ld_stream_v4(codes + row * (K / 2) + kc * 64 + i * 16);
                ring[d].s = ld_stream_u16(scales + row * (K / 16) + kc * 8 + i * 2);
            }
            if (++kc == KCH) {
                kc = 0;
                row += kRowsT;
            }
        }
    }
    pdl_trigger();
    pdl_wait();  // x may come from the previous kernel; y may be read by it

    // Activations, one pass through registers: each thread loads its 16-byte
    // pieces (consecutive per warp, so a warp's 32 pieces lie in one token),
    // the per-token exponent range is reduced, then the pieces are converted
    // and stored. |x| bit patterns (sign cleared) order like the values: the
    // largest and the smallest nonzero pattern per token give its range (and
    // show an infinity or NaN, 0x7F80 and up, or a subnormal, below 0x0080).
    const int npc = N * K / 8;
    uint4 xv[kXP];
#pragma unroll
    for (int r = 0; r < kXP; ++r) {
        const int pc = threadIdx.x + r * kThT;
        if (pc < npc) xv[r] = reinterpret_cast<const uint4*>(x)[pc];
    }
#pragma unroll
    for (int r = 0; r < kXP; ++r) {
        if (r * kThT + warp * kWarp < npc) {  // warp-uniform
            const uint32_t w4[4] = {xv[r].x, xv[r].y, xv[r].z, xv[r].w};
            uint32_t hmax = 0u, hmin = 0xFFFFFFFFu;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint32_t m = w4[h] & 0x7FFF7FFFu;
                hmax = __vmaxu2(hmax, m);
                hmin = __vminu2(hmin, __vsub2(m, 0x00010001u));  // a zero half wraps to 0xFFFF
            }
            const uint32_t bmax = __reduce_max_sync(0xFFFFFFFFu, max(hmax & 0xFFFFu, hmax >> 16));
            const uint32_t bmin = __reduce_min_sync(0xFFFFFFFFu, min(hmin & 0xFFFFu, hmin >> 16)) + 1u;
            if (lane == 0) {
                const int n = (r * kThT + warp * kWarp) / (K / 8);
                atomicMax(&s_emax[n], static_cast<int>(bmax));
                atomicMin(&s_emin[n], static_cast<int>(bmin));  // 0x10000: no nonzero element
            }
        }
    }
    __syncthreads();
    if (threadIdx.x < N) {  // patterns to exponents (a token of zeros keeps emin = INT_MAX)
        const int bmax = s_emax[threadIdx.x], bmin = s_emin[threadIdx.x];
        const bool any = bmin < 0x10000;
        if (bmax >= 0x7F80 || (any && bmin < 0x0080) || (any && (bmax >> 7) - (bmin >> 7) > 31))
            atomicOr(&s_flags, 1);
        s_emax[threadIdx.x] = bmax >> 7;
        s_emin[threadIdx.x] = any ? bmin >> 7 : INT_MAX;
    }
    __syncthreads();
    const bool fast = s_flags == 0;
    if (threadIdx.x < kMaxNT)
        s_sexp[threadIdx.x] =
            fast && threadIdx.x < N && s_emin[threadIdx.x] != INT_MAX ? s_emax[threadIdx.x] - 127 - 14 : 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kXP; ++r) {
        const int pc = threadIdx.x + r * kThT;
        if (pc < npc) {
            const int n = pc / (K / 8), k = (pc - n * (K / 8)) * 8;
            uint4 q = xv[r];
            if (fast) {  // x * 2^-s as two exact multiplies by normal powers of two, to f16
                const int se = s_sexp[n], e1 = max(-126, min(127, -se));
                const float f1 = pow2f(e1), f2 = pow2f(max(-126, min(127, -se - e1)));
                const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
                uint32_t o[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    __half2 hv = __floats2half2_rn(bf16_lo(w4[h]) * f1 * f2, bf16_hi(w4[h]) * f1 * f2);
                    o[h] = *reinterpret_cast<uint32_t*>(&hv);
                }
                q = make_uint4(o[0], o[1], o[2], o[3]);
            }
            *reinterpret_cast<uint4*>(xsb + n * xpitch + x_off(k)) = q;
        }
    }
    __syncthreads();

    float* part = &s_part[warp][0][0];
    const bool hi = N > 8;
    if (fast) {
        if (hi)
            tile_units<true, true>(ring, codes, scales, xsb, xpitch, s_sexp, ts, y, part, M, K, N, t0, u_lo, u_hi, lane);
        else
            tile_units<true, false>(ring, codes, scales, xsb, xpitch, s_sexp, ts, y, part, M, K, N, t0, u_lo, u_hi,
                                    lane);
    } else {
        if (hi)
            tile_units<false, true>(ring, codes, scales, xsb, xpitch, s_sexp, ts, y, part, M, K, N, t0, u_lo, u_hi,
                                    lane);
        else
            tile_units<false, false>(ring, codes, scales, xsb, xpitch, s_sexp, ts, y, part, M, K, N, t0, u_lo, u_hi,
                                     lane);
    }
    __syncthreads();

    // tiles shared by several warps: warp w - 1 takes the tile that warp
    // boundary w falls strictly inside, unless an earlier boundary already
    // fell inside it, and adds the covering warps' segments in warp order
    if (warp < kWpT - 1) {
        const int b = static_cast<int>(static_cast<int64_t>(U) * (warp + 1) / kWpT);
        const int bp = static_cast<int>(static_cast<int64_t>(U) * warp / kWpT);
        const int tl = b / KCH;
        if (b % KCH != 0 && bp <= tl * KCH) {
            const int ua = tl * KCH, ub = ua + KCH;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            for (int w = 0; w < kWpT; ++w) {
                const int lo = static_cast<int>(static_cast<int64_t>(U) * w / kWpT);
                const int hi2 = static_cast<int>(static_cast<int64_t>(U) * (w + 1) / kWpT);
                if (max(lo, ua) < min(hi2, ub)) {  // warp w has units of this tile
                    const float* slot = &s_part[w][lo >= ua ? 0 : 1][lane * 4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] += slot[c];
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int n = g + (c >> 1) * 8;
                const int64_t m = (t0 + tl) * kRowsT + 2 * i + (c & 1);
                if (n < N && m < M) y[static_cast<int64_t>(n) * M + m] = ldexpf(v[c] * ts, s_sexp[n]);
            }
        }
    }
}

}  // namespace

bool tiles_gemv_supported(int64_t M, int64_t K, int N)
{
    return N >= 2 && N <= kMaxNT && M >= 1 && M <= (int64_t(1) << 34) && K >= 1024 && K % 1024 == 0 &&
           static_cast<int64_t>(N) * K <= int64_t{8} * kXP * kThT &&
           (M + kRowsT - 1) / kRowsT * (K / 128) < (int64_t(1) << 31);
}

cudaError_t launch_nvfp4_gemv_tiles(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                    float* y, int64_t M, int64_t K, int N, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(N) * (2 * K + 64);
    static OccCache occ;
    blocks_per_sm(occ, reinterpret_cast<const void*>(gemv_tiles_kernel), dev, kThT, smem);  // sets the opt-in
    int64_t grid = dev_info(dev).sms;
    const int64_t ntile = (M + kRowsT - 1) / kRowsT;
    if (grid > ntile) grid = ntile;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_flags() & kLaunchPdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_tiles_kernel, codes, scales, ts, x, y, M, static_cast<int>(K), N);
}

}  // namespace bqd
