// gemm_prefill.cu -- NVFP4 weights times many bf16 tokens (prefill) on the
// 5th-generation tensor cores: Y[t][m] = ts * sum_k W[m][k] * x[t][k].
//
// The pages' prefill runs its NVFP4 weights through GEMMs over many tokens
// ("Vemloir/LumenLLM" README, Kernels bullet: NVFP4 grouped-MoE prefill, a
// per-expert variable-grid NVFP4 GEMM). This is that GEMM for one weight
// matrix; a grouped MoE prefill runs it per expert on the expert's gathered
// tokens.
//
// A CTA computes a 256 x 256 tile of Y (256 weight rows, 256 tokens) as two
// halves of 128 rows with tcgen05.mma kind::f16 (M = 128, N = 256, K = 16,
// bf16 operands, fp32 accumulators: all 512 columns of tensor memory), both
// operands in shared memory, K-major; the two halves share every tile of B,
// which halves B's traffic per flop against a 128-row tile. Each ring stage
// holds 64 k:
//  - B, 256 tokens x 64 k of x (128 bytes a token), comes in by one 2-D
//    tensor copy with the 128-byte swizzle (tokens past T read as zero) and
//    is read through a matching descriptor (8-row atoms of 1024 bytes, the
//    16 k of an MMA at 32 bytes into the atom). Narrower, unswizzled boxes of
//    16 bytes a row moved twice the bytes through the memory system;
//  - A, 2 x 128 rows x 64 k of W, is written by eight decoder warps, one row
//    per thread, K-major without swizzle (core matrices of 8 rows x 16 bytes;
//    128 bytes between row groups, 2 KiB between 8-k groups): E2M1 codes to
//    f16, times the block's E4M3 scale (exact: the product has at most 6
//    significant bits and lies in [2^-10, 2688]), to bf16 (exact for the
//    same reason), so every product of the MMA is exact and only the fp32
//    accumulation rounds.
// Warp 0 issues the copies, warp 1 the MMAs (one elected lane), warps 2..9
// decode and, at the end, read the accumulators (warp w owns tensor-memory
// lanes 32 (w % 4) .. + 31 of half (w - 2) / 4, its rows) and store ts * D.
// Every wait is bounded; a wait that runs out sets the kernel's device error
// word and the outputs are unspecified.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "host_util.h"
#include "stream.cuh"

namespace bqd {

// Device error word of the prefill GEMM (kErrWaitTimeout); read and cleared
// by read_and_clear_gemm_error().
__device__ unsigned int g_gemm_error = 0;

namespace {

constexpr int kGH = 128;                    // rows per half (MMA M)
constexpr int kGM = 2 * kGH;                // weight rows per tile
constexpr int kGK = 64;                     // k per ring stage
constexpr int kGSMax = 3;                   // ring stages (a fourth at BN = 128 measured no faster)
constexpr int kGDec = kGM / kWarp;          // decoder warps, one row per thread
constexpr int kGThreads = (2 + kGDec) * kWarp;
constexpr int kALoads = 8;                  // stages of a row's codes in flight per decoder thread
constexpr int kAHalf = kGH * kGK * 2;       // 16 KiB of bf16
constexpr int kAStage = 2 * kAHalf;
// BN tokens per tile (the MMA's N): 256 for one weight matrix; 32, 64 or 128
// for the experts' token segments of a grouped call, by the mean tokens per
// expert (an expert of a top-8 layer over 256 experts sees ~32 of 1024
// tokens). B is BN x 64 k of bf16, and the two halves' fp32 accumulators
// take 2 BN columns of tensor memory (a power of two, at least 32).
// The ring has as many stages as fit in shared memory, at most kGSMax.
template <int BN>
struct GemmShape {
    static constexpr int kBStage = BN * kGK * 2;
    static constexpr int kStages = (226 * 1024) / (kAStage + kBStage) < kGSMax ? (226 * 1024) / (kAStage + kBStage)
                                                                              : kGSMax;
    static constexpr int kSmem = kStages * (kAStage + kBStage) + 1024;  // + alignment slack
    static constexpr int kTmemCols = 2 * BN;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "an M = 128 MMA takes N = 16 .. 256 in steps of 16");
    static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                  "tensor memory is allocated in powers of two from 32 to 512 columns");
    static_assert(kStages >= 2, "the ring needs two stages to overlap loads with MMAs");
    static_assert(kSmem <= 227 * 1024, "dynamic shared memory of one CTA");
    static_assert(kBStage % 1024 == 0, "B stages start on 1024-byte boundaries (128-byte swizzle atoms)");
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor, K-major, no swizzle: start address, the
// byte distance between core matrices adjacent in k (lbo) and adjacent in
// rows (sbo), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}

// The same for K-major operands with the 128-byte swizzle, as a 2-D tensor
// copy with CU_TENSOR_MAP_SWIZZLE_128B leaves them: 8-row atoms of 1024
// bytes (sbo), the leading offset unused (1), layout type 2.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

// D[tmem_d] (+)= A[adesc] * B[bdesc]^T, both operands in shared memory.
__device__ __forceinline__ void mma_ss(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ bool elect_one()
{
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h)
{
    const float2 f = f16x2_to_float2(h);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);  // exact: E2M1 x E4M3 products fit in bf16
    return *reinterpret_cast<uint32_t*>(&b);
}

// 64 consecutive k of one row (32 code bytes c0, c1; the 4 block scales in
// s4) to 32 bf16 pairs, pair j = elements 2j (low half) and 2j + 1.
__device__ __forceinline__ void decode64(const uint4& c0, const uint4& c1, uint32_t s4, uint32_t (&a)[32])
{
    const uint32_t s01 = e4m3x2_to_f16x2(s4 & 0xFFFFu), s23 = e4m3x2_to_f16x2(s4 >> 16);
    const uint32_t sb[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232), __byte_perm(s23, 0, 0x1010),
                            __byte_perm(s23, 0, 0x3232)};
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // word i = k 8i .. 8i + 7, block i / 2
        uint32_t h[4];
        e2m1x8_to_f16x2(w[i], h);
#pragma unroll
        for (int j = 0; j < 4; ++j) a[4 * i + j] = f16x2_to_bf16x2(hmul2_bits(h[j], sb[i >> 1]));
    }
}

struct RowLoad {  // 64 k of one weight row
    uint4 c0, c1;
    uint32_t s4;
};

// Grouped form (offsets != nullptr): E experts, weights [E][M][KW], tokens
// [P][K] gathered expert-major, expert e's tokens [offsets[e],
// offsets[e + 1]), its tensor scale ts_e[e]; grid row blockIdx.y is the
// slot-th BN-token tile of all experts' tiles in expert order (slots past
// the last tile do nothing). Dense form: E = 1, tokens [0, T), scale ts.
// K is a multiple of KW: token k meets weight k % KW (KW = K but for the
// MoE down projection, whose tokens hold two parts of h side by side).
template <int BN>
__global__ void __launch_bounds__(kGThreads, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap map_x, const uint8_t* __restrict__ codes,
                      const uint8_t* __restrict__ scales, float ts, const float* __restrict__ ts_e,
                      const int32_t* __restrict__ offsets, int E, float* __restrict__ y, int64_t M, int K, int T,
                      int accumulate, int KW)
{
    using S = GemmShape<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    constexpr int kGS = S::kStages;
    __shared__ __align__(8) uint64_t bfull[kGSMax], afull[kGSMax], empty[kGSMax], dfull;
    __shared__ uint32_t s_tmem;
    __shared__ int s_e, s_n0, s_nend;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* astage = sm;
    uint8_t* bstage = sm + kGS * kAStage;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kGM;
    const int nk = K / kGK;     // stages of B's k
    const int nkw = KW / kGK;   // stages of the weights' k: B's k runs over them K / KW times

    // this CTA's expert and token range [n0, nend); an empty range: nothing to
    // do. Grouped: the experts' tile counts are scanned a block of experts at
    // a time (one per thread), and the thread whose expert holds the slot
    // records it.
    __shared__ int s_wsum[kGThreads / kWarp], s_base;
    if (threadIdx.x == 0) {
        s_e = 0;
        s_n0 = static_cast<int>(blockIdx.y) * BN;
        s_nend = offsets ? s_n0 : min(s_n0 + BN, T);
        s_base = 0;
    }
    __syncthreads();
    if (offsets) {
        const int slot = static_cast<int>(blockIdx.y);
        for (int c0 = 0; c0 < E; c0 += kGThreads) {
            const int x = c0 + threadIdx.x;
            int a = 0, b = 0;
            if (x < E) {
                a = max(0, min(offsets[x], T));  // clamped to [0, P]
                b = max(a, min(offsets[x + 1], T));
            }
            const int tiles = (b - a + BN - 1) / BN;
            int incl = tiles;  // inclusive scan of the tile counts over the block
#pragma unroll
            for (int d = 1; d < kWarp; d <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if ((threadIdx.x & 31) >= d) incl += v;
            }
            if ((threadIdx.x & 31) == 31) s_wsum[threadIdx.x / kWarp] = incl;
            __syncthreads();
            int before = s_base;
            for (int w = 0; w < static_cast<int>(threadIdx.x / kWarp); ++w) before += s_wsum[w];
            const int first = before + incl - tiles;  // this expert's first slot
            if (x < E && slot >= first && slot < first + tiles) {
                s_e = x;
                s_n0 = a + (slot - first) * BN;
                s_nend = min(s_n0 + BN, b);
            }
            __syncthreads();
            if (threadIdx.x == kGThreads - 1) s_base = before + incl;
            __syncthreads();
        }
    }
    if (s_nend <= s_n0) return;  // uniform: before any barrier, copy or tensor-memory allocation
    const int e_cta = s_e, n0 = s_n0, nend = s_nend;
    if (offsets) {
        codes += static_cast<int64_t>(e_cta) * M * (KW / 2);
        scales += static_cast<int64_t>(e_cta) * M * (KW / 16);
        ts = ts_e[e_cta];
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGS; ++s) {
            mbar_init(&bfull[s], 1);
            mbar_init(&afull[s], kGDec);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&dfull, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(S::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    pdl_trigger();
    pdl_wait();  // x may come from the previous kernel in the stream; y may be read by it

    bool ok = true;
    if (warp == 0) {
        // ------------------------------------------------ B: x tiles
        if (lane == 0) {
            for (int s = 0; s < nk && ok; ++s) {
                const int st = s % kGS;
                if (s >= kGS) ok = mbar_wait(&empty[st], static_cast<uint32_t>(((s / kGS) & 1) ^ 1), &g_gemm_error);
                if (!ok) break;
                mbar_arrive_expect_tx(&bfull[st], S::kBStage);
                tma_load_2d(bstage + st * S::kBStage, &map_x, s * kGK, n0, &bfull[st]);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue
        const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                               (static_cast<uint32_t>(kGH >> 4) << 24);  // f32 D, bf16 A and B, N, M
        for (int s = 0; s < nk && ok; ++s) {
            const int st = s % kGS;
            const uint32_t ph = static_cast<uint32_t>((s / kGS) & 1);
            ok = mbar_wait_warp(&bfull[st], ph, &g_gemm_error) && mbar_wait_warp(&afull[st], ph, &g_gemm_error);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
                const uint32_t a0 = smem_u32(astage + st * kAStage), b0 = smem_u32(bstage + st * S::kBStage);
#pragma unroll
                for (int j = 0; j < kGK / 16; ++j) {  // 16 k = two 8-k groups of A, 32 bytes of B's rows
                    const uint64_t bd = smem_desc_sw128(b0 + 32 * j);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t ad = smem_desc(a0 + h * kAHalf + 2 * j * (kGH * 16), kGH * 16, 128);
                        mma_ss(tmem + h * BN, ad, bd, idesc, (s | j) != 0 ? 1u : 0u);
                    }
                }
                mma_commit(&empty[st]);  // the stage is free once these MMAs have read it
            }
            __syncwarp();
        }
        if (ok && elect_one()) mma_commit(&dfull);
        __syncwarp();
    } else {
        // ------------------------------------------------ A: decode, then the epilogue
        const int q = warp % 4;                 // tensor-memory lane quarter of this warp
        const int hf = (warp - 2) / 4;          // half of the tile
        const int r = kGH * hf + 32 * q + lane;  // row of the tile
        const int64_t m = m0 + r;
        const bool live = m < M;
        const uint8_t* crow = codes + (live ? m : 0) * static_cast<int64_t>(KW / 2);
        const uint8_t* srow = scales + (live ? m : 0) * static_cast<int64_t>(KW / 16);
        RowLoad ring[kALoads];
        auto load = [&](int s) -> RowLoad {
            RowLoad v;
            if (live && s < nk) {
                const int sw = s % nkw;
                v.c0 = ld_stream_v4(crow + sw * 32);
                v.c1 = ld_stream_v4(crow + sw * 32 + 16);
                v.s4 = *reinterpret_cast<const uint32_t*>(srow + sw * 4);
            } else {
                v.c0 = v.c1 = make_uint4(0u, 0u, 0u, 0u);
                v.s4 = 0u;
            }
            return v;
        };
#pragma unroll
        for (int d = 0; d < kALoads; ++d) ring[d] = load(d);
        for (int s0 = 0; s0 < nk && ok; s0 += kALoads) {
#pragma unroll
            for (int d = 0; d < kALoads; ++d) {
                const int s = s0 + d;
                if (s < nk && ok) {
                    const int st = s % kGS;
                    const RowLoad cur = ring[d];
                    ring[d] = load(s + kALoads);
                    uint32_t a[32];
                    decode64(cur.c0, cur.c1, cur.s4, a);
                    if (s >= kGS)
                        ok = mbar_wait_warp(&empty[st], static_cast<uint32_t>(((s / kGS) & 1) ^ 1), &g_gemm_error);
                    if (ok) {
                        uint8_t* dst = astage + st * kAStage + hf * kAHalf + (r - kGH * hf) * 16;
#pragma unroll
                        for (int g = 0; g < kGK / 8; ++g)
                            *reinterpret_cast<uint4*>(dst + g * (kGH * 16)) =
                                make_uint4(a[4 * g], a[4 * g + 1], a[4 * g + 2], a[4 * g + 3]);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // read by the tensor cores
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&afull[st]);
                    }
                }
            }
        }
        // ---- epilogue: this warp's 32 rows, 16 tokens per tensor-memory load
        if (ok) ok = mbar_wait_warp(&dfull, 0, &g_gemm_error);
        tc_fence_after();
        if (ok) {
            const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
#pragma unroll 1
            for (int c = 0; c < BN / 16; ++c) {
                uint32_t v[16];
                tmem_ld_x16(tmem + lane_base + hf * BN + 16 * c, v);
                if (live) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = n0 + 16 * c + j;
                        if (n < nend) {
                            float* o = y + static_cast<int64_t>(n) * M + m;
                            *o = accumulate ? *o + __uint_as_float(v[j]) * ts : __uint_as_float(v[j]) * ts;
                        }
                    }
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kTmemCols)
                     : "memory");
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    return fn;
}

}  // namespace

namespace {

// x [P][K] bf16, read in boxes of 64 k x BN tokens (128 bytes a token,
// 128-byte swizzle); tokens past P read as zero.
bool make_x_map(CUtensorMap* map, const uint16_t* x, int64_t K, int64_t P, int bn)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(P)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGK), static_cast<cuuint32_t>(bn)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_gemm(const uint8_t* codes, const uint8_t* scales, float ts, const float* ts_e,
                        const int32_t* offsets, int E, const uint16_t* x, float* y, int64_t M, int64_t K, int64_t P,
                        int64_t tiles, int accumulate, int64_t KW, cudaStream_t s)
{
    CUtensorMap map;
    if (!make_x_map(&map, x, K, P, BN)) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kern = nvfp4_gemm_kernel<BN>;
    static OccCache occ;
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kGThreads, GemmShape<BN>::kSmem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((M + kGM - 1) / kGM), static_cast<unsigned>(tiles));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = GemmShape<BN>::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_flags() & kLaunchPdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, map, codes, scales, ts, ts_e, offsets, E, y, M, static_cast<int>(K),
                              static_cast<int>(P), accumulate, static_cast<int>(KW));
}

}  // namespace

bool gemm_supported(int64_t M, int64_t K, int64_t T)
{
    return M >= 1 && K >= kGK && K % kGK == 0 && K <= (int64_t(1) << 24) && T >= 1 && T <= (int64_t(1) << 24) &&
           M <= (int64_t(1) << 31) && (M + kGM - 1) / kGM <= 0x7FFFFFFF && (T + 255) / 256 <= 65535;
}

bool gemm_grouped_supported(int64_t E, int64_t M, int64_t K, int64_t P)
{
    return E >= 1 && E <= 65535 && M >= 1 && K >= kGK && K % kGK == 0 && K <= (int64_t(1) << 24) && P >= 1 &&
           P <= (int64_t(1) << 24) && E * M <= (int64_t(1) << 31) && (P + 127) / 128 + E <= 65535;
}

cudaError_t launch_nvfp4_gemm(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x, float* y,
                              int64_t M, int64_t K, int64_t T, cudaStream_t s)
{
    return launch_gemm<256>(codes, scales, ts, nullptr, nullptr, 1, x, y, M, K, T, (T + 255) / 256, 0, K, s);
}

// Token-tile width of the grouped form from the mean tokens per expert: a
// tile's MMAs cost BN columns however few of its tokens are real, and an
// expert with more tokens than BN has its weights decoded once per tile,
// which costs more. Measured on 256 experts of 1024 x 2048 (GB300, µs per
// call for BN = 32 / 64 / 128): mean 16: 211 / 220 / 238; 32: 311 / 237 /
// 254; 48: 428 / 243 / 260; 64: 516 / 336 / 265; 128: 904 / 553 / 377.
static int grouped_tile_tokens(int64_t P, int64_t E)
{
    const int64_t mean = (P + E - 1) / E;
    return mean <= 16 ? 32 : (mean <= 48 ? 64 : 128);
}

cudaError_t launch_nvfp4_gemm_grouped(const uint8_t* codes, const uint8_t* scales, const float* ts,
                                      const int32_t* offsets, int E, const uint16_t* x, float* y, int64_t M,
                                      int64_t K, int64_t P, cudaStream_t s, bool accumulate, int64_t weight_k)
{
    if (weight_k <= 0) weight_k = K;
    if (weight_k % kGK != 0 || K % weight_k != 0) return cudaErrorInvalidValue;
    // tile slots: sum over experts of ceil(n_e / BN) <= P / BN + E
    int bn = grouped_tile_tokens(P, E);
    // the tile slots are the grid's y dimension (at most 65535, which
    // gemm_grouped_supported guarantees for 128-token tiles): wider tiles
    // where narrow ones would not fit
    while (bn < 128 && (P + bn - 1) / bn + E > 65535) bn *= 2;
    const int acc = accumulate ? 1 : 0;
    if (bn == 32)
        return launch_gemm<32>(codes, scales, 1.0f, ts, offsets, E, x, y, M, K, P, (P + 31) / 32 + E, acc, weight_k, s);
    if (bn == 64)
        return launch_gemm<64>(codes, scales, 1.0f, ts, offsets, E, x, y, M, K, P, (P + 63) / 64 + E, acc, weight_k, s);
    return launch_gemm<128>(codes, scales, 1.0f, ts, offsets, E, x, y, M, K, P, (P + 127) / 128 + E, acc, weight_k,
                            s);
}

cudaError_t read_and_clear_gemm_error(unsigned int* out)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *out = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace bqd
