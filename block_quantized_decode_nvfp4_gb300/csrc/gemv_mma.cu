// gemv_mma.cu -- tensor-core (tcgen05) GEMV for a few tokens (N <= 16), NVFP4.
//
// Y[n][m] = ts * sum_b scale[m][b] * sum_{k in b} e2m1[m][k] * X[n][k]: the
// multi-token form of the NVFP4 matvec that checks K+1 drafted tokens in one
// batched target forward ("robertbfuentes7-cloud/bw24" README, NVFP4 (W4)
// decode path and speculative decoding bullets).
//
// Every product is exact: an E2M1 element times its E4M3 block scale has at
// most 6 significant bits and lies in [2^-10, 2688], so it is an f16 value,
// and the activations are staged as f16 after an exact power-of-two scaling
// (or, when their range does not allow that, both operands are bf16, which
// also holds every such product). The tensor cores accumulate in fp32.
//
// Work split. Rows go in 128-row tiles (the MMA's M) and k in 256-k stages.
// A thread-block cluster of cs CTAs (up to 8) takes tc <= 4 consecutive
// tiles; rank r of the cluster takes the stages [r K/cs, (r + 1) K/cs) of
// every one of them, so it stages only that slice of the activations and
// uses it for all tc tiles, each tile in its own TMEM accumulator. The fp32
// partial sums of a tile are added in rank order through distributed shared
// memory, so results are deterministic. For 96 tiles of K = 4096 this gives
// 32 clusters of 4 CTAs with 3 tiles x 4 stages each (128 SMs busy, a
// quarter of the activations per CTA). Roles per CTA:
//  * warp 0: producer. 2-D tensor copies (TMA) bring 128 rows x 256 k of
//    codes (16 KiB, 128-byte swizzle) and their scales (2 KiB) into a ring
//    of up to 8 stages; the first four are requested by four lanes at the
//    CTA's start, the rest by lane 0 as the ring turns.
//  * warps 1..17 stage the activations (f16 after an exact power-of-two
//    scaling, or bf16) into shared memory once per CTA.
//  * warps 2..17: decoders in four groups of four warps; group g takes the
//    64-k chunk g of every stage, one row per thread (TMEM lane). A thread
//    decodes its chunk into f16 pairs and writes them to tensor memory
//    (tcgen05.st), which is the A operand of the MMA: the decoded weights
//    never pass through shared memory.
//  * warp 1: allocates all 512 TMEM columns (4 accumulators + 14 A slots of
//    32 columns); one elected lane issues the MMAs (M = 128, N = 16, K = 16
//    each; B = the staged activations in shared memory) into one fp32
//    accumulator of 16 columns per tile and frees A slots with
//    tcgen05.commit.
// Every wait is bounded; one that runs out sets a bit in the device error
// word and the kernel runs to its end without waiting again.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "gemv.h"
#include "host_util.h"
#include "stream.cuh"

namespace bqd {

// Device error word of the tensor-core kernel (kErrWaitTimeout).
__device__ unsigned int g_mma_error = 0;

namespace {

constexpr int kTileM = 128;                   // rows per CTA = MMA M
constexpr int kNPad = 16;                     // MMA N: tokens padded to 16
constexpr int kStageK = 256;                  // k per ring stage
constexpr int kChunkK = 64;                   // k per decode step / A slot
constexpr int kChunksPerStage = kStageK / kChunkK;
constexpr int kMaxStages = 8;                 // ring stages: as many as shared memory allows, 3..8
constexpr int kASlots = 14;                   // A slots in TMEM, 32 columns each
constexpr int kTmemCols = 512;                // D: columns [16 j, 16 j + 16) for tile j < 4; A: [64, 512)
constexpr int kACol0 = 64;
constexpr int kMaxTiles = 4;                  // tiles per cluster (accumulators per CTA)
constexpr int kDecGroups = 4;                 // decoder groups: group g takes chunk g of every stage
constexpr int kDecWarps = 4 * kDecGroups;     // one warp per TMEM lane quarter per group
constexpr int kThreads = (2 + kDecWarps) * kWarp;
constexpr int kCodesStage = kTileM * (kStageK / 2);  // 16 KiB
constexpr int kScalesStage = kTileM * (kStageK / 16);  // 2 KiB
constexpr int kStageBytes = kCodesStage + kScalesStage;
constexpr int kMaxCluster = 8;
constexpr int kLoadsInFlight = 8;             // activation loads per thread in flight
// Ring stages requested at the CTA's start; the producer requests the rest
// once the activations are staged. Requesting all eight at once (about
// 19 MB from 128 CTAs) delayed everything else the CTAs fetched at start by
// up to 3 us; four measured best (12288 x 4096, N = 8: 16.6 us back to back
// against 17.4 us with eight).
constexpr int kInitStages = 4;
// The CTA takes all of TMEM (512 columns). At least 116 KiB of shared
// memory per CTA keeps two CTAs of this kernel (from any launches, on any
// streams) off the same SM, so a TMEM allocation here never waits for a CTA
// that may itself be waiting on a cluster peer.
constexpr int kMinSmem = 116 * 1024;
static_assert(kDecGroups == kChunksPerStage, "one chunk of every stage per decoder group");
constexpr int kSmemLimit = 225 * 1024;  // dynamic part; static shared memory stays below 2 KiB

static_assert(kStageBytes % 1024 == 0, "stages must keep the 1024-byte alignment of the swizzled codes");
static_assert(kACol0 + kASlots * 32 <= kTmemCols, "TMEM layout");
static_assert(kASlots >= kDecGroups, "slot bookkeeping");
static_assert(kMaxTiles * 16 <= kACol0 && kMaxTiles <= kDecGroups, "one accumulator and one epilogue group per tile");

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major, no swizzle: start address, the
// byte distance between core matrices (8 rows x 16 bytes) adjacent in k
// (lbo) and adjacent in rows (sbo), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}

// D[tmem_d] (+)= A[tmem_a] * B[desc]^T, M = 128, N = 16, K = 16, f16 or bf16
// operands (as idesc says), fp32 accumulation.
__device__ __forceinline__ void mma_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 columns of this warp's 32 TMEM lanes from 32 registers per thread.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
        "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
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

// One lane of the (converged) warp; the same lane every time.
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(const void* local, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    return remote;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// 16 bytes from global memory. A thread's batch of these stays in program
// order ahead of the code that uses the values, so the batch is in flight
// at once rather than one load per round trip.
__device__ __forceinline__ uint4 ld_global_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------ decode
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h)
{
    const float2 f = f16x2_to_float2(h);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);  // exact: the products fit in bf16
    return *reinterpret_cast<uint32_t*>(&b);
}

// 64 consecutive k of one row (32 code bytes c0, c1 and the 4 block scales in
// s4) to 32 pairs, pair j = elements 2j (low half) and 2j+1, scaled exactly
// by the block scale; f16 pairs, or bf16 pairs when !F16.
template <bool F16>
__device__ __forceinline__ void decode_chunk(const uint4& c0, const uint4& c1, uint32_t s4, uint32_t (&a)[32])
{
    const uint32_t s01 = e4m3x2_to_f16x2(s4 & 0xFFFFu), s23 = e4m3x2_to_f16x2(s4 >> 16);
    const uint32_t sb[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232), __byte_perm(s23, 0, 0x1010),
                            __byte_perm(s23, 0, 0x3232)};
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // word i = k 8i..8i+7 of the chunk, block i / 2
        uint32_t h[4];
        e2m1x8_to_f16x2(w[i], h);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t p = hmul2_bits(h[j], sb[i >> 1]);
            a[4 * i + j] = F16 ? p : f16x2_to_bf16x2(p);
        }
    }
}

// ------------------------------------------------------------ kernel
// Dynamic shared memory (1024-byte aligned): ring [ns][codes 16 KiB |
// scales 2 KiB], then the activations B of the CTA's k slice (its nsr
// stages, used for every tile of the cluster): 32 groups per stage of
// [brows tokens][8 k] as f16 (or bf16), brows * 16
// bytes per group: the K-major core-matrix layout with brows * 16 bytes
// between k-adjacent core matrices. With brows = 16 the second 8-token core
// matrix follows at +128 bytes; with brows = 8 (N <= 8) the descriptor's
// row-group stride is 0, so MMA columns 8..15 repeat columns 0..7 and are
// never read. With cs > 1, a receive area at recv_off holds the partial sums
// that the cluster's CTAs push to the rank owning each row: [cs ranks][16
// tokens][rows_max rows] fp32. It is used for nothing else, so a peer can
// write it while this CTA still runs its MMAs.
__global__ void __launch_bounds__(kThreads, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_scales,
                    const uint16_t* __restrict__ x, float* __restrict__ y, float ts, int M, int K, int N, int cs, int tc,
                    int tiles, int ns, int brows, int recv_off)
{
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], afull[kASlots], aempty[kASlots], dfull;
    __shared__ uint32_t s_tmem;
    // Exponent range of each token's activations per warp (warp 0 stages
    // none; its row ends up holding the CTA's range): emax | emin << 9 |
    // bad << 18, emax in [0, 255] (0 = no nonzero value), emin in [0, 256]
    // (256 = none).
    __shared__ uint32_t s_range[kThreads / kWarp][kNPad];

    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    unsigned char* ring = smem;
    unsigned char* bsm = smem + ns * kStageBytes;
    const int gbytes = brows * 16;  // bytes of B per 8 k

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int rank = cs > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int nst_all = K / kStageK;
    // The cluster's tiles [tile0, tile0 + tcl); this CTA's stages
    // [s_lo, s_lo + nsr) of each. Units (tile, stage) go tile-major:
    // unit t = tile t / nsr, stage s_lo + t % nsr.
    const int tile0 = static_cast<int>(blockIdx.x / cs) * tc;
    const int tcl = min(tc, tiles - tile0);
    const int s_lo = nst_all * rank / cs, nsr = nst_all * (rank + 1) / cs - s_lo;
    const int nst = tcl * nsr;
    auto unit_stage = [&](int t) { return s_lo + t % nsr; };
    auto unit_row0 = [&](int t) { return (tile0 + t / nsr) * kTileM; };
    auto group_k = [&](int g) { return s_lo * kStageK + 8 * g; };
    // Rows of the cluster: rank o owns rows [R o / cs, R (o + 1) / cs).
    const int R = tcl * kTileM, rows_max = (R + cs - 1) / cs;
    float* recv = reinterpret_cast<float*>(smem + recv_off);

    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < ns; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kDecWarps);
            }
            for (int s = 0; s < kASlots; ++s) {
                mbar_init(&afull[s], 4);  // the four warps of the group that owns the chunk
                mbar_init(&aempty[s], 1);
            }
            mbar_init(&dfull, 1);
            fence_barrier_init();
            prefetch_map(&map_codes);
            prefetch_map(&map_scales);
        }
        __syncwarp();
        // The first stages need no wait. They do not depend on the previous
        // kernel in the stream either, so the first kInitStages of them start
        // at once, while warp 1 allocates tensor memory and before the
        // dependent-launch wait (the weights must not be written by that
        // kernel). Lane t requests stage t.
        const int t = lane;
        if (t < nst && t < ns && t < kInitStages) {
            mbar_arrive_expect_tx(&full[t], kStageBytes);
            tma_load_2d(ring + t * kStageBytes, &map_codes, unit_stage(t) * (kStageK / 2), unit_row0(t), &full[t]);
            tma_load_2d(ring + t * kStageBytes + kCodesStage, &map_scales, unit_stage(t) * (kStageK / 16),
                        unit_row0(t), &full[t]);
        }
    }
    static_assert(kMaxStages <= kWarp, "one lane per initial stage");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    pdl_trigger();

    // ---- activations, pass 1 (warps 1..17; warp 0 has just issued the
    // ring's first copies): B = f16(x * 2^4) written while each token's
    // exponent range is scanned. Each thread keeps one token, with up to
    // eight 16-byte loads in flight together. The 2^4 prescale is exact for
    // 2^-21 <= |x| < 2^11; a token outside that window takes pass 2.
    pdl_wait();  // the activations may come from the previous kernel in the stream
    const int groups = nsr * (kStageK / 8);  // B covers the CTA's stages once; 8 k = one 16-byte piece
    {
        constexpr int kStagers = kThreads - kWarp;
        const int xt = threadIdx.x - kWarp;  // < 0 in warp 0
        const int active = (kStagers / N) * N, gstep = kStagers / N;
        // Every CTA reads the same activations: each starts at its own place
        // so that the CTAs do not all ask for the same lines at once.
        const int rot = static_cast<int>((blockIdx.x * 97u) % static_cast<unsigned>(groups));
        const int n = (xt + N * kWarp) % N;  // lane l of any warp: token l % N when N divides 32
        int emax = 0, emin = INT_MAX, bad = 0;
        if (xt >= 0 && xt < active) {
            const uint16_t* xn = x + static_cast<int64_t>(n) * K;
            for (int gi = xt / N; gi < groups; gi += kLoadsInFlight * gstep) {
                uint4 u[kLoadsInFlight];
#pragma unroll
                for (int j = 0; j < kLoadsInFlight; ++j) {
                    int g = gi + j * gstep + rot;
                    if (g >= groups) g -= groups;
                    u[j] = gi + j * gstep < groups ? ld_global_v4(xn + group_k(g)) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int j = 0; j < kLoadsInFlight; ++j) {
                    if (gi + j * gstep >= groups) break;
                    int g = gi + j * gstep + rot;
                    if (g >= groups) g -= groups;
                    const uint32_t wv[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
                    uint32_t o[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t b = (wv[e2] >> (16 * h)) & 0x7FFFu;
                            const int e = static_cast<int>(b >> 7);
                            if (b != 0) {
                                if (e == 0 || e == 255) bad = 1;  // subnormal, inf or NaN
                                emax = max(emax, e);
                                emin = min(emin, e);
                            }
                        }
                        __half2 hv = __floats2half2_rn(bf16_lo(wv[e2]) * 16.f, bf16_hi(wv[e2]) * 16.f);
                        o[e2] = *reinterpret_cast<uint32_t*>(&hv);
                    }
                    *reinterpret_cast<uint4*>(bsm + g * gbytes + n * 16) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
        // Per-token range: reduce over the warp's lanes of each token, then
        // one plain store per warp and token (shared atomics from every warp
        // on a few words took over a microsecond to settle)
        if ((kWarp % N) == 0) {  // lane l holds token l % N
            for (int off = N; off < kWarp; off <<= 1) {
                emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, off));
                emin = min(emin, __shfl_xor_sync(0xFFFFFFFFu, emin, off));
                bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, off);
            }
        } else {
            // the reductions read every lane's own values, so lane t keeps
            // token t's result apart until the loop ends
            int tmax = 0, tmin = INT_MAX, tbad = 0;
            for (int t = 0; t < N; ++t) {
                const int mx = __reduce_max_sync(0xFFFFFFFFu, n == t ? emax : 0);
                const int mn = __reduce_min_sync(0xFFFFFFFFu, n == t ? emin : INT_MAX);
                const int bd = static_cast<int>(__reduce_or_sync(0xFFFFFFFFu, n == t ? static_cast<unsigned>(bad) : 0u));
                if (lane == t) {
                    tmax = mx;
                    tmin = mn;
                    tbad = bd;
                }
            }
            emax = tmax;
            emin = tmin;
            bad = tbad;
        }
        if (lane < N)  // lane t now holds token t's range over the warp
            s_range[warp][lane] = static_cast<uint32_t>(emax) | static_cast<uint32_t>(min(emin, 256)) << 9 |
                                  static_cast<uint32_t>(bad) << 18;
    }
    __syncthreads();
    // Staging mode of the CTA: 0 = f16 with the fixed 2^4 prescale (pass 1
    // is final); 1 = f16 with a per-token prescale 2^-sexp that puts the
    // token's largest |x| in [2^14, 2^15), exact when every nonzero |x| of
    // the token lies within 31 binades of the largest; 2 = bf16 operands.
    // Thread t < N of warp 1 judges token t; the barriers OR the verdicts.
    int need2 = 0, need1 = 0;
    if (warp == 1 && lane < N) {
        const int t = lane;
        int emax = 0, emin = 256, bad = 0;
        for (int w = 1; w < kThreads / kWarp; ++w) {
            const uint32_t r = s_range[w][t];
            emax = max(emax, static_cast<int>(r & 0x1FFu));
            emin = min(emin, static_cast<int>((r >> 9) & 0x1FFu));
            bad |= static_cast<int>(r >> 18);
        }
        s_range[0][t] = static_cast<uint32_t>(emax) | static_cast<uint32_t>(emin) << 9;  // read by token_sexp
        const bool none = emin == 256;
        need2 = bad || (!none && emax - emin > 31);
        need1 = !none && (emin < 127 - 21 || emax > 127 + 10);
    }
    const int any2 = __syncthreads_or(need2), any1 = __syncthreads_or(need1);
    const int mode = any2 ? 2 : any1 ? 1 : 0;
    const bool f16 = mode != 2;
    auto token_sexp = [&](int n) {
        if (mode == 0) return -4;
        if (mode == 2 || n >= N || (s_range[0][n] >> 9) == 256u) return 0;
        return static_cast<int>(s_range[0][n] & 0x1FFu) - 127 - 14;
    };
    if (mode != 0) {
        // ---- pass 2 (all threads, only for activations outside the window)
        for (int i = threadIdx.x; i < groups * N; i += kThreads) {
            const int n = i % N, g = i / N;
            uint4 u = ld_global_v4(x + static_cast<int64_t>(n) * K + group_k(g));
            if (f16) {
                // 2^-sexp as two exact factors (it can exceed the fp32 range)
                const int e = -token_sexp(n), e1 = e / 2, e2 = e - e1;
                const float f1 = __int_as_float((e1 + 127) << 23), f2 = __int_as_float((e2 + 127) << 23);
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    __half2 hv = __floats2half2_rn(bf16_lo(wv[j]) * f1 * f2, bf16_hi(wv[j]) * f1 * f2);
                    o[j] = *reinterpret_cast<uint32_t*>(&hv);
                }
                u = make_uint4(o[0], o[1], o[2], o[3]);
            }
            *reinterpret_cast<uint4*>(bsm + g * gbytes + n * 16) = u;
        }
        __syncthreads();
    }
    // Tokens N..15 of B are not written: they only feed accumulator
    // columns that are never read.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B is read by the tensor cores
    __syncthreads();

    const int nchunks = nst * kChunksPerStage;  // even
    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            uint32_t slot = 0, phase = 0;
            for (int t = 0; t < nst; ++t) {
                if (t >= kInitStages || t >= ns) {
                    // a slot's first use needs no wait
                    if (t >= ns && ok) ok = mbar_wait(&empty[slot], phase ^ 1u, &g_mma_error);
                    mbar_arrive_expect_tx(&full[slot], kStageBytes);
                    tma_load_2d(ring + slot * kStageBytes, &map_codes, unit_stage(t) * (kStageK / 2), unit_row0(t),
                                &full[slot]);
                    tma_load_2d(ring + slot * kStageBytes + kCodesStage, &map_scales, unit_stage(t) * (kStageK / 16),
                                unit_row0(t), &full[slot]);
                }
                if (++slot == ns) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            // Every copy has landed before the CTA can exit: the decoders
            // waited for all of them, and the last wait below covers a
            // decoder that gave up.
            if (ok) {
                const int first = nst > ns ? nst - ns : 0;
                for (int t = first; t < nst && ok; ++t)
                    ok = mbar_wait(&full[t % ns], static_cast<uint32_t>((t / ns) & 1), &g_mma_error);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue
        // The whole warp runs the loop on warp-uniform values and one
        // elected lane issues: about 33 cycles per MMA, against 50+ when a
        // single lane runs the loop on per-thread values.
        const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
        const uint64_t bdesc0 =
            __shfl_sync(0xFFFFFFFFu, smem_desc(smem_u32(bsm), gbytes, brows == 16 ? 128 : 0), 0);
        const uint32_t bstep = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(gbytes >> 4), 0);  // per 8 k
        const uint32_t idesc = __shfl_sync(0xFFFFFFFFu,
                                           (1u << 4) | (f16 ? 0u : (1u << 7) | (1u << 10)) |
                                               (static_cast<uint32_t>(kNPad >> 3) << 17) |
                                               (static_cast<uint32_t>(kTileM >> 4) << 24),
                                           0);
        // Chunks go in fours (nchunks is a multiple of 4): lanes 0..3 wait
        // for the four chunks' A slots with one instruction, so each barrier
        // round trip (~150 cycles) is paid once per 16 MMAs and overlaps the
        // previous batch's work.
        constexpr int kBatch = 4;
        static_assert(kASlots >= 2 * kBatch, "decoders must be able to run a batch ahead");
        static_assert(kBatch == kChunksPerStage, "a batch is one unit (one stage of one tile)");
        bool ok = true;
        uint32_t slot = 0, phase = 0;
        int sb = 0, ti = 0;  // the batch's unit: stage within B, tile of the cluster
        for (int c = 0; c < nchunks; c += kBatch) {
            uint32_t ws = slot + (lane & (kBatch - 1)), wp = phase;
            if (ws >= kASlots) {
                ws -= kASlots;
                wp ^= 1u;
            }
            if (ok && lane < kBatch) ok = mbar_wait(&afull[ws], wp, &g_mma_error);
            __syncwarp();
            tc_fence_after();
            // the unit's tile accumulator, and whether this batch starts it
            const uint32_t dcol = tm + 16u * static_cast<uint32_t>(ti);
            const bool first = sb == 0;
            if (elect_one()) {
#pragma unroll
                for (int h = 0; h < kBatch; ++h) {
                    uint32_t sl = slot + h;
                    if (sl >= kASlots) sl -= kASlots;
                    const uint32_t a_col = tm + kACol0 + sl * 32;
#pragma unroll
                    for (int j = 0; j < kChunkK / 16; ++j) {
                        // 16 k = two groups of B
                        const uint64_t bdesc =
                            bdesc0 + static_cast<uint64_t>(((sb * kBatch + h) * (kChunkK / 8) + 2 * j) * bstep);
                        mma_tmem_a(dcol, a_col + 8 * j, bdesc, idesc, (first && (h | j) == 0) ? 0u : 1u);
                    }
                    mma_commit(&aempty[sl]);
                }
            }
            __syncwarp();
            slot += kBatch;
            if (slot >= kASlots) {
                slot -= kASlots;
                phase ^= 1u;
            }
            if (++sb == nsr) {
                sb = 0;
                ++ti;
            }
        }
        if (elect_one()) mma_commit(&dfull);
        __syncwarp();
    } else {
        // ------------------------------------------------ decoders
        // Group g decodes chunk g (k 64g .. 64g+63) of every stage; the four
        // warps of a group cover the four TMEM lane quarters (one row per
        // thread). Four warps per scheduler hide each other's latencies.
        const int grp = (warp - 2) / 4;
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int row = q * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const int swz = row & 7;
        bool ok = true;
        uint32_t sslot = 0, sphase = 0;
        uint32_t aslot = grp, aphase = 0;
        for (int t = 0; t < nst; ++t) {
            const int c = t * kChunksPerStage + grp;
            if (ok) ok = mbar_wait_warp(&full[sslot], sphase, &g_mma_error);
            const unsigned char* st = ring + sslot * kStageBytes;
            const uint4 srow = *reinterpret_cast<const uint4*>(st + kCodesStage + row * 16);
            const unsigned char* rp = st + row * 128;
            const uint4 c0 = *reinterpret_cast<const uint4*>(rp + (((2 * grp) ^ swz) << 4));
            const uint4 c1 = *reinterpret_cast<const uint4*>(rp + (((2 * grp + 1) ^ swz) << 4));
            const uint32_t s4 = grp == 0 ? srow.x : grp == 1 ? srow.y : grp == 2 ? srow.z : srow.w;
            uint32_t a[32];
            if (f16)
                decode_chunk<true>(c0, c1, s4, a);
            else
                decode_chunk<false>(c0, c1, s4, a);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sslot]);  // this warp no longer reads the stage
            if (++sslot == ns) {
                sslot = 0;
                sphase ^= 1u;
            }
            if (ok && c >= kASlots) ok = mbar_wait_warp(&aempty[aslot], aphase ^ 1u, &g_mma_error);
            tmem_st_x32(tmem + lane_base + kACol0 + aslot * 32, a);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[aslot]);
            aslot += kDecGroups;  // chunk c + kDecGroups
            if (aslot >= kASlots) {
                aslot -= kASlots;
                aphase ^= 1u;
            }
        }
        // ---- epilogue: decoder group g takes this row's 16 accumulators of
        // the cluster's tile g (groups past the cluster's tiles have nothing
        // to do)
        if (grp < tcl) {
            if (ok) ok = mbar_wait_warp(&dfull, 0, &g_mma_error);
            tc_fence_after();
            uint32_t v[16];
            tmem_ld_x16(tmem + lane_base + 16 * grp, v);
            if (cs == 1) {  // all of k: the result itself
                const int64_t m = static_cast<int64_t>(tile0 + grp) * kTileM + row;
                if (m < M) {
#pragma unroll
                    for (int n = 0; n < kNPad; ++n)
                        if (n < N) y[static_cast<int64_t>(n) * M + m] = ldexpf(__uint_as_float(v[n]), token_sexp(n)) * ts;
                }
            } else {
                // push the row's partial sums (in x's own scale: the staging
                // scale is per CTA) into the receive area of its owner
                const int q = grp * kTileM + row;
                const int o = ((q + 1) * cs - 1) / R;  // the rank with R o / cs <= q < R (o + 1) / cs
                const uint32_t dst =
                    mapa(recv + (rank * kNPad) * rows_max + (q - R * o / cs), static_cast<uint32_t>(o));
#pragma unroll
                for (int n = 0; n < kNPad; ++n)
                    if (n < N) st_cluster_f32(dst + 4u * n * rows_max, ldexpf(__uint_as_float(v[n]), token_sexp(n)));
            }
        }
        tc_fence_before();
    }

    if (cs > 1) {
        // ---- cluster reduction: after the barrier (its release / acquire
        // makes the pushed partials visible) each rank sums its own rows
        // over all ranks, in rank order, from its receive area. Nothing is
        // read or written in a peer's shared memory after the barrier, so
        // CTAs may then exit.
        cluster_sync();
        const int q_lo = R * rank / cs, q_hi = R * (rank + 1) / cs, nq = q_hi - q_lo;
        for (int i = threadIdx.x; i < nq * N; i += kThreads) {
            const int n = i / nq, qq = i % nq, q = q_lo + qq;
            float s = 0.f;
#pragma unroll
            for (int p = 0; p < kMaxCluster; ++p)
                if (p < cs) s += recv[(p * kNPad + n) * rows_max + qq];  // rank order
            const int64_t m = static_cast<int64_t>(tile0) * kTileM + q;
            if (m < M) y[static_cast<int64_t>(n) * M + m] = s * ts;
        }
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ------------------------------------------------------------ host side
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

// 2-D map of a row-major byte matrix [rows][cols] read in boxes of
// box_cols x 128 rows; rows past the end read as zero.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_cols, bool swizzle128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(kTileM)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Receive area of the cluster reduction: [cs][16 tokens][rows per rank].
size_t recv_bytes(int cs, int tc)
{
    return cs > 1 ? static_cast<size_t>(cs) * kNPad * ((tc * kTileM + cs - 1) / cs) * sizeof(float) : 0;
}

// Shared memory of a CTA with `stages_per_cta` stages of k, B rows of
// `brows` tokens, a ring of `ns` stages and `recv` bytes of receive area.
size_t smem_bytes(int stages_per_cta, int brows, int ns, size_t recv)
{
    const size_t s = 1024 + static_cast<size_t>(ns) * kStageBytes +
                     static_cast<size_t>(stages_per_cta) * kStageK * brows * 2 + recv;
    return s < static_cast<size_t>(kMinSmem) ? static_cast<size_t>(kMinSmem) : s;
}

// Clusters of `ks` CTAs with `smem` bytes of dynamic shared memory each that
// fit on the device at once (cached per device and cluster size).
int active_clusters(int dev, int sms, int ks, size_t smem)
{
    static std::mutex mu;
    static int cache[64][kMaxCluster + 1] = {};
    static size_t cache_smem[64][kMaxCluster + 1] = {};
    std::lock_guard<std::mutex> g(mu);
    if (dev >= 0 && dev < 64 && cache[dev][ks] && cache_smem[dev][ks] == smem) return cache[dev][ks];
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ks * sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, gemv_mma_kernel, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = sms / ks;
        if (n < 1) n = 1;
    }
    if (dev >= 0 && dev < 64) {
        cache[dev][ks] = n;
        cache_smem[dev][ks] = smem;
    }
    return n;
}

}  // namespace

bool mma_gemv_supported(int64_t M, int64_t K, int N)
{
    if (N < 1 || N > kNPad || M < 1 || M > (int64_t(1) << 30) || K < kStageK || K % kStageK != 0 ||
        K > (int64_t(1) << 20))
        return false;
    const int64_t per_cta = (K / kStageK + kMaxCluster - 1) / kMaxCluster;
    return smem_bytes(static_cast<int>(per_cta), N <= 8 ? 8 : 16, 3, recv_bytes(kMaxCluster, 1)) <=
           static_cast<size_t>(kSmemLimit);
}

cudaError_t launch_nvfp4_gemv_mma(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                  float* y, int64_t M, int64_t K, int N, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const DevInfo di = dev_info(dev);
    const int limit = di.max_smem_optin < kSmemLimit ? di.max_smem_optin : kSmemLimit;
    static OccCache occ;
    blocks_per_sm(occ, reinterpret_cast<const void*>(gemv_mma_kernel), dev, kThreads,
                  smem_bytes(1, 8, 3, 0));  // sets the shared-memory opt-in

    const int tiles = static_cast<int>((M + kTileM - 1) / kTileM);
    const int nst_all = static_cast<int>(K / kStageK);
    const int brows = N <= 8 ? 8 : 16;
    // Clusters of cs CTAs over tc tiles. Cost in tenths of a stage's time:
    // per wave, the CTA's units plus a fixed 2 stages plus ~0.6 stage per
    // stage of activations staged; a cluster reduction adds ~3 stages. Ties
    // go to the smaller cluster, then to fewer tiles per cluster.
    int cs = 0, tc = 0;
    int64_t best_cost = INT64_MAX;
    for (int c = 1; c <= kMaxCluster && c <= nst_all; ++c) {
        const int xst = (nst_all + c - 1) / c;  // stages of k per CTA
        for (int t = 1; t <= kMaxTiles && t <= tiles; ++t) {
            const size_t sm = smem_bytes(xst, brows, 3, recv_bytes(c, t));
            if (sm > static_cast<size_t>(limit)) continue;
            // one CTA per SM whatever its shared memory (see kMinSmem), so
            // the count depends on c alone; asked once per c at the limit
            const int act = active_clusters(dev, di.sms, c, static_cast<size_t>(limit));
            const int64_t clusters = (tiles + t - 1) / t;
            const int64_t waves = (clusters + act - 1) / act;
            const int64_t cost = waves * (10 * t * xst + 20 + 6 * xst) + (c > 1 ? 30 : 0);
            if (cost < best_cost) {
                best_cost = cost;
                cs = c;
                tc = t;
            }
        }
    }
    if (cs == 0) return cudaErrorInvalidValue;
    const int per_cta = (nst_all + cs - 1) / cs;  // stages of k per CTA (B holds them once)
    // Ring: as many stages as shared memory holds (up to 8, no more than the
    // CTA's stages); at least 3 fit by the choice of cs and tc.
    const size_t recv = recv_bytes(cs, tc);
    const int64_t bbytes = static_cast<int64_t>(per_cta) * kStageK * brows * 2;
    int ns = static_cast<int>((limit - 1024 - bbytes - static_cast<int64_t>(recv)) / kStageBytes);
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns > per_cta * tc) ns = per_cta * tc;
    const size_t smem = smem_bytes(per_cta, brows, ns, recv);
    const int recv_off = static_cast<int>(ns * kStageBytes + bbytes);

    CUtensorMap map_codes, map_scales;
    if (!make_map(&map_codes, codes, M, K / 2, kStageK / 2, true) ||
        !make_map(&map_scales, scales, M, K / 16, kStageK / 16, false))
        return cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    const int clusters = (tiles + tc - 1) / tc;
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cs > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(cs);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (launch_flags() & kLaunchPdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemv_mma_kernel, map_codes, map_scales, x, y, ts, static_cast<int>(M),
                              static_cast<int>(K), N, cs, tc, tiles, ns, brows, recv_off);
}

cudaError_t read_and_clear_mma_error(unsigned int* out)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_mma_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *out = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_mma_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace bqd
