// gemv_stream.cu -- HBM-streaming GEMV for one token (N = 1), NVFP4 and Q8_0.
//
// y[m] = ts * sum_b scale[m][b] * sum_{k in b} elem[m][k] * x[k]
// ("robertbfuentes7-cloud/bw24" README, NVFP4 (W4) decode path;
// "avifenesh/memra" README, Decode kernels: NVFP4 and Q8_0 matvecs).
//
// One persistent CTA per SM owns a balanced, contiguous range of rows. Warp
// 0 is a producer: it streams the rows' codes and scales, tile by tile
// (16 rows x up to 2048 k), with 1-D bulk copies into a ring of shared-
// memory stages completed on mbarriers, so ~150-200 KB per SM are in flight
// without holding any register; only the first two stages are requested
// before the activations are staged. Eight consumer warps take two rows each of
// a stage, lanes along k, and decode in registers:
//  * NVFP4: E2M1 pairs -> f16x2 (hardware convert); the activations are
//    staged once per CTA as f16, pre-multiplied by an exact power of two
//    2^-s chosen from their largest exponent, and multiplied in by the
//    mixed-precision FMA (f16 x f16 products are exact in fp32, the sum is
//    fp32). The block scale is applied per 16-element block. f16 holds
//    every bf16 value exactly when all nonzero magnitudes lie within 31
//    binades below the largest; otherwise (or with inf/NaN/subnormal x) the
//    CTA takes an exact path with fp32 activations and fp32 FMAs.
//  * Q8_0: int8 -> f16 exactly (byte permute into 1024 + q + 128, subtract),
//    then the same mixed-precision FMAs (exact path: int8 -> fp32).
// Rows finish with a warp-shuffle reduction; results are deterministic.
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

// Device error word of the streaming kernels (kErrWaitTimeout); read and
// cleared by read_and_clear_stream_error().
__device__ unsigned int g_stream_error = 0;

namespace {

constexpr int kCW = 8;                      // consumer warps
constexpr int kCT = kCW * kWarp;            // consumer threads
constexpr int kThreadsS = (kCW + 1) * kWarp;
constexpr int kSmemLimit = 227 * 1024;
// Ring stages requested before the activations are staged; the rest follow
// once they are. A smaller first burst lets the activations and the first
// stages through sooner: back to back with dependent launch, NVFP4
// 12288 x 4096 took 9.8 us with two against 11.0 us with the whole ring at
// once (Q8_0 12288 x 4096: 12.1 against 13.2 us).
constexpr int kInitStagesS = 2;

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

struct FmtNvfp4 {
    static constexpr int kCodeNum = 1, kCodeDen = 2;  // code bytes per k
};
struct FmtQ8 {
    static constexpr int kCodeNum = 1, kCodeDen = 1;
};

// Activations in shared memory, 2 bytes per element (f16 in fast mode, the
// raw bf16 in exact mode), 32-element chunks of 64 bytes with the 16-byte
// piece p of chunk c at slot p ^ ((c >> 1) & 3): the 32 lanes, which read the
// same piece of 32 consecutive chunks, hit distinct banks.
__device__ __forceinline__ int x_index(int c, int p) { return c * 32 + ((p ^ ((c >> 1) & 3)) << 3); }

// 32-element chunk cl of two rows, activation chunk cg; accumulates into
// acc[2]. FAST: f16 activations and mixed-precision FMAs. Otherwise exact:
// bf16 activations widened to fp32, fp32 FMAs.
template <bool FAST>
__device__ __forceinline__ void chunk_nvfp4(const uint8_t* c0, const uint8_t* c1, const uint8_t* s0,
                                            const uint8_t* s1, int cl, const uint16_t* xs, int cg, float (&acc)[2])
{
    const uint4 code[2] = {*reinterpret_cast<const uint4*>(c0 + 16 * cl),
                           *reinterpret_cast<const uint4*>(c1 + 16 * cl)};
    const float2 sc[2] = {e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(s0 + 2 * cl)),
                          e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(s1 + 2 * cl))};
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        float a0[2] = {0.f, 0.f}, a1[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int wi = 2 * b + j;
            const uint4 xq = *reinterpret_cast<const uint4*>(xs + x_index(cg, wi));
            const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t words[4] = {code[r].x, code[r].y, code[r].z, code[r].w};
                uint32_t h[4];
                e2m1x8_to_f16x2(words[wi], h);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (FAST) {
                        fma_f16x2(h[q], xp[q], a0[r], a1[r]);
                    } else {
                        const float2 wf = f16x2_to_float2(h[q]);
                        a0[r] = fmaf(wf.x, bf16_lo(xp[q]), a0[r]);
                        a1[r] = fmaf(wf.y, bf16_hi(xp[q]), a1[r]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) acc[r] = fmaf(b ? sc[r].y : sc[r].x, a0[r] + a1[r], acc[r]);
    }
}

template <bool FAST>
__device__ __forceinline__ void chunk_q8(const uint8_t* c0, const uint8_t* c1, const uint8_t* s0, const uint8_t* s1,
                                         int cl, const uint16_t* xs, int cg, float (&acc)[2])
{
    const uint4 qv[2][2] = {{*reinterpret_cast<const uint4*>(c0 + 32 * cl),
                             *reinterpret_cast<const uint4*>(c0 + 32 * cl + 16)},
                            {*reinterpret_cast<const uint4*>(c1 + 32 * cl),
                             *reinterpret_cast<const uint4*>(c1 + 32 * cl + 16)}};
    const float d[2] = {fp16_to_float(*reinterpret_cast<const uint16_t*>(s0 + 2 * cl)),
                        fp16_to_float(*reinterpret_cast<const uint16_t*>(s1 + 2 * cl))};
    float a0[2] = {0.f, 0.f}, a1[2] = {0.f, 0.f};
#pragma unroll
    for (int p = 0; p < 4; ++p) {  // 16-byte activation pieces = 8 elements = 2 int8 words
        const uint4 xq = *reinterpret_cast<const uint4*>(xs + x_index(cg, p));
        const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint4 half = p < 2 ? qv[r][0] : qv[r][1];
            const uint32_t words[4] = {half.x, half.y, half.z, half.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t w = words[(p & 1) * 2 + h];
                if constexpr (FAST) {
                    uint32_t q01, q23;
                    s8x4_to_f16x2(w, q01, q23);
                    fma_f16x2(q01, xp[2 * h], a0[r], a1[r]);
                    fma_f16x2(q23, xp[2 * h + 1], a0[r], a1[r]);
                } else {
                    float2 lo, hi;
                    s8x4_to_float(w, lo, hi);
                    a0[r] = fmaf(lo.x, bf16_lo(xp[2 * h]), a0[r]);
                    a1[r] = fmaf(lo.y, bf16_hi(xp[2 * h]), a1[r]);
                    a0[r] = fmaf(hi.x, bf16_lo(xp[2 * h + 1]), a0[r]);
                    a1[r] = fmaf(hi.y, bf16_hi(xp[2 * h + 1]), a1[r]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) acc[r] = fmaf(d[r], a0[r] + a1[r], acc[r]);
}

// Griddepcontrol (programmatic dependent launch). Without a dependent
// launch both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Dynamic shared memory: [x: K * 2 bytes][ring: ns stages][full, empty
// barriers]. A stage holds `rs` whole rows (codes then scales, exactly as in
// HBM), copied by two bulk copies. The 8 consumer warps are arranged as
// rs/2 row pairs x q = 16/rs parts of k; partial sums of the parts are added
// through shared memory.
template <class F>
__global__ void __launch_bounds__(kThreadsS, 1)
    gemv_stream_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, float ts,
                       const uint16_t* __restrict__ x, float* __restrict__ y, int64_t M, int64_t K, int rs, int ns,
                       long long wait_limit, int withhold_last)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_emax, s_emin, s_flags;
    __shared__ __align__(8) uint64_t xready;  // the activations are staged
    __shared__ float red[2][16][8];  // [stage parity][row of stage][k part]

    const int64_t cpitch = K * F::kCodeNum / F::kCodeDen, spitch = K / 16;
    const int64_t codes_stage = rs * cpitch, stage_bytes = codes_stage + rs * spitch;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
    unsigned char* ring = smem + K * 2;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + ns * stage_bytes);
    uint64_t* empty = full + ns;

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t r_lo = M * blockIdx.x / gridDim.x, r_hi = M * (blockIdx.x + 1) / gridDim.x;
    const int64_t nstages = (r_hi - r_lo + rs - 1) / rs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        s_emax = 0;
        s_emin = INT_MAX;
        s_flags = 0;
        mbar_init(&xready, 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_trigger();  // one resident CTA per SM: a dependent grid can only start as CTAs here exit

    if (warp == 0) {
        // ------------------------------------------------ producer
        bool ok = true;
        int64_t issued = 0;
        for (int64_t t = 0; t < nstages; ++t) {
            const int slot = static_cast<int>(t % ns);
            if (t >= ns)
                ok = mbar_wait(&empty[slot], static_cast<uint32_t>(((t / ns) - 1) & 1), &g_stream_error, wait_limit);
            if (t == kInitStagesS && ok) ok = mbar_wait(&xready, 0u, &g_stream_error, wait_limit);
            ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            if (withhold_last && t == nstages - 1) break;  // failure-path test: this stage never arrives
            const int64_t row0 = r_lo + t * rs;
            const int rows = static_cast<int>(r_hi - row0 < rs ? r_hi - row0 : rs);
            unsigned char* st = ring + slot * stage_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(rows * (cpitch + spitch)));
                bulk_g2s(st, codes + row0 * cpitch, static_cast<uint32_t>(rows * cpitch), &full[slot]);
                bulk_g2s(st + codes_stage, scales + row0 * spitch, static_cast<uint32_t>(rows * spitch),
                         &full[slot]);
            }
            issued = t + 1;
        }
        // Wait for every copy issued into the ring to land before exiting.
        if (lane == 0) {
            const int64_t first = issued > ns ? issued - ns : 0;
            for (int64_t t = first; t < issued; ++t)
                if (!mbar_wait(&full[t % ns], static_cast<uint32_t>((t / ns) & 1), &g_stream_error, wait_limit))
                    break;
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int ctid = threadIdx.x - kWarp;
    pdl_wait();  // the activations may come from the previous kernel in the stream
    // exponent range of the nonzero activations (bf16 biased exponents)
    int emax = 0, emin = INT_MAX, flags = 0;
    for (int64_t i = ctid; i < K / 2; i += kCT) {
        const uint32_t v = reinterpret_cast<const uint32_t*>(x)[i];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t b = (v >> (16 * h)) & 0x7FFFu;
            const int e = static_cast<int>(b >> 7);
            if (b == 0) continue;
            if (e == 0 || e == 255) flags = 1;  // subnormal, inf or NaN
            emax = max(emax, e);
            emin = min(emin, e);
        }
    }
    if (flags) atomicOr(&s_flags, 1);
    atomicMax(&s_emax, emax);
    atomicMin(&s_emin, emin);
    named_sync(1, kCT);
    // f16 holds x * 2^-sexp exactly when every nonzero |x| is within 31
    // binades of the largest; the largest lands in [2^14, 2^15).
    const bool fast = !s_flags && (s_emin == INT_MAX || s_emax - s_emin <= 31);
    const int sexp = fast && s_emin != INT_MAX ? s_emax - 127 - 14 : 0;
    for (int64_t i = ctid; i < K / 8; i += kCT) {  // 8 elements = one 16-byte piece
        uint4 u = reinterpret_cast<const uint4*>(x)[i];
        if (fast) {
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                __half2 hv = __floats2half2_rn(ldexpf(bf16_lo(w[q]), -sexp), ldexpf(bf16_hi(w[q]), -sexp));
                o[q] = *reinterpret_cast<uint32_t*>(&hv);
            }
            u = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>(xs + x_index(static_cast<int>(i / 4), static_cast<int>(i % 4))) = u;
    }
    named_sync(1, kCT);
    if (ctid == 0) mbar_arrive(&xready);

    const int cw = warp - 1;
    const int pairs = rs / 2, parts = kCW / pairs;
    const int pr = cw % pairs, part = cw / pairs;
    const int chunks = static_cast<int>(K / 32);
    const int c_lo = chunks * part / parts, c_hi = chunks * (part + 1) / parts;
    bool ok = true;
    for (int64_t t = 0; t < nstages; ++t) {
        const int slot = static_cast<int>(t % ns);
        if (ok) ok = mbar_wait(&full[slot], static_cast<uint32_t>((t / ns) & 1), &g_stream_error, wait_limit);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        const int64_t row0 = r_lo + t * rs;
        const int rows = static_cast<int>(r_hi - row0 < rs ? r_hi - row0 : rs);
        float acc[2] = {0.f, 0.f};
        if (ok && 2 * pr < rows) {
            const unsigned char* st = ring + slot * stage_bytes;
            const int ra = 2 * pr, rb = 2 * pr + 1 < rows ? 2 * pr + 1 : 2 * pr;
            const uint8_t* ca = st + ra * cpitch;
            const uint8_t* cb = st + rb * cpitch;
            const uint8_t* sa = st + codes_stage + ra * spitch;
            const uint8_t* sb = st + codes_stage + rb * spitch;
            for (int c = c_lo + lane; c < c_hi; c += kWarp) {
                if constexpr (F::kCodeDen == 2) {
                    if (fast)
                        chunk_nvfp4<true>(ca, cb, sa, sb, c, xs, c, acc);
                    else
                        chunk_nvfp4<false>(ca, cb, sa, sb, c, xs, c, acc);
                } else {
                    if (fast)
                        chunk_q8<true>(ca, cb, sa, sb, c, xs, c, acc);
                    else
                        chunk_q8<false>(ca, cb, sa, sb, c, xs, c, acc);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        const float v0 = warp_sum(acc[0]), v1 = warp_sum(acc[1]);
        if (parts == 1) {
            if (lane == 0 && ok) {
                if (2 * pr < rows) y[row0 + 2 * pr] = ldexpf(v0 * ts, sexp);
                if (2 * pr + 1 < rows) y[row0 + 2 * pr + 1] = ldexpf(v1 * ts, sexp);
            }
        } else {
            const int par = static_cast<int>(t & 1);
            if (lane == 0) {
                red[par][2 * pr][part] = v0;
                red[par][2 * pr + 1][part] = v1;
            }
            named_sync(2, kCT);
            if (part == 0 && lane < 2 && ok && 2 * pr + lane < rows) {
                float v = 0.f;
                for (int q = 0; q < parts; ++q) v += red[par][2 * pr + lane][q];
                y[row0 + 2 * pr + lane] = ldexpf(v * ts, sexp);
            }
        }
    }
}

// Failure-path test setting (bqd_debug_stream_fault): wait limit of the
// kernel's bounded waits, and whether the producer withholds the last stage.
struct StreamFault {
    long long wait_limit = kWaitCycles;
    int withhold_last = 0;
};
std::mutex g_fault_mu;
StreamFault g_fault;

StreamFault stream_fault()
{
    std::lock_guard<std::mutex> g(g_fault_mu);
    return g_fault;
}

template <class F>
cudaError_t launch_stream(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x, float* y,
                          int64_t M, int64_t K, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const DevInfo di = dev_info(dev);
    const int limit = di.max_smem_optin < kSmemLimit ? di.max_smem_optin : kSmemLimit;
    const int64_t room = limit - K * 2 - 2048;  // barriers + static shared memory
    const int64_t row_bytes = K * F::kCodeNum / F::kCodeDen + K / 16;
    // Largest row block (16, 8, 4 or 2 rows) that leaves at least three stages.
    int rs = 16;
    while (rs > 2 && room / (rs * row_bytes + 16) < 3) rs /= 2;
    int ns = static_cast<int>(room / (rs * row_bytes + 16));
    if (ns > 16) ns = 16;
    if (ns < 2) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(K * 2 + ns * rs * row_bytes + 16 * ns);
    auto kern = gemv_stream_kernel<F>;
    static OccCache occ;
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kThreadsS, smem);  // sets the smem opt-in
    int64_t grid = di.sms;
    if (grid > M) grid = M;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreadsS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_flags() & kLaunchPdl ? 1 : 0;
    const StreamFault f = stream_fault();
    return cudaLaunchKernelEx(&cfg, kern, codes, scales, ts, x, y, M, K, rs, ns, f.wait_limit, f.withhold_last);
}

}  // namespace

bool stream_gemv_supported(int64_t M, int64_t K, int N)
{
    // two rows of up to 16384 Q8_0 elements per stage, three stages: fits
    return N == 1 && M >= 1 && K >= 256 && K % 256 == 0 && K <= 16384;
}

cudaError_t launch_nvfp4_gemv_stream(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                     float* y, int64_t M, int64_t K, cudaStream_t s)
{
    return launch_stream<FmtNvfp4>(codes, scales, ts, x, y, M, K, s);
}

cudaError_t launch_q8_0_gemv_stream(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M,
                                    int64_t K, cudaStream_t s)
{
    return launch_stream<FmtQ8>(reinterpret_cast<const uint8_t*>(q), reinterpret_cast<const uint8_t*>(d), 1.0f, x,
                                y, M, K, s);
}

void set_stream_fault(int withhold_last, long long wait_limit)
{
    std::lock_guard<std::mutex> g(g_fault_mu);
    g_fault.withhold_last = withhold_last ? 1 : 0;
    g_fault.wait_limit = wait_limit > 0 ? wait_limit : kWaitCycles;
}

cudaError_t read_and_clear_stream_error(unsigned int* out)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_stream_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *out = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace bqd
