// moe_stream.cu -- the two projections of the routed MoE layer as HBM streams
// (sm_103a): gate_up (g, u and h = SiLU(g) * u) and down, for experts whose
// sizes keep every row pitch a multiple of 16 bytes (H % 256 == 0 and
// I % 256 == 0).
//
// What is computed is the MoE layer of moe.cu ("robertbfuentes7-cloud/bw24"
// README, MoE bullet: routed tokens batched expert-major, each selected
// expert's weights decoded once for all of its tokens).
//
// Work split. The rows of all active experts (experts with a non-empty
// segment of the expert-major list, in increasing order) form one virtual
// row space, cut into equal contiguous ranges, one per CTA (one CTA per SM).
// Warp 0 streams a CTA's rows with 1-D bulk copies into a ring of shared-
// memory stages (a stage never spans two experts); sixteen consumer warps
// multiply each stage by all of that expert's tokens, staged once per
// expert in shared memory, so an expert's weights leave HBM once however
// many tokens it has. A gate_up stage holds matching gate and up rows
// (rows i and I + i of the expert), so h = SiLU(g) * u is formed at once;
// the down stage multiplies by h.
//
// Device-side checks as in moe.cu: a token or slot id out of range sets
// BQD_MOE_BAD_PAIR in the status word and that pair's outputs are skipped; a
// CSR that is not monotone sets BQD_MOE_BAD_OFFSETS (reported by the gate_up
// kernel) and the affected experts are skipped. Every wait is bounded.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "gemv.h"
#include "host_util.h"
#include "stream.cuh"

namespace bqd {

// Device error word of the MoE stream kernels (kErrWaitTimeout).
__device__ unsigned int g_moe_stream_error = 0;

namespace {

constexpr int kCW = 16;                    // consumer warps
constexpr int kCT = kCW * kWarp;           // consumer threads
constexpr int kThreadsM = kCT + kWarp;     // + producer warp
constexpr int kMaxStagesM = 12;
constexpr int kStageTarget = 18 * 1024;    // bytes of weights per stage
constexpr int kMaxTok = 8;                 // tokens staged per pass over a stage
constexpr int kMaxC = 4;                   // tokens per compute pass (register budget)
constexpr int kSmemLimitM = 226 * 1024;
constexpr int kStatusBadOffsets = 1;
constexpr int kStatusBadPair = 2;

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Token-count class of a group of ng tokens (the compute loops are unrolled
// for 1, 2 or 4 tokens; staged rows past ng hold no token and their results
// are dropped).
__device__ __forceinline__ int tok_class(int ng) { return ng <= 1 ? 1 : (ng <= 2 ? 2 : 4); }

// Relative cost of one row of an expert with ntok tokens: the decode (2)
// plus the unrolled token passes (classes of at most kMaxC tokens).
__host__ __device__ __forceinline__ long long row_cost(int ntok)
{
    long long c = 2;
    for (int n0 = 0; n0 < ntok; n0 += kMaxC) {
        const int nt = ntok - n0 < kMaxC ? ntok - n0 : kMaxC;
        c += nt <= 1 ? 1 : (nt <= 2 ? 2 : 4);
    }
    return c;
}

// Bytes of the per-CTA tables in shared memory (offsets, active experts,
// cumulative row costs), rounded up to 128.
__host__ __device__ __forceinline__ int table_bytes(int E) { return (16 * E + 12 + 127) & ~127; }

// Activations in shared memory, fp32 per token: chunk c of 32 elements is
// 128 bytes, its 16-byte piece p (4 elements) at slot p ^ (c & 7), so lanes
// that read the same piece of consecutive chunks hit distinct banks.
__device__ __forceinline__ int xf_index(int c, int p) { return c * 32 + ((p ^ (c & 7)) << 2); }

// The active experts (non-empty segment) in increasing order into act[],
// their count into *n_act, and cum[a] = sum over active experts before a of
// R * row_cost(tokens). offsets[] is read once into shared memory; segment
// bounds are clamped to [0, P] so that a malformed list cannot send a later
// access out of range.
__device__ void list_active_experts(const int32_t* __restrict__ offsets, int E, int P, int R, int* off_s, int* act,
                                    long long* cum, int* n_act)
{
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        int v = offsets[e];
        off_s[e] = v < 0 ? 0 : (v > P ? P : v);
    }
    __syncthreads();
    if (threadIdx.x < kWarp) {
        const int lane = threadIdx.x;
        int base = 0;
        for (int e0 = 0; e0 < E; e0 += kWarp) {
            const int e = e0 + lane;
            const bool on = e < E && off_s[e + 1] > off_s[e];
            const unsigned m = __ballot_sync(0xFFFFFFFFu, on);
            if (on) act[base + __popc(m & ((1u << lane) - 1u))] = e;
            base += __popc(m);
        }
        __syncwarp();
        // cumulative costs: each lane a contiguous run of active experts
        const int per = (base + kWarp - 1) / kWarp, a0 = lane * per;
        long long run = 0;
        for (int a = a0; a < a0 + per && a < base; ++a) run += static_cast<long long>(R) * row_cost(off_s[act[a] + 1] - off_s[act[a]]);
        long long incl = run;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const long long v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        long long c = incl - run;
        for (int a = a0; a < a0 + per && a < base; ++a) {
            cum[a] = c;
            c += static_cast<long long>(R) * row_cost(off_s[act[a] + 1] - off_s[act[a]]);
        }
        if (lane == kWarp - 1) cum[base] = incl;
        if (lane == 0) *n_act = base;
    }
    __syncthreads();
}

// Row (a * R + row within expert a) of the virtual row space at cumulative
// cost wpos: monotone in wpos, so consecutive CTAs get adjacent ranges.
__device__ int weighted_row(long long wpos, const long long* cum, int nact, int R)
{
    if (nact == 0 || wpos >= cum[nact]) return nact * R;
    int lo = 0, hi = nact - 1;  // largest a with cum[a] <= wpos
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (cum[mid] <= wpos) lo = mid;
        else hi = mid - 1;
    }
    const long long per_row = (cum[lo + 1] - cum[lo]) / R;
    long long row = (wpos - cum[lo]) / per_row;
    if (row > R) row = R;
    return lo * R + static_cast<int>(row);
}

// Walk of one CTA through its rows [r_lo, r_hi) of the virtual row space
// (R rows per active expert), `rs` rows at most per stage.
struct Walk {
    int cur, r_hi, R, rs;
    __device__ bool next(int& a, int& off, int& rows)
    {
        if (cur >= r_hi) return false;
        a = cur / R;
        off = cur - a * R;
        rows = R - off;
        if (rows > rs) rows = rs;
        if (rows > r_hi - cur) rows = r_hi - cur;
        cur += rows;
        return true;
    }
};

// One (gate, up) row pair of a stage against NT staged fp32 tokens: this
// lane's partial sums (chunks lane, lane + 32, ...) into gsum[n], usum[n],
// block scales applied, tensor scale not. Elements are widened E2M1 -> f16
// -> fp32 and multiplied by packed fp32 FMAs; every product is exact in
// fp32 (11 x 8 significant bits).
template <int NT>
__device__ __forceinline__ void gu_pair(const unsigned char* cg, const unsigned char* cu, const unsigned char* sg,
                                        const unsigned char* su, const float* xs, int H, float (&gsum)[kMaxC],
                                        float (&usum)[kMaxC])
{
    const int lane = threadIdx.x % kWarp;
#pragma unroll
    for (int n = 0; n < NT; ++n) gsum[n] = usum[n] = 0.f;
    for (int c = lane; c < H / 32; c += kWarp) {
        const uint4 wg = *reinterpret_cast<const uint4*>(cg + 16 * c);
        const uint4 wu = *reinterpret_cast<const uint4*>(cu + 16 * c);
        const float2 scg = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(sg + 2 * c));
        const float2 scu = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(su + 2 * c));
        const uint32_t wgv[4] = {wg.x, wg.y, wg.z, wg.w}, wuv[4] = {wu.x, wu.y, wu.z, wu.w};
#pragma unroll
        for (int b = 0; b < 2; ++b) {  // 16-element blocks of the chunk
            float2 g2[2][NT], u2[2][NT];  // one accumulator pair per word: two short chains
#pragma unroll
            for (int n = 0; n < NT; ++n) g2[0][n] = g2[1][n] = u2[0][n] = u2[1][n] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int wi = 2 * b + j;  // elements 8wi .. 8wi+7 = activation pieces 2wi, 2wi+1
                uint32_t hg[4], hu[4];
                e2m1x8_to_f16x2(wgv[wi], hg);
                e2m1x8_to_f16x2(wuv[wi], hu);
                float2 fg[4], fu[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    fg[q] = f16x2_to_float2(hg[q]);
                    fu[q] = f16x2_to_float2(hu[q]);
                }
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const float4 x0 = *reinterpret_cast<const float4*>(xs + n * H + xf_index(c, 2 * wi));
                    const float4 x1 = *reinterpret_cast<const float4*>(xs + n * H + xf_index(c, 2 * wi + 1));
                    const float2 xv[4] = {make_float2(x0.x, x0.y), make_float2(x0.z, x0.w), make_float2(x1.x, x1.y),
                                          make_float2(x1.z, x1.w)};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        g2[j][n] = __ffma2_rn(fg[q], xv[q], g2[j][n]);
                        u2[j][n] = __ffma2_rn(fu[q], xv[q], u2[j][n]);
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const float gb = (g2[0][n].x + g2[0][n].y) + (g2[1][n].x + g2[1][n].y);
                const float ub = (u2[0][n].x + u2[0][n].y) + (u2[1][n].x + u2[1][n].y);
                gsum[n] = fmaf(b ? scg.y : scg.x, gb, gsum[n]);
                usum[n] = fmaf(b ? scu.y : scu.x, ub, usum[n]);
            }
        }
    }
}

// One row of a down stage against NT staged fp32 tokens (lanes gl, gl + lg,
// ... of the row's chunks): partial sums into acc[n], block scales applied.
template <int NT>
__device__ __forceinline__ void dn_row(const unsigned char* cr, const unsigned char* sr, const float* hs, int I,
                                       int gl, int lg, float (&acc)[kMaxC])
{
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n] = 0.f;
    for (int c = gl; c < I / 32; c += lg) {
        const uint4 w = *reinterpret_cast<const uint4*>(cr + 16 * c);
        const float2 sc = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(sr + 2 * c));
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float2 a2[2][NT];  // one accumulator pair per word: two short chains
#pragma unroll
            for (int n = 0; n < NT; ++n) a2[0][n] = a2[1][n] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int wi = 2 * b + j;  // elements 8wi .. 8wi+7 = h pieces 2wi, 2wi+1
                uint32_t hw[4];
                e2m1x8_to_f16x2(wv[wi], hw);
                const float2 f0 = f16x2_to_float2(hw[0]), f1 = f16x2_to_float2(hw[1]);
                const float2 f2 = f16x2_to_float2(hw[2]), f3 = f16x2_to_float2(hw[3]);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const float4 h0 = *reinterpret_cast<const float4*>(hs + n * I + xf_index(c, 2 * wi));
                    const float4 h1 = *reinterpret_cast<const float4*>(hs + n * I + xf_index(c, 2 * wi + 1));
                    a2[j][n] = __ffma2_rn(f0, make_float2(h0.x, h0.y), a2[j][n]);
                    a2[j][n] = __ffma2_rn(f1, make_float2(h0.z, h0.w), a2[j][n]);
                    a2[j][n] = __ffma2_rn(f2, make_float2(h1.x, h1.y), a2[j][n]);
                    a2[j][n] = __ffma2_rn(f3, make_float2(h1.z, h1.w), a2[j][n]);
                }
            }
#pragma unroll
            for (int n = 0; n < NT; ++n)
                acc[n] = fmaf(b ? sc.y : sc.x, (a2[0][n].x + a2[0][n].y) + (a2[1][n].x + a2[1][n].y), acc[n]);
        }
    }
}

// ------------------------------------------------------------------ gate_up
// Stage layout: [gate codes rsp x cp][up codes rsp x cp][gate scales rsp x
// sp][up scales rsp x sp], cp = H/2, sp = H/16; rsp row pairs at most.
__global__ void __launch_bounds__(kThreadsM, 1)
    moe_gu_stream_kernel(const uint8_t* __restrict__ gu_codes, const uint8_t* __restrict__ gu_scales,
                         const float* __restrict__ gu_ts, const uint16_t* __restrict__ x,
                         const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_token, MoeWorkspace ws,
                         int E, int H, int I, int T, int topk, int rsp, int ns)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kMaxStagesM], empty[kMaxStagesM];
    __shared__ int s_nact;
    const int P = T * topk;
    const int64_t cp = H / 2, sp = H / 16;
    const int64_t stage_bytes = 2 * rsp * (cp + sp);
    int* off_s = reinterpret_cast<int*>(smem);                               // [E + 1]
    int* act = off_s + (E + 1);                                                // [E]
    long long* cum = reinterpret_cast<long long*>(smem + ((8 * E + 4 + 7) & ~7));  // [E + 1]
    float* xs = reinterpret_cast<float*>(smem + table_bytes(E));              // [kMaxTok][H] fp32
    unsigned char* ring = reinterpret_cast<unsigned char*>(xs) + static_cast<size_t>(kMaxTok) * H * 4;

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_barrier_init();
    }
    pdl_wait();  // the list and activations may come from the previous kernel
    if (blockIdx.x == 0) {
        // CSR check, and the per-(token, slot) counters the down kernel fills
        bool bad = false;
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            if (offsets[e + 1] < offsets[e]) bad = true;
        if (threadIdx.x == 0 && (offsets[0] != 0 || offsets[E] != P)) bad = true;
        if (bad) atomicOr(ws.status, kStatusBadOffsets);
        for (int i = threadIdx.x; i < P; i += blockDim.x) {
            ws.count[i] = 0;
            ws.wts[i] = 0.f;
        }
    }
    list_active_experts(offsets, E, P, I, off_s, act, cum, &s_nact);
    const int nact = s_nact;
    // equal shares of the total cost, not of the rows
    const long long W = cum[nact];
    Walk walk{weighted_row(W * blockIdx.x / gridDim.x, cum, nact, I),
              weighted_row(W * (blockIdx.x + 1) / gridDim.x, cum, nact, I), I, rsp};

    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            int a, off, rows, t = 0;
            while (walk.next(a, off, rows)) {
                const int slot = t % ns;
                if (t >= ns && ok) ok = mbar_wait(&empty[slot], static_cast<uint32_t>(((t / ns) - 1) & 1),
                                                  &g_moe_stream_error);
                const int e = act[a];
                const uint8_t* ce = gu_codes + static_cast<int64_t>(e) * 2 * I * cp;
                const uint8_t* se = gu_scales + static_cast<int64_t>(e) * 2 * I * sp;
                unsigned char* st = ring + slot * stage_bytes;
                const uint32_t cb = static_cast<uint32_t>(rows * cp), sb = static_cast<uint32_t>(rows * sp);
                mbar_arrive_expect_tx(&full[slot], 2 * (cb + sb));
                bulk_g2s(st, ce + off * cp, cb, &full[slot]);
                bulk_g2s(st + rsp * cp, ce + (I + off) * cp, cb, &full[slot]);
                bulk_g2s(st + 2 * rsp * cp, se + off * sp, sb, &full[slot]);
                bulk_g2s(st + 2 * rsp * cp + rsp * sp, se + (I + off) * sp, sb, &full[slot]);
                ++t;
            }
            const int first = t > ns ? t - ns : 0;  // every copy lands before the CTA exits
            for (int u = first; u < t && ok; ++u)
                ok = mbar_wait(&full[u % ns], static_cast<uint32_t>((u / ns) & 1), &g_moe_stream_error);
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int cw = warp - 1, ctid = threadIdx.x - kWarp;
    int staged_a = -1, staged_g0 = -1;
    bool ok = true;
    int a, off, rows, t = 0;
    while (walk.next(a, off, rows)) {
        const int slot = t % ns;
        const int e = act[a];
        const int p0 = off_s[e], p1 = off_s[e + 1];
        const float ts = gu_ts[e];
        if (ok) ok = mbar_wait_warp(&full[slot], static_cast<uint32_t>((t / ns) & 1), &g_moe_stream_error);
        const unsigned char* st = ring + slot * stage_bytes;
        for (int g0 = p0; g0 < p1; g0 += kMaxTok) {
            const int ng = p1 - g0 < kMaxTok ? p1 - g0 : kMaxTok;
            if (staged_a != a || staged_g0 != g0) {
                // restage the tokens g0 .. g0+ng-1 of this expert as fp32
                named_sync(1, kCT);
                for (int i = ctid; i < ng * (H / 8); i += kCT) {
                    const int n = i / (H / 8), v = i - n * (H / 8);
                    const int tok = pair_token[g0 + n];
                    uint4 u = make_uint4(0u, 0u, 0u, 0u);
                    if (tok >= 0 && tok < T)
                        u = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(tok) * H + 8 * v);
                    else if (v == 0)
                        atomicOr(ws.status, kStatusBadPair);
                    // 8 elements = two fp32 pieces of chunk v / 4
                    const int c = v >> 2, p = 2 * (v & 3);
                    *reinterpret_cast<float4*>(xs + n * H + xf_index(c, p)) =
                        make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
                    *reinterpret_cast<float4*>(xs + n * H + xf_index(c, p + 1)) =
                        make_float4(bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w));
                }
                named_sync(1, kCT);
                staged_a = a;
                staged_g0 = g0;
            }
            for (int pr = cw; pr < rows; pr += kCW) {
                const unsigned char* cg = st + pr * cp;
                const unsigned char* cu = st + rsp * cp + pr * cp;
                const unsigned char* sg = st + 2 * rsp * cp + pr * sp;
                const unsigned char* su = st + 2 * rsp * cp + rsp * sp + pr * sp;
                for (int n0 = 0; n0 < ng; n0 += kMaxC) {
                    const int nt = ng - n0 < kMaxC ? ng - n0 : kMaxC;
                    const float* xn = xs + n0 * H;
                    float gsum[kMaxC], usum[kMaxC];
                    switch (tok_class(nt)) {
                        case 1: gu_pair<1>(cg, cu, sg, su, xn, H, gsum, usum); break;
                        case 2: gu_pair<2>(cg, cu, sg, su, xn, H, gsum, usum); break;
                        default: gu_pair<4>(cg, cu, sg, su, xn, H, gsum, usum); break;
                    }
#pragma unroll
                    for (int n = 0; n < kMaxC; ++n) {
                        if (n < nt) {
                            const float gv = warp_sum(gsum[n]) * ts;
                            const float uv = warp_sum(usum[n]) * ts;
                            if (lane == 0 && ok)
                                ws.h[static_cast<int64_t>(g0 + n0 + n) * I + off + pr] = gv / (1.0f + expf(-gv)) * uv;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        ++t;
    }
    pdl_trigger();
}

// ------------------------------------------------------------------ down
// Stage layout: [codes rs x cp][scales rs x sp], cp = I/2, sp = I/16.
__global__ void __launch_bounds__(kThreadsM, 1)
    moe_dn_stream_kernel(const uint8_t* __restrict__ dn_codes, const uint8_t* __restrict__ dn_scales,
                         const float* __restrict__ dn_ts, const int32_t* __restrict__ offsets,
                         const int32_t* __restrict__ pair_token, const float* __restrict__ pair_weight,
                         const int32_t* __restrict__ pair_slot, MoeWorkspace ws, int E, int H, int I, int T, int topk,
                         int rs, int ns)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kMaxStagesM], empty[kMaxStagesM];
    __shared__ int s_nact;
    __shared__ int s_flat[kMaxTok];  // token * topk + slot of each staged pair, -1 if invalid
    const int P = T * topk;
    const int64_t cp = I / 2, sp = I / 16;
    const int64_t stage_bytes = rs * (cp + sp);
    int* off_s = reinterpret_cast<int*>(smem);
    int* act = off_s + (E + 1);
    long long* cum = reinterpret_cast<long long*>(smem + ((8 * E + 4 + 7) & ~7));
    float* hs = reinterpret_cast<float*>(smem + table_bytes(E));  // [kMaxTok][I] fp32
    unsigned char* ring = reinterpret_cast<unsigned char*>(hs) + static_cast<size_t>(kMaxTok) * I * 4;

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_barrier_init();
    }
    pdl_wait();  // h, the counters and the list come from the previous kernels
    list_active_experts(offsets, E, P, H, off_s, act, cum, &s_nact);
    const int nact = s_nact;
    const long long W = cum[nact];
    Walk walk{weighted_row(W * blockIdx.x / gridDim.x, cum, nact, H),
              weighted_row(W * (blockIdx.x + 1) / gridDim.x, cum, nact, H), H, rs};

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            int a, off, rows, t = 0;
            while (walk.next(a, off, rows)) {
                const int slot = t % ns;
                if (t >= ns && ok) ok = mbar_wait(&empty[slot], static_cast<uint32_t>(((t / ns) - 1) & 1),
                                                  &g_moe_stream_error);
                const int e = act[a];
                const uint8_t* ce = dn_codes + static_cast<int64_t>(e) * H * cp;
                const uint8_t* se = dn_scales + static_cast<int64_t>(e) * H * sp;
                unsigned char* st = ring + slot * stage_bytes;
                const uint32_t cb = static_cast<uint32_t>(rows * cp), sb = static_cast<uint32_t>(rows * sp);
                mbar_arrive_expect_tx(&full[slot], cb + sb);
                bulk_g2s(st, ce + off * cp, cb, &full[slot]);
                bulk_g2s(st + rs * cp, se + off * sp, sb, &full[slot]);
                ++t;
            }
            const int first = t > ns ? t - ns : 0;
            for (int u = first; u < t && ok; ++u)
                ok = mbar_wait(&full[u % ns], static_cast<uint32_t>((u / ns) & 1), &g_moe_stream_error);
        }
        return;
    }

    const int cw = warp - 1, ctid = threadIdx.x - kWarp;
    const int nch = I / 32;  // chunks per row (8 .. 128)
    int lg = kWarp;          // lanes per row: the largest power of two <= nch / 2, at most 32
    while (lg > 1 && 2 * lg > nch) lg >>= 1;
    const int rpp = kWarp / lg;                // rows per warp pass
    const int sub = lane / lg, gl = lane % lg;
    int staged_a = -1, staged_g0 = -1;
    bool ok = true;
    int a, off, rows, t = 0;
    while (walk.next(a, off, rows)) {
        const int slot = t % ns;
        const int e = act[a];
        const int p0 = off_s[e], p1 = off_s[e + 1];
        const float ts = dn_ts[e];
        if (ok) ok = mbar_wait_warp(&full[slot], static_cast<uint32_t>((t / ns) & 1), &g_moe_stream_error);
        const unsigned char* st = ring + slot * stage_bytes;
        for (int g0 = p0; g0 < p1; g0 += kMaxTok) {
            const int ng = p1 - g0 < kMaxTok ? p1 - g0 : kMaxTok;
            if (staged_a != a || staged_g0 != g0) {
                named_sync(1, kCT);
                if (ctid < kMaxTok) {
                    int flat = -1;
                    if (ctid < ng) {
                        const int tok = pair_token[g0 + ctid], s = pair_slot[g0 + ctid];
                        if (tok >= 0 && tok < T && s >= 0 && s < topk) {
                            flat = tok * topk + s;
                            if (off == 0) {  // the CTA holding the expert's first row records the pair once
                                ws.wts[flat] = pair_weight[g0 + ctid];
                                atomicAdd(ws.count + flat, 1);
                            }
                        } else {
                            atomicOr(ws.status, kStatusBadPair);
                        }
                    }
                    s_flat[ctid] = flat;
                }
                for (int i = ctid; i < ng * (I / 4); i += kCT) {
                    const int n = i / (I / 4), v = i - n * (I / 4);
                    const float4 hv = reinterpret_cast<const float4*>(ws.h + static_cast<int64_t>(g0 + n) * I)[v];
                    *reinterpret_cast<float4*>(hs + n * I + xf_index(v >> 3, v & 7)) = hv;
                }
                named_sync(1, kCT);
                staged_a = a;
                staged_g0 = g0;
            }
            for (int rb = cw * rpp; rb < rows; rb += kCW * rpp) {
                const int r = rb + sub;
                const bool live = r < rows;
                const int rr = live ? r : rb;  // lanes past the last row repeat a valid one
                const unsigned char* cr = st + rr * cp;
                const unsigned char* sr = st + rs * cp + rr * sp;
                for (int n0 = 0; n0 < ng; n0 += kMaxC) {
                    const int nt = ng - n0 < kMaxC ? ng - n0 : kMaxC;
                    float acc[kMaxC];
                    switch (tok_class(nt)) {
                        case 1: dn_row<1>(cr, sr, hs + n0 * I, I, gl, lg, acc); break;
                        case 2: dn_row<2>(cr, sr, hs + n0 * I, I, gl, lg, acc); break;
                        default: dn_row<4>(cr, sr, hs + n0 * I, I, gl, lg, acc); break;
                    }
#pragma unroll
                    for (int n = 0; n < kMaxC; ++n) {
                        if (n < nt) {
                            float v = acc[n];
                            for (int o = lg / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                            const int flat = s_flat[n0 + n];
                            if (gl == 0 && live && flat >= 0 && ok)
                                ws.part[static_cast<int64_t>(flat) * H + off + r] = v * ts;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        ++t;
    }
    pdl_trigger();
}

size_t moe_stream_smem(int E, int64_t act_bytes, int64_t stage_bytes, int ns)
{
    return static_cast<size_t>(table_bytes(E) + act_bytes + stage_bytes * ns);
}

}  // namespace

bool moe_stream_supported(int E, int H, int I)
{
    // row pitches of codes and scales in multiples of 16 bytes; the ring and
    // the staged activations fit in shared memory
    if (H % 256 != 0 || I % 256 != 0 || H > 8192 || I > 4096) return false;
    const size_t a = moe_stream_smem(E, static_cast<int64_t>(kMaxTok) * H * 4, 2 * (H / 2 + H / 16), 3);
    const size_t b = moe_stream_smem(E, static_cast<int64_t>(kMaxTok) * I * 4, I / 2 + I / 16, 3);
    return a <= static_cast<size_t>(kSmemLimitM) && b <= static_cast<size_t>(kSmemLimitM);
}

cudaError_t launch_moe_stream_layer(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                                    const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts,
                                    const uint16_t* x, const int32_t* offsets, const int32_t* pair_token,
                                    const float* pair_weight, const int32_t* pair_slot, const MoeWorkspace& ws, int E,
                                    int H, int I, int T, int topk, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const DevInfo di = dev_info(dev);
    const int limit = di.max_smem_optin < kSmemLimitM ? di.max_smem_optin : kSmemLimitM;
    const bool pdl = (launch_flags() & kLaunchPdl) != 0;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    {  // gate_up
        // one row pair per consumer warp per stage
        const int64_t pair_bytes = 2 * (H / 2 + H / 16);
        int rsp = static_cast<int>(2 * kStageTarget / pair_bytes);
        if (rsp < 1) rsp = 1;
        if (rsp > kCW) rsp = kCW;
        const int64_t stage = rsp * pair_bytes;
        const int64_t actb = static_cast<int64_t>(kMaxTok) * H * 4;
        int ns = static_cast<int>((limit - static_cast<int64_t>(moe_stream_smem(E, actb, 0, 0))) / stage);
        if (ns > kMaxStagesM) ns = kMaxStagesM;
        if (ns < 2) return cudaErrorInvalidValue;
        const size_t smem = moe_stream_smem(E, actb, stage, ns);
        static OccCache occ;
        blocks_per_sm(occ, reinterpret_cast<const void*>(moe_gu_stream_kernel), dev, kThreadsM, smem);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(di.sms));
        cfg.blockDim = dim3(kThreadsM);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        err = cudaLaunchKernelEx(&cfg, moe_gu_stream_kernel, gu_codes, gu_scales, gu_ts, x, offsets, pair_token, ws,
                                 E, H, I, T, topk, rsp, ns);
        if (err != cudaSuccess) return err;
    }
    {  // down
        const int64_t row_bytes = I / 2 + I / 16;
        int rs = static_cast<int>(kStageTarget / row_bytes);
        if (rs < 1) rs = 1;
        if (rs > 128) rs = 128;
        const int64_t stage = rs * row_bytes;
        const int64_t actb = static_cast<int64_t>(kMaxTok) * I * 4;
        int ns = static_cast<int>((limit - static_cast<int64_t>(moe_stream_smem(E, actb, 0, 0))) / stage);
        if (ns > kMaxStagesM) ns = kMaxStagesM;
        if (ns < 2) return cudaErrorInvalidValue;
        const size_t smem = moe_stream_smem(E, actb, stage, ns);
        static OccCache occ;
        blocks_per_sm(occ, reinterpret_cast<const void*>(moe_dn_stream_kernel), dev, kThreadsM, smem);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(di.sms));
        cfg.blockDim = dim3(kThreadsM);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        err = cudaLaunchKernelEx(&cfg, moe_dn_stream_kernel, dn_codes, dn_scales, dn_ts, offsets, pair_token,
                                 pair_weight, pair_slot, ws, E, H, I, T, topk, rs, ns);
    }
    return err;
}

cudaError_t read_and_clear_moe_stream_error(unsigned int* out)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_moe_stream_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *out = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_moe_stream_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace bqd
