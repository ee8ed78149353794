// moe_small.cu -- the routed MoE layer for decode and verify batches (T <= 16
// tokens, T * topk <= 128 routed pairs): two kernels, each a GEMV over
// gathered rows.
//
// What is computed is the MoE layer of moe.cu ("robertbfuentes7-cloud/bw24"
// README, MoE bullet: routed tokens batched expert-major, each selected
// expert's weights decoded once for all of its tokens):
//   g = W_gu[e][0:I] . x_t,  u = W_gu[e][I:2I] . x_t,  h = SiLU(g) * u,
//   y_t = sum over slots s of w_{t,s} * ts_dn[e_{t,s}] * (W_dn[e_{t,s}] . h_{t,s}).
//
// With so few tokens each SM streams only tens of kilobytes per projection,
// so the layer is latency-bound. The two kernels are built like the direct
// N = 1 GEMV (gemv_direct.cu): warps own contiguous row ranges, rows are
// read with coalesced 16-byte loads into a register ring whose slots and
// offsets are compile-time constants, activations sit in shared memory.
//  * Routing, when the layer is given router logits (moe_layer), is done by
//    every CTA of both kernels for itself (route_token, the router's own
//    code, so the experts and weights are those moe_route_topk picks): no
//    route kernel and no list in global memory.
//  * Gate_up: the rows of all active experts (2I each: gate then up) form one
//    row space (an expert with more than four tokens appears once per group
//    of at most four); each row is dotted with the group's tokens,
//    staged once per CTA as exactly prescaled f16 with mixed-precision FMAs;
//    g and u of every (pair, row) go to the workspace.
//  * Down with the combine folded in: h = SiLU(g) * u is formed while it is
//    staged in shared memory, already multiplied by its pair's routing weight
//    and down tensor scale (h' = w * ts * h); output (t, j) is then one dot
//    product of length topk * I between h'_t (the token's slots side by side)
//    and row j of each of its experts, gathered: no partial outputs and no
//    combine kernel. Its weight loads are issued before it waits for the
//    gate_up kernel (programmatic dependent launch).
// Results are deterministic. Caller-supplied lists are checked as in moe.cu
// (status bits; never a fault).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "gemv.h"
#include "host_util.h"
#include "moe_route.cuh"

namespace bqd {

namespace {

constexpr int kTh = 768;            // threads per CTA (24 warps), one CTA per SM
constexpr int kWp = kTh / kWarp;
constexpr int kMaxT = 16;           // tokens
constexpr int kMaxP = 128;          // routed (token, slot) pairs
constexpr int kMaxE = 512;          // experts
constexpr int kDepth = 2;           // 32-element chunks in flight per lane
constexpr int kStatusBadOffsets = 1;
constexpr int kStatusBadPair = 2;
constexpr int kStatusCoverage = 4;

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Two fp32 accumulators += (lo, hi) f16 halves of w2 times those of x2
// (exact products, one fp32 rounding each).
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

// f16 (or raw bf16) activations: 32-element chunks of 64 bytes, 16-byte piece
// p of chunk c at slot p ^ ((c >> 1) & 3) (lanes reading the same piece of
// consecutive chunks hit distinct banks).
__device__ __forceinline__ int xh_index(int c, int p) { return c * 32 + ((p ^ ((c >> 1) & 3)) << 3); }
// fp32 rows (h): chunk c of 32 floats is 128 bytes, piece p at slot p ^ (c & 7).
__device__ __forceinline__ int xf_index(int c, int p) { return c * 32 + ((p ^ (c & 7)) << 2); }

// The routed pairs in expert-major order (experts ascending, tokens
// ascending inside an expert: the order moe_route_topk writes), in shared
// memory.
struct PairList {
    int n_act;               // token groups (find_active)
    int act[kMaxP];          // expert of group a (ascending)
    int act_p0[kMaxP + 1];   // its pairs [act_p0[a], act_p0[a+1]), at most kGroup
    int pe[kMaxP];           // expert of pair p
    int pt[kMaxP];           // token of pair p (-1: invalid pair, skipped)
    float pw[kMaxP];         // routing weight of pair p
    int qp[kMaxP];           // pair of (token, slot) q = t * topk + s (-1: none)
    int cover[kMaxP];        // times (token, slot) q appears
    int sel_e[kMaxP];        // routing scratch: expert of q
    float sel_w[kMaxP];      // routing scratch: weight of q
    int status;
};

// Token groups from pe[0..P) (expert-major): every expert's segment of pairs
// cut into groups of at most kGroup pairs (tokens), in order; the gate_up
// kernel reads a group's rows once for its tokens (an expert with more
// tokens is read once per group). By warp 0 in runs of 32 pairs. Needs a
// barrier before use.
constexpr int kGroup = 4;
__device__ void find_active(PairList& L, int P)
{
    if (threadIdx.x < kWarp) {
        const int lane = threadIdx.x;
        int base = 0, carry = 0;  // groups so far; segment start carried into the next run
        for (int p0 = 0; p0 < P; p0 += kWarp) {
            const int p = p0 + lane;
            const bool first = p < P && (p == 0 || L.pe[p - 1] != L.pe[p]);
            const unsigned m = __ballot_sync(0xFFFFFFFFu, first);
            const unsigned below = m & ((2u << lane) - 1u);  // segment starts at or before this lane
            const int seg = below ? p0 + 31 - __clz(below) : carry;
            const bool gstart = p < P && (p - seg) % kGroup == 0;
            const unsigned gm = __ballot_sync(0xFFFFFFFFu, gstart);
            if (gstart) {
                const int a = base + __popc(gm & ((1u << lane) - 1u));
                L.act[a] = L.pe[p];
                L.act_p0[a] = p;
            }
            base += __popc(gm);
            carry = __shfl_sync(0xFFFFFFFFu, seg, 31);
        }
        if (lane == 0) {
            L.n_act = base;
            L.act_p0[base] = P;
        }
    }
}

// Block-wide exclusive scan of one int per thread (kTh threads); s_scan
// holds kWp + 1 ints. Returns the exclusive prefix; *total gets the sum.
__device__ __forceinline__ int block_scan(int v, int* s_scan, int* total)
{
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    int incl = v;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == kWarp - 1) s_scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int t = lane < kWp ? s_scan[lane] : 0;
        int it = t;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, it, o);
            if (lane >= o) it += n;
        }
        if (lane < kWp) s_scan[lane] = it - t;
        if (lane == kWp - 1) s_scan[kWp] = it;
    }
    __syncthreads();
    const int r = s_scan[warp] + incl - v;
    *total = s_scan[kWp];
    __syncthreads();
    return r;
}

// Routing of T tokens from their logits, every CTA for itself (warp w routes
// token w), and the expert-major list of the routed pairs: every token sets
// its bit in the token masks of its experts; an exclusive scan over experts
// of (pairs, groups) gives each expert's first pair and first token group;
// a pair's place is its expert's first pair plus the number of lower tokens
// in the expert's mask (tokens ascending inside an expert, the order
// moe_route_topk writes). E <= kTh, T <= 32.
__device__ void route_in_cta(const float* __restrict__ logits, int T, int E, int topk, PairList& L,
                             uint32_t* s_mask, int* s_eoff, int* s_scan)
{
    const int P = T * topk;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    for (int e = threadIdx.x; e < E; e += kTh) s_mask[e] = 0u;
    for (int t = warp; t < T; t += kWp) {
        int e_s = 0;
        float w_s = 0.f;
        route_token(logits + static_cast<int64_t>(t) * E, E, topk, lane, &e_s, &w_s);
        if (lane < topk) {
            L.sel_e[t * topk + lane] = e_s;
            L.sel_w[t * topk + lane] = w_s;
        }
    }
    __syncthreads();
    if (threadIdx.x < P) atomicOr(&s_mask[L.sel_e[threadIdx.x]], 1u << (threadIdx.x / topk));
    if (threadIdx.x == 0) L.status = 0;
    __syncthreads();
    const int e = threadIdx.x;
    const int c = e < E ? __popc(s_mask[e]) : 0;  // pairs of expert e
    const int g = (c + kGroup - 1) / kGroup;       // its token groups
    int total = 0;
    const int excl = block_scan((g << 16) | c, s_scan, &total);
    if (c) {
        const int off = excl & 0xFFFF, goff = excl >> 16;
        s_eoff[e] = off;
        for (int k = 0; k < g; ++k) {
            L.act[goff + k] = e;
            L.act_p0[goff + k] = off + k * kGroup;
        }
    }
    if (threadIdx.x == 0) {
        L.n_act = total >> 16;
        L.act_p0[total >> 16] = P;
    }
    __syncthreads();
    if (threadIdx.x < P) {
        const int q = threadIdx.x, ee = L.sel_e[q], t = q / topk;
        const int r = s_eoff[ee] + __popc(s_mask[ee] & ((1u << t) - 1u));
        L.pe[r] = ee;
        L.pt[r] = t;
        L.pw[r] = L.sel_w[q];
        L.qp[q] = r;
    }
    __syncthreads();
}

// The caller's expert-major list, checked: a CSR that is not monotone or does
// not cover [0, P) sets BQD_MOE_BAD_OFFSETS (nothing is computed); a token or
// slot out of range sets BQD_MOE_BAD_PAIR (the pair is skipped); a (token,
// slot) present zero or several times sets BQD_MOE_COVERAGE.
__device__ void read_list(const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_token,
                          const float* __restrict__ pair_weight, const int32_t* __restrict__ pair_slot, int T, int E,
                          int topk, PairList& L)
{
    const int P = T * topk;
    __shared__ int s_bad;
    if (threadIdx.x == 0) {
        s_bad = (offsets[0] != 0 || offsets[E] != P) ? 1 : 0;
        L.status = 0;
    }
    if (threadIdx.x < P) {
        L.cover[threadIdx.x] = 0;
        L.qp[threadIdx.x] = -1;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kTh)
        if (offsets[e + 1] < offsets[e]) s_bad = 1;
    __syncthreads();
    if (s_bad) {
        if (threadIdx.x == 0) {
            L.status = kStatusBadOffsets;
            L.n_act = 0;
        }
        __syncthreads();
        return;
    }
    for (int e = threadIdx.x; e < E; e += kTh) {
        const int a = offsets[e], b = offsets[e + 1];
        for (int r = a; r < b; ++r) L.pe[r] = e;  // monotone, within [0, P]
    }
    if (threadIdx.x < P) {
        const int r = threadIdx.x;
        const int t = pair_token[r], s = pair_slot[r];
        if (t >= 0 && t < T && s >= 0 && s < topk) {
            L.pt[r] = t;
            L.pw[r] = pair_weight[r];
            atomicAdd(&L.cover[t * topk + s], 1);
            L.qp[t * topk + s] = r;
        } else {
            L.pt[r] = -1;
            atomicOr(&L.status, kStatusBadPair);
        }
    }
    __syncthreads();
    if (threadIdx.x < P && L.cover[threadIdx.x] != 1) {
        atomicOr(&L.status, kStatusCoverage);
        if (L.cover[threadIdx.x] == 0) L.qp[threadIdx.x] = -1;
    }
    find_active(L, P);
    __syncthreads();
}

// ------------------------------------------------------------------ items
struct Item {  // 32 elements of one NVFP4 row: 16 code bytes, two E4M3 scales
    uint4 c;
    uint32_t s;
};

__device__ __forceinline__ Item load_item(const uint8_t* c, const uint8_t* s)
{
    Item it;
    it.c = ld_stream_v4(c);
    it.s = ld_stream_u16(s);
    return it;
}

// One chunk of an expert row against its tokens (at most NT, ne of them,
// listed in tok[]): xc is this lane's chunk of token 0's staged activations
// (token t's start t * H elements later), sw the lane's swizzle. The chunk is
// decoded once for all tokens.
template <bool FAST, int NT>
__device__ __forceinline__ void gu_dot(const Item& it, const uint16_t* xc, int H, const int* tok, int ne, int sw,
                                       float (&acc)[NT])
{
    const float2 sc = e4m3x2_to_float2(it.s);
    const uint32_t words[4] = {it.c.x, it.c.y, it.c.z, it.c.w};
    uint32_t h[16];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t a[4];
        e2m1x8_to_f16x2(words[w], a);
#pragma unroll
        for (int q = 0; q < 4; ++q) h[4 * w + q] = a[q];
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        if (n < ne) {
            const int t = tok[n];
            if (t >= 0) {
                const uint16_t* xr = xc + t * H;
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int wi = 2 * b + j;
                        const uint4 xq = *reinterpret_cast<const uint4*>(xr + ((wi ^ sw) << 3));
                        const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if constexpr (FAST) {
                                fma_f16x2(h[4 * wi + q], xp[q], a0, a1);
                            } else {
                                const float2 wf = f16x2_to_float2(h[4 * wi + q]);
                                a0 = fmaf(wf.x, bf16_lo(xp[q]), a0);
                                a1 = fmaf(wf.y, bf16_hi(xp[q]), a1);
                            }
                        }
                    }
                    acc[n] = fmaf(b ? sc.y : sc.x, a0 + a1, acc[n]);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ gate_up
// Virtual row v of the gate_up row space: active expert a = v / (2I), row
// l = v % (2I) of its gate_up weight (gate rows first, then up rows).
// go[p][l] = the row's dot product with pair p's token, tensor scale and the
// token's prescale applied.
template <int CPL, int NT, bool FAST>
__device__ __forceinline__ void gu_rows(Item (&buf)[kDepth], const uint8_t* __restrict__ gu_codes,
                                        const uint8_t* __restrict__ gu_scales, const float* __restrict__ gu_ts,
                                        const uint16_t* xs, const int* sexp, const PairList& L, float* __restrict__ go,
                                        int H, int I, int v_lo, int v_hi, int lane)
{
    static_assert(CPL % kDepth == 0 || kDepth % CPL == 0, "ring depth must divide a row or be a multiple of one");
    constexpr int U = kDepth > CPL ? kDepth / CPL : 1;
    const int64_t cp = H / 2, sp = H / 16;
    const int sw = (lane >> 1) & 3;
    const int sh = __ffs(2 * I) - 1, lmask = 2 * I - 1;  // 2I is a power of two
    for (int v0 = v_lo; v0 < v_hi; v0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u;
            if (v < v_hi) {
                const int a = v >> sh, l = v & lmask;
                const int p0 = L.act_p0[a], ne = L.act_p0[a + 1] - p0;
                float acc[NT];
#pragma unroll
                for (int n = 0; n < NT; ++n) acc[n] = 0.f;
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    const int g = u * CPL + i;
                    const Item cur = buf[g % kDepth];
                    const int nr = (g + kDepth) / CPL, nc = (g + kDepth) % CPL;
                    const int vn = v0 + nr;
                    if (vn < v_hi) {
                        const int an = vn >> sh, ln = vn & lmask;
                        const int64_t row = static_cast<int64_t>(L.act[an]) * 2 * I + ln;
                        buf[g % kDepth] = load_item(gu_codes + row * cp + nc * 512 + lane * 16,
                                                    gu_scales + row * sp + nc * 64 + lane * 2);
                    }
                    gu_dot<FAST, NT>(cur, xs + lane * 32 + i * 1024, H, L.pt + p0, ne, sw, acc);
                    asm volatile("" ::: "memory");
                }
                const float ts = gu_ts[L.act[a]];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if (n < ne) {
                        const int t = L.pt[p0 + n];
                        const float sum = warp_sum(acc[n]);
                        if (lane == 0 && t >= 0) go[static_cast<int64_t>(p0 + n) * 2 * I + l] = ldexpf(sum * ts, sexp[t]);
                    }
                }
            }
        }
    }
}

// Dynamic shared memory: the activations, T * H f16 (or bf16).
template <int CPL, int NT>
__global__ void __launch_bounds__(kTh, 1)
    moe_small_gu_kernel(const float* __restrict__ logits, const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ pair_token, const float* __restrict__ pair_weight,
                        const int32_t* __restrict__ pair_slot, const uint8_t* __restrict__ gu_codes,
                        const uint8_t* __restrict__ gu_scales, const float* __restrict__ gu_ts,
                        const uint16_t* __restrict__ x, MoeWorkspace ws, int E, int I, int T, int topk)
{
    constexpr int H = 1024 * CPL;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ PairList L;
    __shared__ int s_emax[kMaxT], s_emin[kMaxT], s_sexp[kMaxT], s_flags;
    __shared__ uint32_t s_mask[kMaxE];
    __shared__ int s_eoff[kMaxE], s_scan[kWp + 1];
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
    float* go = ws.part;  // [P][2I] gate and up outputs

    if (threadIdx.x == 0) s_flags = 0;  // ordered before their use by the barriers of the routing
    if (threadIdx.x < kMaxT) {
        s_emax[threadIdx.x] = 0;
        s_emin[threadIdx.x] = INT_MAX;
    }
    pdl_wait();  // logits, the list and x may come from the previous kernel
    if (logits)
        route_in_cta(logits, T, E, topk, L, s_mask, s_eoff, s_scan);
    else
        read_list(offsets, pair_token, pair_weight, pair_slot, T, E, topk, L);
    pdl_trigger();
    // the compact list the down kernel reads: per (token, slot) q its pair
    // (bits 16..) and expert (bits 0..15), or -1, and its routing weight
    if (blockIdx.x == 0) {
        const int P = T * topk;
        if (threadIdx.x < P) {
            const int p = L.qp[threadIdx.x];
            ws.count[threadIdx.x] = p >= 0 && L.status != kStatusBadOffsets ? (p << 16) | L.pe[p] : -1;
            ws.wts[threadIdx.x] = p >= 0 ? L.pw[p] : 0.f;
        }
        if (threadIdx.x == 0) *ws.status = L.status;
    }

    // this warp's rows: an even split of all active experts' 2I rows
    const int nv = L.n_act * 2 * I;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWp + warp, nw = static_cast<int64_t>(gridDim.x) * kWp;
    const int v_lo = static_cast<int>(nv * gw / nw), v_hi = static_cast<int>(nv * (gw + 1) / nw);
    const int64_t cp = H / 2, sp = H / 16;
    Item buf[kDepth];
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
        const int v = v_lo + d / CPL;
        if (v < v_hi) {
            const int a = v >> (__ffs(2 * I) - 1), l = v & (2 * I - 1);
            const int64_t row = static_cast<int64_t>(L.act[a]) * 2 * I + l;
            buf[d] = load_item(gu_codes + row * cp + (d % CPL) * 512 + lane * 16,
                               gu_scales + row * sp + (d % CPL) * 64 + lane * 2);
        }
    }

    // each token's exponent range (bf16 biased exponents of its nonzero
    // elements): warp t scans token t (T <= kWp), loads issued eight at a time
    for (int t = warp; t < T; t += kWp) {
        int emax = 0, emin = INT_MAX, flags = 0;
        const uint32_t* xr = reinterpret_cast<const uint32_t*>(x + static_cast<int64_t>(t) * H);
#pragma unroll 8
        for (int i = lane; i < H / 2; i += kWarp) {
            const uint32_t vv = xr[i];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint32_t b = (vv >> (16 * hh)) & 0x7FFFu;
                const int e = static_cast<int>(b >> 7);
                if (b == 0) continue;
                if (e == 0 || e == 255) flags = 1;
                emax = max(emax, e);
                emin = min(emin, e);
            }
        }
        emax = __reduce_max_sync(0xFFFFFFFFu, emax);
        emin = __reduce_min_sync(0xFFFFFFFFu, emin);
        flags = __reduce_or_sync(0xFFFFFFFFu, flags);
        if (lane == 0) {
            s_emax[t] = emax;
            s_emin[t] = emin;
            if (flags) atomicOr(&s_flags, 1);
        }
    }
    __syncthreads();
    // f16 holds x * 2^-s exactly when every nonzero |x| of the token is within
    // 31 binades of its largest; the largest lands in [2^14, 2^15)
    if (threadIdx.x < T && s_emin[threadIdx.x] != INT_MAX && s_emax[threadIdx.x] - s_emin[threadIdx.x] > 31)
        atomicOr(&s_flags, 1);
    __syncthreads();
    const bool fast = s_flags == 0;
    if (threadIdx.x < kMaxT)
        s_sexp[threadIdx.x] = fast && threadIdx.x < T && s_emin[threadIdx.x] != INT_MAX
                                  ? s_emax[threadIdx.x] - 127 - 14
                                  : 0;
    __syncthreads();
    for (int i = threadIdx.x; i < T * (H / 8); i += kTh) {
        const int t = i / (H / 8), v = i - t * (H / 8);
        uint4 uu = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H)[v];
        if (fast) {
            const int se = s_sexp[t];
            const uint32_t w[4] = {uu.x, uu.y, uu.z, uu.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                __half2 hv = __floats2half2_rn(ldexpf(bf16_lo(w[q]), -se), ldexpf(bf16_hi(w[q]), -se));
                o[q] = *reinterpret_cast<uint32_t*>(&hv);
            }
            uu = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>(xs + t * H + xh_index(v / 4, v % 4)) = uu;
    }
    __syncthreads();
    if (fast)
        gu_rows<CPL, NT, true>(buf, gu_codes, gu_scales, gu_ts, xs, s_sexp, L, go, H, I, v_lo, v_hi, lane);
    else
        gu_rows<CPL, NT, false>(buf, gu_codes, gu_scales, gu_ts, xs, s_sexp, L, go, H, I, v_lo, v_hi, lane);
}

// ------------------------------------------------------------------ down + combine
// Output (t, j) is the dot product of h'_t = [h'_{t,0} .. h'_{t,topk-1}] (the
// token's slots side by side, K' = topk * I elements) with row j of each of
// its experts, gathered. Lane l takes the chunks l + 32 i (i < CPLD) of that
// gathered row: slot s = (l + 32 i) / CS (CS = I / 32 chunks per slot),
// chunk (l + 32 i) % CS = l % CS of the slot's expert row (CS divides 32).
__device__ __forceinline__ float dn_dot(const Item& it, const float* hc)
{
    const float2 sc = e4m3x2_to_float2(it.s);
    const uint32_t w[4] = {it.c.x, it.c.y, it.c.z, it.c.w};
    const int sw = (threadIdx.x & 31) & 7;  // fp32 chunks: piece p at slot p ^ (c & 7), c = lane + 32 i
    float acc = 0.f;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int wi = 2 * b + jj;  // elements 8 wi .. 8 wi + 7 = h' pieces 2 wi, 2 wi + 1
            uint32_t hw[4];
            e2m1x8_to_f16x2(w[wi], hw);
            const float4 h0 = *reinterpret_cast<const float4*>(hc + (((2 * wi) ^ sw) << 2));
            const float4 h1 = *reinterpret_cast<const float4*>(hc + (((2 * wi + 1) ^ sw) << 2));
            float2& a = jj ? a1 : a0;
            a = __ffma2_rn(f16x2_to_float2(hw[0]), make_float2(h0.x, h0.y), a);
            a = __ffma2_rn(f16x2_to_float2(hw[1]), make_float2(h0.z, h0.w), a);
            a = __ffma2_rn(f16x2_to_float2(hw[2]), make_float2(h1.x, h1.y), a);
            a = __ffma2_rn(f16x2_to_float2(hw[3]), make_float2(h1.z, h1.w), a);
        }
        acc = fmaf(b ? sc.y : sc.x, (a0.x + a0.y) + (a1.x + a1.y), acc);
    }
    return acc;
}

// Dynamic shared memory: h' of the tokens whose rows the CTA computes, topk
// * I fp32 per token (the token's slots side by side). The pair list comes
// from the gate_up kernel (workspace count and wts, one entry per (token,
// slot)): nothing is routed here.
template <int CPLD, int CS>
__global__ void __launch_bounds__(kTh, 1)
    moe_small_dn_kernel(const uint8_t* __restrict__ dn_codes, const uint8_t* __restrict__ dn_scales,
                        const float* __restrict__ dn_ts, float* __restrict__ y, MoeWorkspace ws, int H, int T,
                        int topk)
{
    constexpr int I = 32 * CS;
    constexpr int64_t cp = I / 2, sp = I / 16;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_eh[kMaxP];    // expert * H of (token, slot) q, -1 if missing
    __shared__ int s_p[kMaxP];     // its pair, -1 if missing
    __shared__ float s_sc[kMaxP];  // its routing weight times the expert's down tensor scale
    __shared__ int s_ok;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int P = T * topk, KC = topk * CS;  // chunks per gathered row
    float* hs = reinterpret_cast<float*>(smem);
    const float* go = ws.part;

    pdl_wait();  // the list, g and u come from the gate_up kernel; y may be read by earlier kernels
    if (threadIdx.x < P) {
        const int v = ws.count[threadIdx.x];
        const int e = v & 0xFFFF, p = v >> 16;
        s_eh[threadIdx.x] = v >= 0 ? e * H : -1;
        s_p[threadIdx.x] = v >= 0 ? p : -1;
        s_sc[threadIdx.x] = v >= 0 ? ws.wts[threadIdx.x] * dn_ts[e] : 0.f;
    }
    if (threadIdx.x == 0) s_ok = (*ws.status & kStatusBadOffsets) == 0;
    __syncthreads();
    const bool ok = s_ok != 0;

    // rows (t, j), t = r / H: an even split over the CTAs, then over the warps;
    // the CTA stages h' only for the tokens its rows belong to
    const int nr = ok ? T * H : 0;
    const int c_lo = static_cast<int>(static_cast<int64_t>(nr) * blockIdx.x / gridDim.x);
    const int c_hi = static_cast<int>(static_cast<int64_t>(nr) * (blockIdx.x + 1) / gridDim.x);
    const int t_first = c_lo / H, t_end = c_hi > c_lo ? (c_hi - 1) / H + 1 : t_first;  // tokens [t_first, t_end)
    const int r_lo = c_lo + static_cast<int>(static_cast<int64_t>(c_hi - c_lo) * warp / kWp);
    const int r_hi = c_lo + static_cast<int>(static_cast<int64_t>(c_hi - c_lo) * (warp + 1) / kWp);
    const int cc = lane % CS;
    const int hsh = __ffs(H) - 1;  // H is a power of two
    // the gathered row's expert rows for this lane's chunks, per token
    int eh[CPLD];
    int cur_t = -1;
    auto set_token = [&](int t) {
#pragma unroll
        for (int i = 0; i < CPLD; ++i) {
            const int c = lane + 32 * i;
            eh[i] = c < KC ? s_eh[t * topk + c / CS] : -1;
        }
        cur_t = t;
    };
    auto load_at = [&](int r, int i) -> Item {
        Item it;
        it.c = make_uint4(0u, 0u, 0u, 0u);
        it.s = 0u;
        const int t = r >> hsh, j = r & (H - 1);
        if (t != cur_t) set_token(t);
        if (eh[i] >= 0) it = load_item(dn_codes + static_cast<int64_t>(eh[i] + j) * cp + cc * 16,
                                       dn_scales + static_cast<int64_t>(eh[i] + j) * sp + cc * 2);
        return it;
    };
    static_assert(CPLD % kDepth == 0 || kDepth % CPLD == 0, "ring depth must divide a row or be a multiple of one");
    constexpr int U = kDepth > CPLD ? kDepth / CPLD : 1;
    Item buf[kDepth];
#pragma unroll
    for (int d = 0; d < kDepth; ++d)
        if (r_lo + d / CPLD < r_hi) buf[d] = load_at(r_lo + d / CPLD, d % CPLD);

    // h' = w * ts_dn * SiLU(g) * u of the CTA's tokens' (token, slot) pairs,
    // token-major; h itself also goes to the workspace (the same value from
    // every CTA that stages it)
    const int q0 = t_first * topk, nq = (t_end - t_first) * topk;
#pragma unroll 4
    for (int i = threadIdx.x; i < nq * I; i += kTh) {
        const int ql = i / I, k = i - ql * I, q = q0 + ql;
        const int p = s_p[q];
        float hv = 0.f;
        if (p >= 0) {
            const float g = go[static_cast<int64_t>(p) * 2 * I + k], u = go[static_cast<int64_t>(p) * 2 * I + I + k];
            const float h = g / (1.0f + expf(-g)) * u;
            ws.h[static_cast<int64_t>(p) * I + k] = h;
            hv = h * s_sc[q];
        }
        const int tl = ql / topk, c = (ql - tl * topk) * CS + k / 32;  // chunk of the token's gathered row
        hs[tl * KC * 32 + c * 32 + (((k / 4 % 8) ^ (c & 7)) << 2) + k % 4] = hv;
    }
    __syncthreads();

    for (int r0 = r_lo; r0 < r_hi; r0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u;
            if (r < r_hi) {
                const int t = r >> hsh;
                const float* hrow = hs + (t - t_first) * KC * 32;
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < CPLD; ++i) {
                    const int g = u * CPLD + i;
                    const Item it = buf[g % kDepth];
                    const int rn = r0 + (g + kDepth) / CPLD;
                    if (rn < r_hi) buf[g % kDepth] = load_at(rn, (g + kDepth) % CPLD);
                    const int c = lane + 32 * i;
                    if (c < KC) acc += dn_dot(it, hrow + c * 32);
                    asm volatile("" ::: "memory");
                }
                const float v = warp_sum(acc);
                if (lane == 0) y[r] = v;  // r = t * H + j
            }
        }
    }
    if (!ok)  // malformed CSR: outputs unspecified, written as zero
        for (int i = blockIdx.x * kTh + threadIdx.x; i < T * H; i += gridDim.x * kTh) y[i] = 0.f;
}

size_t small_smem(int64_t bytes) { return static_cast<size_t>(bytes); }

template <int CPL, int NT>
cudaError_t launch_gu(cudaLaunchConfig_t& cfg, int dev, const float* logits, const int32_t* offsets,
                      const int32_t* pair_token, const float* pair_weight, const int32_t* pair_slot,
                      const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts, const uint16_t* x,
                      const MoeWorkspace& ws, int E, int I, int T, int topk)
{
    auto kern = moe_small_gu_kernel<CPL, NT>;
    static OccCache occ;
    cfg.dynamicSmemBytes = small_smem(static_cast<int64_t>(T) * 1024 * CPL * 2);
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kTh, cfg.dynamicSmemBytes);
    return cudaLaunchKernelEx(&cfg, kern, logits, offsets, pair_token, pair_weight, pair_slot, gu_codes, gu_scales,
                              gu_ts, x, ws, E, I, T, topk);
}

template <int CPLD, int CS>
cudaError_t launch_dn(cudaLaunchConfig_t& cfg, int dev, const uint8_t* dn_codes, const uint8_t* dn_scales,
                      const float* dn_ts, float* y, const MoeWorkspace& ws, int H, int T, int topk)
{
    auto kern = moe_small_dn_kernel<CPLD, CS>;
    static OccCache occ;
    // a CTA's rows span at most rows_per_cta / H + 2 tokens
    const int64_t rows_per_cta = (static_cast<int64_t>(T) * H + cfg.gridDim.x - 1) / cfg.gridDim.x;
    int64_t tok = rows_per_cta / H + 2;
    if (tok > T) tok = T;
    cfg.dynamicSmemBytes = small_smem(tok * topk * 32 * CS * 4);
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kTh, cfg.dynamicSmemBytes);
    return cudaLaunchKernelEx(&cfg, kern, dn_codes, dn_scales, dn_ts, y, ws, H, T, topk);
}

}  // namespace

bool moe_small_supported(int E, int H, int I, int T, int topk)
{
    const bool h_ok = H == 1024 || H == 2048 || H == 4096 || H == 8192;
    const bool i_ok = I == 256 || I == 512 || I == 1024;
    // g and u of all pairs live in the workspace's partial-output area (needs H >= 2I);
    // a gathered down row is at most 8 * 1024 elements; the staged activations
    // (T * H f16) at most 64 KiB
    return T >= 1 && T <= kMaxT && T * topk <= kMaxP && topk <= kWarp && E >= 1 && E <= kMaxE && h_ok && i_ok &&
           H >= 2 * I && topk * I <= 8192 && T * H <= 32768;
}

cudaError_t launch_moe_small_layer(const float* logits, const uint8_t* gu_codes, const uint8_t* gu_scales,
                                   const float* gu_ts, const uint8_t* dn_codes, const uint8_t* dn_scales,
                                   const float* dn_ts, const uint16_t* x, const int32_t* offsets,
                                   const int32_t* pair_token, const float* pair_weight, const int32_t* pair_slot,
                                   float* y, const MoeWorkspace& ws, int E, int H, int I, int T, int topk,
                                   cudaStream_t stream)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int sms = dev_info(dev).sms;
    const bool pdl = (launch_flags() & kLaunchPdl) != 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(kTh);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;

    // a token group holds at most min(T, kGroup) pairs
    const int nt = T == 1 ? 1 : (T == 2 ? 2 : 4);
#define BQD_GU1(CPL_, NT_)                                                                                            \
    launch_gu<CPL_, NT_>(cfg, dev, logits, offsets, pair_token, pair_weight, pair_slot, gu_codes, gu_scales, gu_ts, x, \
                         ws, E, I, T, topk)
#define BQD_GU(CPL_) (nt == 1 ? BQD_GU1(CPL_, 1) : (nt == 2 ? BQD_GU1(CPL_, 2) : BQD_GU1(CPL_, 4)))
    switch (H) {
        case 1024: err = BQD_GU(1); break;
        case 2048: err = BQD_GU(2); break;
        case 4096: err = BQD_GU(4); break;
        default: err = BQD_GU(8); break;
    }
#undef BQD_GU
#undef BQD_GU1
    if (err != cudaSuccess) return err;
    // The down kernel always follows programmatically: it reads nothing that
    // the gate_up kernel writes before its griddepcontrol.wait.
    cfg.numAttrs = 1;
    const int kc = topk * (I / 32);  // chunks of a gathered down row
    const int cpld = kc <= 32 ? 1 : (kc <= 64 ? 2 : (kc <= 128 ? 4 : 8));
#define BQD_DN(CPLD_)                                                                                                 \
    (I == 256   ? launch_dn<CPLD_, 8>(cfg, dev, dn_codes, dn_scales, dn_ts, y, ws, H, T, topk)                        \
     : I == 512 ? launch_dn<CPLD_, 16>(cfg, dev, dn_codes, dn_scales, dn_ts, y, ws, H, T, topk)                       \
                : launch_dn<CPLD_, 32>(cfg, dev, dn_codes, dn_scales, dn_ts, y, ws, H, T, topk))
    switch (cpld) {
        case 1: return BQD_DN(1);
        case 2: return BQD_DN(2);
        case 4: return BQD_DN(4);
        default: return BQD_DN(8);
    }
#undef BQD_DN
}

}  // namespace bqd
