// moe_small.cu -- the routed MoE layer for a few tokens (T <= 4 tokens and
// T * topk <= 32 routed pairs): decode with one to four tokens in flight.
//
// What is computed is the MoE layer of moe.cu ("robertbfuentes7-cloud/bw24"
// README, MoE bullet: routed tokens batched expert-major, each selected
// expert's weights decoded once for all of its tokens):
//   g = W_gu[e][0:I] . x_t,  u = W_gu[e][I:2I] . x_t,  h = SiLU(g) * u,
//   y_t = sum over slots s = 0..topk-1, in order, of w_{t,s} * (W_dn[e_{t,s}] . h_{t,s}).
//
// With so few tokens each SM streams only tens of kilobytes per projection,
// so the layer is latency-bound; the design removes every step of the chain
// that the larger-batch path needs:
//  * Routing, when the layer is given router logits (moe_layer), is done by
//    every CTA of both kernels for itself (route_token_warp, the router's
//    own code, so the experts and weights are those moe_route_topk picks):
//    no route kernel and no list in global memory.
//  * Gate_up kernel: the rows (gate row i and up row I + i) of all active
//    experts form one row space split evenly over all warps of the grid;
//    every warp streams its rows with 16-byte loads kept four items deep in
//    registers; the activations are staged once per CTA as f16, each token
//    scaled by its own exact power of two, and multiplied in by mixed-
//    precision FMAs (exact products, fp32 sums), as in the N = 1 GEMV.
//  * Down kernel with the combine folded in: every warp owns output rows j
//    and, for each of them, walks the routed pairs in token-major slot
//    order, streams row j of the pair's expert and accumulates
//    y_t[j] = fma(w_{t,s}, d_{t,s}[j], y_t[j]) in slot order -- no partial
//    outputs in global memory and no combine kernel. Its weight loads are
//    issued before it waits for the gate_up kernel (programmatic dependent
//    launch), so they overlap that kernel.
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

constexpr int kTh = 256;            // threads per CTA (8 warps)
constexpr int kWp = kTh / kWarp;
constexpr int kMaxT = 4;            // tokens
constexpr int kMaxP = 32;           // routed (token, slot) pairs
constexpr int kMaxE = 512;          // experts
constexpr int kDepth = 4;           // items in flight per lane
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
    int n_act;               // active experts
    int act[kMaxP];          // active expert a (ascending)
    int act_p0[kMaxP + 1];   // its pairs [act_p0[a], act_p0[a+1])
    int pe[kMaxP];           // expert of pair p
    int pt[kMaxP];           // token of pair p (-1: invalid pair, skipped)
    float pw[kMaxP];         // routing weight of pair p
    float pts[kMaxP];        // down projection tensor scale of pair p's expert (down kernel)
    int qp[kMaxP];           // pair of (token, slot) q = t * topk + s (-1: none)
    int cover[kMaxP];        // times (token, slot) q appears
    int sel_e[kMaxP];        // routing scratch: expert of q
    float sel_w[kMaxP];      // routing scratch: weight of q
    int status;
};

// Active experts from pe[0..P) (expert-major). Needs a barrier before use.
__device__ void find_active(PairList& L, int P)
{
    if (threadIdx.x < kWarp) {
        const int lane = threadIdx.x;
        const bool first = lane < P && (lane == 0 || L.pe[lane - 1] != L.pe[lane]);
        const unsigned m = __ballot_sync(0xFFFFFFFFu, first);
        if (first) {
            const int a = __popc(m & ((1u << lane) - 1u));
            L.act[a] = L.pe[lane];
            L.act_p0[a] = lane;
        }
        if (lane == 0) {
            L.n_act = __popc(m);
            L.act_p0[__popc(m)] = P;
        }
    }
}

// Routing of T tokens from their logits, every CTA for itself (warp w
// routes tokens w, w + 8, ...).
__device__ void route_in_cta(const float* __restrict__ logits, int T, int E, int topk, PairList& L)
{
    const int P = T * topk;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
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
    // expert-major position of (token t, slot s): experts ascending, then tokens
    if (threadIdx.x < P) {
        const int q = threadIdx.x, e = L.sel_e[q], t = q / topk;
        int r = 0;
        for (int q2 = 0; q2 < P; ++q2) {
            const int e2 = L.sel_e[q2];
            r += (e2 < e || (e2 == e && q2 / topk < t)) ? 1 : 0;
        }
        L.pe[r] = e;
        L.pt[r] = t;
        L.pw[r] = L.sel_w[q];
        L.qp[q] = r;
    }
    if (threadIdx.x == 0) L.status = 0;
    __syncthreads();
    find_active(L, P);
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

// ------------------------------------------------------------------ gate_up
struct GuItem {
    uint4 g, u;     // 16 code bytes (32 elements) of the gate row and of the up row
    uint32_t sg, su;  // their two E4M3 block scales
};

template <bool FAST, int NT>
__device__ __forceinline__ void gu_item(const GuItem& it, const uint16_t* xs, int H, const PairList& L, int p0, int ne,
                                        int c, float (&g)[NT], float (&u)[NT])
{
    const float2 sg = e4m3x2_to_float2(it.sg), su = e4m3x2_to_float2(it.su);
    const uint32_t wg[4] = {it.g.x, it.g.y, it.g.z, it.g.w}, wu[4] = {it.u.x, it.u.y, it.u.z, it.u.w};
    uint32_t hg[16], hu[16];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t a[4], b[4];
        e2m1x8_to_f16x2(wg[w], a);
        e2m1x8_to_f16x2(wu[w], b);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            hg[4 * w + q] = a[q];
            hu[4 * w + q] = b[q];
        }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        if (n < ne) {
            const int t = L.pt[p0 + n];
            if (t >= 0) {
                const uint16_t* xr = xs + t * H;
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int wi = 2 * b + j;
                        const uint4 xq = *reinterpret_cast<const uint4*>(xr + xh_index(c, wi));
                        const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if constexpr (FAST) {
                                fma_f16x2(hg[4 * wi + q], xp[q], g0, g1);
                                fma_f16x2(hu[4 * wi + q], xp[q], u0, u1);
                            } else {
                                const float2 fg = f16x2_to_float2(hg[4 * wi + q]);
                                const float2 fu = f16x2_to_float2(hu[4 * wi + q]);
                                g0 = fmaf(fg.x, bf16_lo(xp[q]), g0);
                                g1 = fmaf(fg.y, bf16_hi(xp[q]), g1);
                                u0 = fmaf(fu.x, bf16_lo(xp[q]), u0);
                                u1 = fmaf(fu.y, bf16_hi(xp[q]), u1);
                            }
                        }
                    }
                    g[n] = fmaf(b ? sg.y : sg.x, g0 + g1, g[n]);
                    u[n] = fmaf(b ? su.y : su.x, u0 + u1, u[n]);
                }
            }
        }
    }
}

// Row pair v of the warp's row space: active expert v / I, row pair v % I.
template <bool FAST, int NT>
__device__ __forceinline__ void gu_loop(GuItem (&buf)[kDepth], const uint8_t* __restrict__ gu_codes,
                                        const uint8_t* __restrict__ gu_scales, const float* __restrict__ gu_ts,
                                        const uint16_t* xs, const int* sexp, const PairList& L, float* __restrict__ h,
                                        int H, int I, int v_lo, int v_hi, int lv, int li, int lane)
{
    const int cpl = H / 1024;  // 32-element chunks per lane per row
    const int64_t cp = H / 2, sp = H / 16;
    const int total = (v_hi - v_lo) * cpl;
    int cv = v_lo, ci = 0;
    float g[NT], u[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) g[n] = u[n] = 0.f;
    for (int j0 = 0; j0 < total; j0 += kDepth) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int j = j0 + d;
            if (j < total) {
                const GuItem cur = buf[d];
                if (j + kDepth < total) {
                    const int a = lv / I, i = lv - a * I, e = L.act[a];
                    const int64_t rg = static_cast<int64_t>(e) * 2 * I + i;
                    const int c = lane + 32 * li;
                    buf[d].g = ld_stream_v4(gu_codes + rg * cp + 16 * c);
                    buf[d].u = ld_stream_v4(gu_codes + (rg + I) * cp + 16 * c);
                    buf[d].sg = ld_stream_u16(gu_scales + rg * sp + 2 * c);
                    buf[d].su = ld_stream_u16(gu_scales + (rg + I) * sp + 2 * c);
                    if (++li == cpl) {
                        li = 0;
                        ++lv;
                    }
                }
                const int a = cv / I;
                const int p0 = L.act_p0[a], ne = L.act_p0[a + 1] - p0;
                gu_item<FAST, NT>(cur, xs, H, L, p0, ne, lane + 32 * ci, g, u);
                if (++ci == cpl) {
                    const int i = cv - a * I;
                    const float ts = gu_ts[L.act[a]];
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        if (n < ne) {
                            const int t = L.pt[p0 + n];
                            const float gs = warp_sum(g[n]), us = warp_sum(u[n]);
                            if (lane == 0 && t >= 0) {
                                const float gv = ldexpf(gs * ts, sexp[t]), uv = ldexpf(us * ts, sexp[t]);
                                h[static_cast<int64_t>(p0 + n) * I + i] = gv / (1.0f + expf(-gv)) * uv;
                            }
                        }
                        g[n] = u[n] = 0.f;
                    }
                    ci = 0;
                    ++cv;
                }
            }
        }
    }
}

// Dynamic shared memory: the activations, kMaxT * H * 2 bytes.
__global__ void __launch_bounds__(kTh, 2)
    moe_small_gu_kernel(const float* __restrict__ logits, const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ pair_token, const float* __restrict__ pair_weight,
                        const int32_t* __restrict__ pair_slot, const uint8_t* __restrict__ gu_codes,
                        const uint8_t* __restrict__ gu_scales, const float* __restrict__ gu_ts,
                        const uint16_t* __restrict__ x, MoeWorkspace ws, int E, int H, int I, int T, int topk)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ PairList L;
    __shared__ int s_emax[kMaxT], s_emin[kMaxT], s_sexp[kMaxT], s_flags;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);

    if (threadIdx.x == 0) s_flags = 0;  // ordered before their use by the barriers of the routing
    if (threadIdx.x < kMaxT) {
        s_emax[threadIdx.x] = 0;
        s_emin[threadIdx.x] = INT_MAX;
    }
    pdl_wait();  // logits, the list and x may come from the previous kernel
    if (logits)
        route_in_cta(logits, T, E, topk, L);
    else
        read_list(offsets, pair_token, pair_weight, pair_slot, T, E, topk, L);
    pdl_trigger();  // the down kernel may start: its inputs are complete
    if (blockIdx.x == 0 && threadIdx.x == 0) *ws.status = L.status;

    // this warp's row pairs, an even split of all active experts' I row pairs
    const int nv = L.n_act * I;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWp + warp, nw = static_cast<int64_t>(gridDim.x) * kWp;
    const int v_lo = static_cast<int>(nv * gw / nw), v_hi = static_cast<int>(nv * (gw + 1) / nw);
    const int cpl = H / 1024;
    const int64_t cp = H / 2, sp = H / 16;
    const int total = (v_hi - v_lo) * cpl;
    GuItem buf[kDepth];
    int lv = v_lo, li = 0;
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
        if (d < total) {
            const int a = lv / I, i = lv - a * I, e = L.act[a];
            const int64_t rg = static_cast<int64_t>(e) * 2 * I + i;
            const int c = lane + 32 * li;
            buf[d].g = ld_stream_v4(gu_codes + rg * cp + 16 * c);
            buf[d].u = ld_stream_v4(gu_codes + (rg + I) * cp + 16 * c);
            buf[d].sg = ld_stream_u16(gu_scales + rg * sp + 2 * c);
            buf[d].su = ld_stream_u16(gu_scales + (rg + I) * sp + 2 * c);
            if (++li == cpl) {
                li = 0;
                ++lv;
            }
        }
    }

    // each token's exponent range (bf16 biased exponents of its nonzero
    // elements), all threads over all tokens, reduced per warp then per CTA
    for (int t = 0; t < T; ++t) {
        int emax = 0, emin = INT_MAX, flags = 0;
        const uint32_t* xr = reinterpret_cast<const uint32_t*>(x + static_cast<int64_t>(t) * H);
#pragma unroll 4
        for (int i = threadIdx.x; i < H / 2; i += kTh) {
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
            atomicMax(&s_emax[t], emax);
            atomicMin(&s_emin[t], emin);
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
    // an expert has at most T of the pairs (one per token)
#define BQD_GU(F_, NT_) gu_loop<F_, NT_>(buf, gu_codes, gu_scales, gu_ts, xs, s_sexp, L, ws.h, H, I, v_lo, v_hi, lv, li, lane)
    if (fast) {
        if (T == 1) BQD_GU(true, 1);
        else if (T == 2) BQD_GU(true, 2);
        else BQD_GU(true, kMaxT);
    } else {
        if (T == 1) BQD_GU(false, 1);
        else if (T == 2) BQD_GU(false, 2);
        else BQD_GU(false, kMaxT);
    }
#undef BQD_GU
}

// ------------------------------------------------------------------ down + combine
struct DnItem {
    uint4 c;     // 16 code bytes (32 elements) of row j of the pair's expert
    uint32_t s;  // their two E4M3 block scales
};

// Loads of item (row j, step st): lane takes chunk lane % LP of pair
// q = st * PP + lane / LP (token-major order) if that pair exists.
__device__ __forceinline__ void dn_load(DnItem& it, const uint8_t* __restrict__ dn_codes,
                                        const uint8_t* __restrict__ dn_scales, const PairList& L, int H, int I, int P,
                                        int j, int st, int lane, int LP, int PP)
{
    const int q = st * PP + lane / LP, c = lane % LP;
    const int p = q < P ? L.qp[q] : -1;
    if (p >= 0) {
        const int64_t row = static_cast<int64_t>(L.pe[p]) * H + j;
        it.c = ld_stream_v4(dn_codes + row * (I / 2) + 16 * c);
        it.s = ld_stream_u16(dn_scales + row * (I / 16) + 2 * c);
    } else {
        it.c = make_uint4(0u, 0u, 0u, 0u);
        it.s = 0u;
    }
}

__device__ __forceinline__ float dn_dot(const DnItem& it, const float* hrow, int c)
{
    const float2 sc = e4m3x2_to_float2(it.s);
    const uint32_t w[4] = {it.c.x, it.c.y, it.c.z, it.c.w};
    float acc = 0.f;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int wi = 2 * b + jj;  // elements 8wi .. 8wi+7 = h pieces 2wi, 2wi+1
            uint32_t hw[4];
            e2m1x8_to_f16x2(w[wi], hw);
            const float4 h0 = *reinterpret_cast<const float4*>(hrow + xf_index(c, 2 * wi));
            const float4 h1 = *reinterpret_cast<const float4*>(hrow + xf_index(c, 2 * wi + 1));
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

// Dynamic shared memory: h, P * I fp32.
__global__ void __launch_bounds__(kTh, 2)
    moe_small_dn_kernel(const float* __restrict__ logits, const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ pair_token, const float* __restrict__ pair_weight,
                        const int32_t* __restrict__ pair_slot, const uint8_t* __restrict__ dn_codes,
                        const uint8_t* __restrict__ dn_scales, const float* __restrict__ dn_ts, float* __restrict__ y,
                        MoeWorkspace ws, int E, int H, int I, int T, int topk)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ PairList L;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int P = T * topk;
    float* hs = reinterpret_cast<float*>(smem);

    // The routing inputs are complete: the gate_up kernel let this kernel
    // start only after its own wait for the kernel before it.
    if (logits)
        route_in_cta(logits, T, E, topk, L);
    else
        read_list(offsets, pair_token, pair_weight, pair_slot, T, E, topk, L);
    if (threadIdx.x < P) L.pts[threadIdx.x] = dn_ts[L.pe[threadIdx.x]];
    __syncthreads();

    const int LP = I / 32, PP = kWarp / LP;  // lanes per pair, pairs per warp step
    const int steps = (P + PP - 1) / PP;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWp + warp, nw = static_cast<int64_t>(gridDim.x) * kWp;
    const int j_lo = static_cast<int>(H * gw / nw), j_hi = static_cast<int>(H * (gw + 1) / nw);
    const bool ok = L.status != kStatusBadOffsets;
    const int total = ok ? (j_hi - j_lo) * steps : 0;
    DnItem buf[kDepth];
    int lj = j_lo, ls = 0;
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
        if (d < total) {
            dn_load(buf[d], dn_codes, dn_scales, L, H, I, P, lj, ls, lane, LP, PP);
            if (++ls == steps) {
                ls = 0;
                ++lj;
            }
        }
    }

    pdl_wait();  // h comes from the gate_up kernel; y may be read by earlier kernels
#pragma unroll 4
    for (int i = threadIdx.x; i < P * (I / 4); i += kTh) {
        const int p = i / (I / 4), v = i - p * (I / 4);
        float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (L.pt[p] >= 0) hv = reinterpret_cast<const float4*>(ws.h + static_cast<int64_t>(p) * I)[v];
        *reinterpret_cast<float4*>(hs + p * I + xf_index(v >> 3, v & 7)) = hv;
    }
    __syncthreads();

    float acc[kMaxT];
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) acc[t] = 0.f;
    int cj = j_lo, cs = 0;
    for (int j0 = 0; j0 < total; j0 += kDepth) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int jdx = j0 + d;
            if (jdx < total) {
                const DnItem cur = buf[d];
                if (jdx + kDepth < total) {
                    dn_load(buf[d], dn_codes, dn_scales, L, H, I, P, lj, ls, lane, LP, PP);
                    if (++ls == steps) {
                        ls = 0;
                        ++lj;
                    }
                }
                const int q = cs * PP + lane / LP;
                const int p = q < P ? L.qp[q] : -1;
                float v = p >= 0 ? dn_dot(cur, hs + p * I, lane % LP) : 0.f;
                for (int o = LP / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                // the combine, in token-major slot order
                for (int g = 0; g < PP; ++g) {
                    const float d_g = __shfl_sync(0xFFFFFFFFu, v, g * LP);
                    const int qg = cs * PP + g;
                    const int pg = qg < P ? L.qp[qg] : -1;
                    if (pg >= 0) {
                        const float dv = d_g * L.pts[pg];
                        const int t = qg / topk;
#pragma unroll
                        for (int tt = 0; tt < kMaxT; ++tt)
                            if (tt == t) acc[tt] = fmaf(L.pw[pg], dv, acc[tt]);
                    }
                }
                if (++cs == steps) {
                    if (lane == 0)
                        for (int t = 0; t < T; ++t) y[static_cast<int64_t>(t) * H + cj] = acc[t];
#pragma unroll
                    for (int t = 0; t < kMaxT; ++t) acc[t] = 0.f;
                    cs = 0;
                    ++cj;
                }
            }
        }
    }
    if (!ok && lane == 0)  // malformed CSR: outputs unspecified, written as zero
        for (int j = j_lo; j < j_hi; ++j)
            for (int t = 0; t < T; ++t) y[static_cast<int64_t>(t) * H + j] = 0.f;
}

size_t small_smem(int64_t bytes) { return static_cast<size_t>(bytes); }

}  // namespace

bool moe_small_supported(int E, int H, int I, int T, int topk)
{
    return T >= 1 && T <= kMaxT && T * topk <= kMaxP && topk <= kWarp && E >= 1 && E <= kMaxE && H >= 1024 &&
           H % 1024 == 0 && H <= 8192 && (I == 256 || I == 512 || I == 1024);
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

    const size_t smem_gu = small_smem(static_cast<int64_t>(kMaxT) * H * 2);
    const size_t smem_dn = small_smem(static_cast<int64_t>(T) * topk * I * 4);
    static OccCache occ_gu, occ_dn;
    blocks_per_sm(occ_gu, reinterpret_cast<const void*>(moe_small_gu_kernel), dev, kTh, smem_gu);
    blocks_per_sm(occ_dn, reinterpret_cast<const void*>(moe_small_dn_kernel), dev, kTh, smem_dn);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(kTh);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.dynamicSmemBytes = smem_gu;
    err = cudaLaunchKernelEx(&cfg, moe_small_gu_kernel, logits, offsets, pair_token, pair_weight, pair_slot, gu_codes,
                             gu_scales, gu_ts, x, ws, E, H, I, T, topk);
    if (err != cudaSuccess) return err;
    // The down kernel always follows programmatically: it reads nothing that
    // the gate_up kernel writes before its griddepcontrol.wait.
    cfg.numAttrs = 1;
    cfg.dynamicSmemBytes = smem_dn;
    return cudaLaunchKernelEx(&cfg, moe_small_dn_kernel, logits, offsets, pair_token, pair_weight, pair_slot,
                              dn_codes, dn_scales, dn_ts, y, ws, E, H, I, T, topk);
}

}  // namespace bqd
