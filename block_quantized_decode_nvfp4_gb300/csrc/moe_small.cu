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
#include "stream.cuh"

namespace bqd {

// Device error word of the small-batch MoE kernels (kErrWaitTimeout: the
// activations' copy did not land in time); read and cleared by
// read_and_clear_moe_small_error().
__device__ unsigned int g_moe_small_error = 0;

namespace {

constexpr int kThG = 512;           // threads per CTA of the gate_up kernel (16 warps, 128 registers each)
constexpr int kWpG = kThG / kWarp;
constexpr int kMaxT = 16;           // tokens
constexpr int kMaxTH = 32768;       // tokens x hidden size (staged activations, 64 KiB)
constexpr int kMaxP = 128;          // routed (token, slot) pairs
constexpr int kMaxE = 512;          // experts
constexpr int kGDepth = 4;          // the same, row-wise gate_up
constexpr int kStatusBadOffsets = 1;
constexpr int kStatusBadPair = 2;
constexpr int kStatusCoverage = 4;

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 2^e for a normal exponent e (-126 .. 127).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }


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
    int pq[kMaxP];           // (token, slot) of pair p (-1: invalid pair)
    int cover[kMaxP];        // times (token, slot) q appears
    int sel_e[kMaxP];        // routing scratch: expert of q
    float sel_w[kMaxP];      // routing scratch: weight of q
    int status;
};

// Token groups from pe[0..P) (expert-major): every expert's segment of pairs
// cut into groups of at most `group` pairs (tokens), in order; the gate_up
// kernel reads a group's rows once for its tokens (an expert with more
// tokens is read once per group). By warp 0 in runs of 32 pairs. Needs a
// barrier before use.
__device__ void find_active(PairList& L, int P, int group)
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
            const bool gstart = p < P && (p - seg) % group == 0;
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

// Block-wide exclusive scan of one int per thread (any block of at most
// 1024 threads); s_scan holds one int per warp plus one. Returns the
// exclusive prefix; *total gets the sum.
__device__ __forceinline__ int block_scan(int v, int* s_scan, int* total)
{
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp, nwp = blockDim.x / kWarp;
    int incl = v;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == kWarp - 1) s_scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int t = lane < nwp ? s_scan[lane] : 0;
        int it = t;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, it, o);
            if (lane >= o) it += n;
        }
        if (lane < nwp) s_scan[lane] = it - t;
        if (lane == nwp - 1) s_scan[nwp] = it;
    }
    __syncthreads();
    const int r = s_scan[warp] + incl - v;
    *total = s_scan[nwp];
    __syncthreads();
    return r;
}

// Routing of T tokens from their logits, every CTA for itself (warp w routes
// token w), and the expert-major list of the routed pairs: every token sets
// its bit in the token masks of its experts; an exclusive scan over experts
// of (pairs, groups) gives each expert's first pair and first token group;
// a pair's place is its expert's first pair plus the number of lower tokens
// in the expert's mask (tokens ascending inside an expert, the order
// moe_route_topk writes). E <= blockDim.x, T <= 32.
__device__ void route_in_cta(const float* __restrict__ logits, int T, int E, int topk, int group, PairList& L,
                             uint32_t* s_mask, int* s_eoff, int* s_scan)
{
    const int P = T * topk;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0u;
    for (int t = warp; t < T; t += blockDim.x / kWarp) {
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
    const int g = (c + group - 1) / group;         // its token groups
    int total = 0;
    const int excl = block_scan((g << 16) | c, s_scan, &total);
    if (c) {
        const int off = excl & 0xFFFF, goff = excl >> 16;
        s_eoff[e] = off;
        for (int k = 0; k < g; ++k) {
            L.act[goff + k] = e;
            L.act_p0[goff + k] = off + k * group;
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
        L.pq[r] = q;
    }
    __syncthreads();
}

// The caller's expert-major list, checked: a CSR that is not monotone or does
// not cover [0, P) sets BQD_MOE_BAD_OFFSETS (nothing is computed); a token or
// slot out of range sets BQD_MOE_BAD_PAIR (the pair is skipped); a (token,
// slot) present zero or several times sets BQD_MOE_COVERAGE.
__device__ void read_list(const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_token,
                          const float* __restrict__ pair_weight, const int32_t* __restrict__ pair_slot, int T, int E,
                          int topk, int group, PairList& L)
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
    for (int e = threadIdx.x; e < E; e += blockDim.x)
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
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
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
            L.pq[r] = t * topk + s;
        } else {
            L.pt[r] = -1;
            L.pq[r] = -1;
            atomicOr(&L.status, kStatusBadPair);
        }
    }
    __syncthreads();
    if (threadIdx.x < P && L.cover[threadIdx.x] != 1) {
        atomicOr(&L.status, kStatusCoverage);
        if (L.cover[threadIdx.x] == 0) L.qp[threadIdx.x] = -1;
    }
    find_active(L, P, group);
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

// One chunk of an expert row against its NE tokens (listed in tok[]; a
// negative entry, an invalid pair of a caller's list, reads token 0 and its
// result is dropped by the caller): xc is this lane's chunk of token 0's
// staged activations (token t's start t * H elements later), sw the lane's
// swizzle. The chunk is decoded once for all tokens.
template <bool FAST, int NE, int NT>
__device__ __forceinline__ void gu_dot(const Item& it, const uint16_t* xc, int H, const int* tok, int sw,
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
    for (int n = 0; n < NE; ++n) {
        const uint16_t* xr = xc + max(tok[n], 0) * H;
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

// gu_dot for the group's token count ne (1 .. NT), so that only ne tokens'
// work is issued.
template <bool FAST, int NT>
__device__ __forceinline__ void gu_dot_n(const Item& it, const uint16_t* xc, int H, const int* tok, int ne, int sw,
                                         float (&acc)[NT])
{
    if constexpr (NT == 1) {
        gu_dot<FAST, 1, NT>(it, xc, H, tok, sw, acc);
    } else {
        static_assert(NT == 2, "row-wise gate_up takes groups of 1 or 2 tokens");
        if (ne == 1)
            gu_dot<FAST, 1, NT>(it, xc, H, tok, sw, acc);
        else
            gu_dot<FAST, 2, NT>(it, xc, H, tok, sw, acc);
    }
}

// h = SiLU(g) * u of pair p at row l: to the workspace's h (pair order) and,
// times the pair's routing weight and the expert's down tensor scale, to the
// down kernel's input h' (workspace partial area, (token, slot) order).
__device__ __forceinline__ void put_h(const PairList& L, const MoeWorkspace& ws, int p, int I, int l, float g, float u,
                                      float dsc)
{
    const float h = g / (1.0f + expf(-g)) * u;
    ws.h[static_cast<int64_t>(p) * I + l] = h;
    ws.part[static_cast<int64_t>(L.pq[p]) * I + l] = h * (L.pw[p] * dsc);
}

// ------------------------------------------------------------------ gate_up, by rows (T <= 2)
// Virtual row v of the gate_up row space: active group a = v / (2I), then
// gate row l and up row l alternate (v % (2I) = 2l for the gate, 2l + 1 for
// the up projection), so that a warp, whose range starts at an even v, has
// g in registers when it finishes the matching u row.
__device__ __forceinline__ int64_t gu_row(const PairList& L, int v, int sh, int lmask, int I)
{
    const int a = v >> sh, l2 = v & lmask;
    return static_cast<int64_t>(L.act[a]) * 2 * I + ((l2 & 1) ? I : 0) + (l2 >> 1);
}

template <int CPL>
__device__ __forceinline__ void gu_rows_prologue(Item (&buf)[kGDepth], const uint8_t* __restrict__ gu_codes,
                                                 const uint8_t* __restrict__ gu_scales, const PairList& L, int I,
                                                 int v_lo, int v_hi, int lane)
{
    constexpr int H = 1024 * CPL;
    const int64_t cp = H / 2, sp = H / 16;
    const int sh = __ffs(2 * I) - 1, lmask = 2 * I - 1;
#pragma unroll
    for (int d = 0; d < kGDepth; ++d) {
        const int v = v_lo + d / CPL;
        if (v < v_hi) {
            const int64_t row = gu_row(L, v, sh, lmask, I);
            buf[d] = load_item(gu_codes + row * cp + (d % CPL) * 512 + lane * 16,
                               gu_scales + row * sp + (d % CPL) * 64 + lane * 2);
        }
    }
}

template <int CPL, int NT, bool FAST>
__device__ __forceinline__ void gu_rows(Item (&buf)[kGDepth], const uint8_t* __restrict__ gu_codes,
                                        const uint8_t* __restrict__ gu_scales, const float* __restrict__ gu_ts,
                                        const float* __restrict__ dn_ts, const uint16_t* xs, const int* sexp,
                                        const PairList& L, const MoeWorkspace& ws, int I, int v_lo, int v_hi, int lane)
{
    static_assert(CPL % kGDepth == 0 || kGDepth % CPL == 0, "ring depth must divide a row or be a multiple of one");
    constexpr int H = 1024 * CPL;
    constexpr int U = kGDepth > CPL ? kGDepth / CPL : 1;
    const int64_t cp = H / 2, sp = H / 16;
    const int sw = (lane >> 1) & 3;
    const int sh = __ffs(2 * I) - 1, lmask = 2 * I - 1;  // 2I is a power of two
    float gsave[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) gsave[n] = 0.f;
    for (int v0 = v_lo; v0 < v_hi; v0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u;
            if (v < v_hi) {
                const int a = v >> sh, l2 = v & lmask;
                const int p0 = L.act_p0[a], ne = L.act_p0[a + 1] - p0;
                float acc[NT];
#pragma unroll
                for (int n = 0; n < NT; ++n) acc[n] = 0.f;
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    const int g = u * CPL + i;
                    const Item cur = buf[g % kGDepth];
                    const int nr = (g + kGDepth) / CPL, nc = (g + kGDepth) % CPL;
                    const int vn = v0 + nr;
                    if (vn < v_hi) {
                        const int64_t row = gu_row(L, vn, sh, lmask, I);
                        buf[g % kGDepth] = load_item(gu_codes + row * cp + nc * 512 + lane * 16,
                                                    gu_scales + row * sp + nc * 64 + lane * 2);
                    }
                    gu_dot_n<FAST, NT>(cur, xs + lane * 32 + i * 1024, H, L.pt + p0, ne, sw, acc);
                    asm volatile("" ::: "memory");
                }
                const int e = L.act[a];
                const float ts = gu_ts[e];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if (n < ne) {
                        const int t = L.pt[p0 + n];
                        const float val = ldexpf(warp_sum(acc[n]) * ts, sexp[max(t, 0)]);
                        if (!(l2 & 1))
                            gsave[n] = val;
                        else if (lane == 0 && t >= 0)
                            put_h(L, ws, p0 + n, I, l2 >> 1, gsave[n], val, dn_ts[e]);
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------ gate_up, by tensor-core tiles (T >= 3)
// A warp tile is gate rows l0 .. l0+7 of a group's expert and the matching up
// rows, against the group's tokens (at most 8), with mma.sync m16n8k16
// (f16 or bf16 operands, fp32 accumulation): A = the 16 weight rows (gate
// rows as rows 0..7, up rows as rows 8..15), B = the tokens' activations,
// one token per column. Lane (g, i) = (lane / 4, lane % 4) loads 16 code
// bytes (32 elements, k = 32 i .. 32 i + 31 of each 128-element chunk) of
// gate row l0 + g and of up row l0 + g, and the chunk's activations of token
// slot g at the same k. The k order inside an mma is free as long as A and B
// agree: step j of a chunk takes, for quad i, elements 32 i + 4 j .. + 3
// (logical k 2i, 2i+1, 2i+8, 2i+9), which both fragments hold in the same
// registers. Weights enter as w * s (E2M1 code times its E4M3 block scale),
// exact in f16 and bf16 (at most 6 significant bits, magnitudes in
// [2^-10, 2688]). The accumulators end as (gate, token 2i), (gate, 2i+1),
// (up, 2i), (up, 2i+1) of row l0 + g: SiLU(g) * u is formed in the lane.
constexpr int kMDepth = 4;  // 128-element chunks in flight per lane

struct MSlot {
    uint4 gc, uc;  // gate and up code bytes
    uint32_t sc;   // gate block scales (low 16 bits), up block scales (high 16 bits)
};

// Staged activations of the tile path: token t's row of H f16 (or bf16)
// values at xs + t * H, 16-byte piece p at slot xm_piece(t, p): the eight
// lanes of one shared-memory wavefront (two token slots x four quads) then
// hit distinct banks when the two tokens differ in parity.
__device__ __forceinline__ int xm_piece(int t, int p) { return p ^ (t & 1) ^ (((p >> 3) & 1) << 1); }

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

// One 128-element chunk of a tile: xk points at token slot g's staged
// activations of the chunk (null for an empty slot: zeros), xo the lane's
// four swizzled piece offsets. The two mma steps of each 32-bit code word go
// to separate accumulators (two dependency chains).
template <bool FAST>
__device__ __forceinline__ void mma_chunk(const MSlot& cur, const uint16_t* xk, const int (&xo)[4],
                                          float (&acc0)[4], float (&acc1)[4])
{
    const uint32_t gs = e4m3x2_to_f16x2(cur.sc & 0xFFFFu), us = e4m3x2_to_f16x2(cur.sc >> 16);
    const uint32_t gsl = __byte_perm(gs, 0, 0x1010), gsh = __byte_perm(gs, 0, 0x3232);
    const uint32_t usl = __byte_perm(us, 0, 0x1010), ush = __byte_perm(us, 0, 0x3232);
    const uint32_t gw[4] = {cur.gc.x, cur.gc.y, cur.gc.z, cur.gc.w};
    const uint32_t uw[4] = {cur.uc.x, cur.uc.y, cur.uc.z, cur.uc.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t gp[4], up[4];
        e2m1x8_to_f16x2(gw[w], gp);
        e2m1x8_to_f16x2(uw[w], up);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            gp[q] = hmul2_bits(gp[q], w < 2 ? gsl : gsh);
            up[q] = hmul2_bits(up[q], w < 2 ? usl : ush);
        }
        uint4 xq = make_uint4(0u, 0u, 0u, 0u);
        if (xk) xq = *reinterpret_cast<const uint4*>(xk + xo[w]);
        if constexpr (FAST) {
            mma_f16(acc0, gp[0], up[0], gp[1], up[1], xq.x, xq.y);
            mma_f16(acc1, gp[2], up[2], gp[3], up[3], xq.z, xq.w);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                gp[q] = f16x2_as_bf16x2(gp[q]);
                up[q] = f16x2_as_bf16x2(up[q]);
            }
            mma_bf16(acc0, gp[0], up[0], gp[1], up[1], xq.x, xq.y);
            mma_bf16(acc1, gp[2], up[2], gp[3], up[3], xq.z, xq.w);
        }
    }
}

// The lane's row pointers of one tile: gate and up code bytes and block
// scales at k = 32 i of chunk 0 (chunk kc is 64 code bytes and 8 scale
// bytes further).
struct TilePtr {
    const uint8_t *gc, *uc, *gs, *us;
};

template <int CPL>
struct TileIo {
    static constexpr int H = 1024 * CPL, KCH = H / 128;  // 128-element chunks per row
    const uint8_t* codes;
    const uint8_t* scales;
    const PairList* L;
    int I, tsh, g, i;  // tsh: log2 of the tiles per group (I / 8)
    __device__ __forceinline__ TilePtr ptrs(int tile) const
    {
        const int a = tile >> tsh, l0 = (tile & ((1 << tsh) - 1)) * 8;
        const int64_t rg = static_cast<int64_t>(L->act[a]) * 2 * I + l0 + g;
        TilePtr t;
        t.gc = codes + rg * (H / 2) + i * 16;
        t.uc = t.gc + static_cast<int64_t>(I) * (H / 2);
        t.gs = scales + rg * (H / 16) + i * 2;
        t.us = t.gs + static_cast<int64_t>(I) * (H / 16);
        return t;
    }
    static __device__ __forceinline__ MSlot load(const TilePtr& t, int kc)
    {
        MSlot s;
        s.gc = ld_stream_v4(t.gc + kc * 64);
        s.uc = ld_stream_v4(t.uc + kc * 64);
        s.sc = ld_stream_u16(t.gs + kc * 8) | (ld_stream_u16(t.us + kc * 8) << 16);
        return s;
    }
};

// The warp's tiles [t_lo, t_hi); the ring holds chunks 0 .. kMDepth-1 of
// tile t_lo on entry. Refills within a tile use the tile's pointers plus
// compile-time offsets; the last kMDepth chunks of a tile refill the first
// ones of the next.
template <int CPL, bool FAST>
__device__ __forceinline__ void gu_tiles(MSlot (&ring)[kMDepth], const TileIo<CPL>& io, const float* __restrict__ gu_ts,
                                         const float* __restrict__ dn_ts, const uint16_t* xs, const int* sexp,
                                         const PairList& L, const MoeWorkspace& ws, int t_lo, int t_hi)
{
    constexpr int H = TileIo<CPL>::H, KCH = TileIo<CPL>::KCH;
    static_assert(KCH % kMDepth == 0 && KCH > kMDepth, "ring depth must divide the chunks of a row");
    const int I = io.I, g = io.g, i = io.i;
    TilePtr cur = io.ptrs(t_lo);
    for (int tile = t_lo; tile < t_hi; ++tile) {
        const bool more = tile + 1 < t_hi;
        const TilePtr nxt = more ? io.ptrs(tile + 1) : cur;
        const int a = tile >> io.tsh, l0 = (tile & ((1 << io.tsh) - 1)) * 8;
        const int p0 = L.act_p0[a], ne = L.act_p0[a + 1] - p0;
        const int tg = g < ne ? L.pt[p0 + g] : -1;
        const int tx = max(tg, 0);
        // token slot g's activations, lane quad i's four pieces of each chunk
        const uint16_t* xr = tg >= 0 ? xs + tx * H : nullptr;
        int xo[4];
        const int xm = (tx & 1) | ((i >> 1) << 1);
#pragma unroll
        for (int w = 0; w < 4; ++w) xo[w] = ((4 * i + w) ^ xm) << 3;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kc0 = 0; kc0 < KCH - kMDepth; kc0 += kMDepth) {
#pragma unroll
            for (int d = 0; d < kMDepth; ++d) {
                const MSlot c = ring[d];
                ring[d] = TileIo<CPL>::load(cur, kc0 + d + kMDepth);
                mma_chunk<FAST>(c, xr ? xr + (kc0 + d) * 128 : nullptr, xo, acc0, acc1);
                asm volatile("" ::: "memory");
            }
        }
#pragma unroll
        for (int d = 0; d < kMDepth; ++d) {
            const MSlot c = ring[d];
            if (more) ring[d] = TileIo<CPL>::load(nxt, d);
            mma_chunk<FAST>(c, xr ? xr + (KCH - kMDepth + d) * 128 : nullptr, xo, acc0, acc1);
            asm volatile("" ::: "memory");
        }
        const int e = L.act[a];
        const float ts = gu_ts[e], dsc = dn_ts[e];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int n = 2 * i + c;
            if (n < ne) {
                const int p = p0 + n, t = L.pt[p];
                if (t >= 0)
                    put_h(L, ws, p, I, l0 + g, ldexpf((acc0[c] + acc1[c]) * ts, sexp[t]),
                          ldexpf((acc0[2 + c] + acc1[2 + c]) * ts, sexp[t]), dsc);
            }
        }
        cur = nxt;
    }
}

// ------------------------------------------------------------------ gate_up kernel
// NT = 1, 2: rows (groups of NT tokens); NT = 8: tensor-core tiles (groups
// of up to 8 tokens). Dynamic shared memory: the staged activations, T * H
// f16 (or bf16), then x as given (T * H bf16).
template <int CPL, int NT>
__global__ void __launch_bounds__(kThG, 1)
    moe_small_gu_kernel(const float* __restrict__ logits, const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ pair_token, const float* __restrict__ pair_weight,
                        const int32_t* __restrict__ pair_slot, const uint8_t* __restrict__ gu_codes,
                        const uint8_t* __restrict__ gu_scales, const float* __restrict__ gu_ts,
                        const uint16_t* __restrict__ x, const float* __restrict__ dn_ts, MoeWorkspace ws, int E, int I,
                        int T, int topk)
{
    constexpr int H = 1024 * CPL;
    constexpr bool kTiles = NT == 8;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ PairList L;
    __shared__ int s_emax[kMaxT], s_emin[kMaxT], s_sexp[kMaxT], s_flags;
    __shared__ int s_need[kMaxT], s_nneed;  // the tokens whose activations this CTA stages
    __shared__ uint32_t s_mask[kMaxE];
    __shared__ int s_eoff[kMaxE], s_scan[kWpG + 1];
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);  // staged activations
    uint16_t* xraw = xs + T * H;                          // x as given
    __shared__ uint64_t s_xbar;                           // x's bulk copy landed

    if (threadIdx.x == 0) {  // ordered before their use by the barriers of the routing
        s_flags = 0;
        mbar_init(&s_xbar, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < kMaxT) {
        s_emax[threadIdx.x] = 0;
        s_emin[threadIdx.x] = INT_MAX;
    }
    pdl_wait();  // logits, the list and x may come from the previous kernel
    // x, copied to shared memory by one bulk copy (its latency overlaps the
    // routing; an mbarrier tracks it, so waiting for it never waits for the
    // weight loads in flight), then staged in one pass through registers
    constexpr int kXP = kMaxTH / 8 / kThG;  // 16-byte pieces per thread
    if (threadIdx.x == 0) {
        const uint32_t xb = static_cast<uint32_t>(T) * H * 2;
        mbar_arrive_expect_tx(&s_xbar, xb);
        bulk_g2s(xraw, x, xb, &s_xbar);
    }
    if (logits)
        route_in_cta(logits, T, E, topk, NT, L, s_mask, s_eoff, s_scan);
    else
        read_list(offsets, pair_token, pair_weight, pair_slot, T, E, topk, NT, L);
    pdl_trigger();
    // the compact list the down kernel reads: per (token, slot) q its pair
    // (bits 16..) and expert (bits 0..15), or -1
    if (blockIdx.x == 0) {
        const int P = T * topk;
        if (threadIdx.x < P) {
            const int p = L.qp[threadIdx.x];
            ws.count[threadIdx.x] = p >= 0 && L.status != kStatusBadOffsets ? (p << 16) | L.pe[p] : -1;
        }
        if (threadIdx.x == 0) *ws.status = L.status;
    }

    // Activations: each token's exponent range (bf16 biased exponents of its
    // nonzero elements; the 32 pieces of a warp belong to one token), then
    // the staged copy. f16 holds x * 2^-s exactly when every nonzero |x| of
    // the token is within 31 binades of its largest; the largest lands in
    // [2^14, 2^15). Otherwise (or with a subnormal, infinite or NaN element)
    // the raw bf16 values are staged and the kernel computes in fp32 (rows)
    // or with bf16 operands (tiles).
    // Only the tokens in s_need[0 .. s_nneed) are staged (piece pc of the
    // compact order is piece pc % (H / 8) of token s_need[pc / (H / 8)]).
    auto stage_x = [&]() -> bool {
        mbar_wait(&s_xbar, 0, &g_moe_small_error);  // bounded; on time-out the outputs are unspecified
        __syncthreads();
        const int nps = s_nneed * (H / 8);
        uint4 xv[kXP];  // piece threadIdx.x + r kThG (consecutive per warp: no bank conflicts)
#pragma unroll
        for (int r = 0; r < kXP; ++r) {
            const int pc = threadIdx.x + r * kThG;
            if (pc < nps) {
                const int t = s_need[pc / (H / 8)], v = pc % (H / 8);
                xv[r] = *reinterpret_cast<const uint4*>(xraw + (t * (H / 8) + v) * 8);
            }
        }
        // |x| bit patterns (sign cleared) order like the values: the largest
        // and the smallest nonzero pattern per token give its exponent range
        // (and show an infinity or NaN, 0x7F80 and up, or a subnormal, below
        // 0x0080), a halfword max and min per 32-bit word; a warp's 32
        // pieces lie in one token
#pragma unroll
        for (int r = 0; r < kXP; ++r) {
            if (r * kThG + warp * kWarp < nps) {  // warp-uniform
                const uint32_t w4[4] = {xv[r].x, xv[r].y, xv[r].z, xv[r].w};
                uint32_t hmax = 0u, hmin = 0xFFFFFFFFu;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t m = w4[q] & 0x7FFF7FFFu;
                    hmax = __vmaxu2(hmax, m);
                    hmin = __vminu2(hmin, __vsub2(m, 0x00010001u));  // a zero half wraps to 0xFFFF
                }
                const uint32_t bmax = __reduce_max_sync(0xFFFFFFFFu, max(hmax & 0xFFFFu, hmax >> 16));
                const uint32_t bmin = __reduce_min_sync(0xFFFFFFFFu, min(hmin & 0xFFFFu, hmin >> 16)) + 1u;
                if (lane == 0) {
                    const int t = s_need[(r * kThG + warp * kWarp) / (H / 8)];
                    atomicMax(&s_emax[t], static_cast<int>(bmax));
                    atomicMin(&s_emin[t], static_cast<int>(bmin));  // 0x10000: no nonzero element
                }
            }
        }
        __syncthreads();
        if (threadIdx.x < T) {  // patterns to exponents (a token of zeros keeps emin = INT_MAX)
            const int bmax = s_emax[threadIdx.x], bmin = s_emin[threadIdx.x];
            const bool any = bmin < 0x10000;
            if (bmax >= 0x7F80 || (any && bmin < 0x0080) || (any && (bmax >> 7) - (bmin >> 7) > 31))
                atomicOr(&s_flags, 1);
            s_emax[threadIdx.x] = bmax >> 7;
            s_emin[threadIdx.x] = any ? bmin >> 7 : INT_MAX;
        }
        __syncthreads();
        const bool fast = s_flags == 0;
        if (threadIdx.x < kMaxT)
            s_sexp[threadIdx.x] = fast && threadIdx.x < T && s_emin[threadIdx.x] != INT_MAX
                                      ? s_emax[threadIdx.x] - 127 - 14
                                      : 0;
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kXP; ++r) {
            const int pc = threadIdx.x + r * kThG;
            if (pc >= nps) continue;
            const int t = s_need[pc / (H / 8)], v = pc % (H / 8);
            uint4 uu = xv[r];
            if (fast) {
                // x * 2^-s as two exact multiplies by normal powers of two
                const int se = s_sexp[t], e1 = max(-126, min(127, -se));
                const float f1 = pow2f(e1), f2 = pow2f(max(-126, min(127, -se - e1)));
                const uint32_t w4[4] = {uu.x, uu.y, uu.z, uu.w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    __half2 hv = __floats2half2_rn(bf16_lo(w4[q]) * f1 * f2, bf16_hi(w4[q]) * f1 * f2);
                    o[q] = *reinterpret_cast<uint32_t*>(&hv);
                }
                uu = make_uint4(o[0], o[1], o[2], o[3]);
            }
            const int slot = kTiles ? (xm_piece(t, v) << 3) : xh_index(v / 4, v % 4);
            *reinterpret_cast<uint4*>(xs + t * H + slot) = uu;
        }
        __syncthreads();
        return fast;
    };

    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWpG + warp, nw = static_cast<int64_t>(gridDim.x) * kWpG;
    if constexpr (kTiles) {
        // this warp's tiles: an even split of all groups' I / 8 tiles
        const int tsh = __ffs(I / 8) - 1;
        const int ntile = L.n_act << tsh;
        const int t_lo = static_cast<int>(ntile * gw / nw), t_hi = static_cast<int>(ntile * (gw + 1) / nw);
        TileIo<CPL> io{gu_codes, gu_scales, &L, I, tsh, lane >> 2, lane & 3};
        // the tokens of the CTA's tiles' groups (a group's tiles share its tokens)
        const int64_t gw0 = static_cast<int64_t>(blockIdx.x) * kWpG;
        const int c_lo = static_cast<int>(ntile * gw0 / nw), c_hi = static_cast<int>(ntile * (gw0 + kWpG) / nw);
        if (threadIdx.x == 0) s_nneed = 0;
        if (threadIdx.x < kMaxT) s_need[threadIdx.x] = 0;
        __syncthreads();
        if (c_lo < c_hi) {
            const int a_lo = c_lo >> tsh, a_hi = (c_hi - 1) >> tsh;
            for (int k = threadIdx.x; k < (a_hi - a_lo + 1) * NT; k += kThG) {
                const int a = a_lo + k / NT, p = L.act_p0[a] + k % NT;
                if (p < L.act_p0[a + 1] && L.pt[p] >= 0) s_need[L.pt[p]] = 1;
            }
        }
        __syncthreads();
        if (threadIdx.x < kWarp) {  // compact, ascending
            const bool nd = threadIdx.x < T && s_need[threadIdx.x] != 0;
            const uint32_t m = __ballot_sync(0xFFFFFFFFu, nd);
            __syncwarp();
            if (nd) s_need[__popc(m & ((1u << threadIdx.x) - 1u))] = threadIdx.x;
            if (threadIdx.x == 0) s_nneed = __popc(m);
        }
        MSlot ring[kMDepth];
        if (t_lo < t_hi) {
            const TilePtr first = io.ptrs(t_lo);
#pragma unroll
            for (int d = 0; d < kMDepth; ++d) ring[d] = TileIo<CPL>::load(first, d);
        }
        if (stage_x())
            gu_tiles<CPL, true>(ring, io, gu_ts, dn_ts, xs, s_sexp, L, ws, t_lo, t_hi);
        else
            gu_tiles<CPL, false>(ring, io, gu_ts, dn_ts, xs, s_sexp, L, ws, t_lo, t_hi);
    } else {
        // this warp's rows: an even split of all groups' gate/up row pairs
        const int nv2 = L.n_act * I;
        const int v_lo = 2 * static_cast<int>(nv2 * gw / nw), v_hi = 2 * static_cast<int>(nv2 * (gw + 1) / nw);
        if (threadIdx.x < T) s_need[threadIdx.x] = threadIdx.x;
        if (threadIdx.x == 0) s_nneed = T;
        Item buf[kGDepth];
        gu_rows_prologue<CPL>(buf, gu_codes, gu_scales, L, I, v_lo, v_hi, lane);
        if (stage_x())
            gu_rows<CPL, NT, true>(buf, gu_codes, gu_scales, gu_ts, dn_ts, xs, s_sexp, L, ws, I, v_lo, v_hi, lane);
        else
            gu_rows<CPL, NT, false>(buf, gu_codes, gu_scales, gu_ts, dn_ts, xs, s_sexp, L, ws, I, v_lo, v_hi, lane);
    }
}

// ------------------------------------------------------------------ down + combine
// Output (t, j) is the dot product of h'_t = [h'_{t,0} .. h'_{t,topk-1}] (the
// token's slots side by side, K' = topk * I elements) with row j of each of
// its experts, gathered. A warp computes R adjacent outputs (t, j) ..
// (t, j + R - 1) together (R = 2 when there are enough row pairs to keep
// every warp busy), so every h' value it reads from shared memory serves R
// rows. Lane l takes the chunks l + 32 i (i < CPLD) of the gathered rows:
// slot s = (l + 32 i) / CS (CS = I / 32 chunks per slot), chunk
// (l + 32 i) % CS = l % CS of the slot's expert rows (CS divides 32).
constexpr int kThD = 768;  // down kernel threads (24 warps), one CTA per SM
constexpr int kWpD = kThD / kWarp;
constexpr int kDDepth = 2;  // 32-element chunks in flight per lane

template <int R>
struct ItemRows {  // the same chunk of R adjacent rows
    Item r[R];
};

// hc: the chunk's staged h' (32 fp32; 16-byte piece p at ho[p] floats from
// hc: the lane's swizzle), read once for all R rows. One fp32 pair
// accumulator per row and scale block.
template <int R>
__device__ __forceinline__ void dn_dot(const ItemRows<R>& it, const float* hc, const int (&ho)[8], float (&acc)[R])
{
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        float2 a[R];
#pragma unroll
        for (int k = 0; k < R; ++k) a[k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int wi = 2 * b + jj;  // elements 8 wi .. 8 wi + 7 = h' pieces 2 wi, 2 wi + 1
            const float4 h0 = *reinterpret_cast<const float4*>(hc + ho[2 * wi]);
            const float4 h1 = *reinterpret_cast<const float4*>(hc + ho[2 * wi + 1]);
            const float2 xp[4] = {make_float2(h0.x, h0.y), make_float2(h0.z, h0.w), make_float2(h1.x, h1.y),
                                  make_float2(h1.z, h1.w)};
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const uint32_t w[4] = {it.r[k].c.x, it.r[k].c.y, it.r[k].c.z, it.r[k].c.w};
                uint32_t hw[4];
                e2m1x8_to_f16x2(w[wi], hw);
#pragma unroll
                for (int q = 0; q < 4; ++q) a[k] = __ffma2_rn(f16x2_to_float2(hw[q]), xp[q], a[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const float2 sc = e4m3x2_to_float2(it.r[k].s);
            acc[k] = fmaf(b ? sc.y : sc.x, a[k].x + a[k].y, acc[k]);
        }
    }
}

// Dynamic shared memory: h' of the tokens whose rows the CTA computes, topk
// * I fp32 per token (the token's slots side by side; chunk c's 16-byte
// piece p at slot p ^ (c & 7)). The pair list (the workspace count, one
// entry per (token, slot)) and h' (the workspace partial area, (token,
// slot) order) come from the gate_up kernel: nothing is routed here.
template <int CPLD, int CS, int R>
__global__ void __launch_bounds__(kThD, 1)
    moe_small_dn_kernel(const uint8_t* __restrict__ dn_codes, const uint8_t* __restrict__ dn_scales,
                        float* __restrict__ y, MoeWorkspace ws, int H, int T, int topk)
{
    constexpr int I = 32 * CS;
    constexpr uint32_t cp = I / 2, sp = I / 16;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_eh[kMaxP];  // expert * H of (token, slot) q, -1 if missing
    __shared__ int s_ok;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int P = T * topk, KC = topk * CS;  // chunks per gathered row
    float* hs = reinterpret_cast<float*>(smem);

    pdl_wait();  // the list and h' come from the gate_up kernel; y may be read by earlier kernels
    if (threadIdx.x < P) {
        const int v = ws.count[threadIdx.x];
        s_eh[threadIdx.x] = v >= 0 ? (v & 0xFFFF) * H : -1;
    }
    if (threadIdx.x == 0) s_ok = (*ws.status & kStatusBadOffsets) == 0;
    __syncthreads();
    const bool ok = s_ok != 0;

    // units u = rows R u .. R u + R - 1 (all of token t = R u / H, as R divides
    // H): an even split over the CTAs, then over the warps; the CTA stages h'
    // only for the tokens its rows belong to
    const int nr = ok ? T * H / R : 0;
    const int c_lo = static_cast<int>(static_cast<int64_t>(nr) * blockIdx.x / gridDim.x);
    const int c_hi = static_cast<int>(static_cast<int64_t>(nr) * (blockIdx.x + 1) / gridDim.x);
    const int hsh = __ffs(H) - 1;  // H is a power of two
    const int t_first = (R * c_lo) >> hsh;
    const int t_end = c_hi > c_lo ? ((R * (c_hi - 1)) >> hsh) + 1 : t_first;  // tokens [t_first, t_end)
    const int r_lo = c_lo + static_cast<int>(static_cast<int64_t>(c_hi - c_lo) * warp / kWpD);
    const int r_hi = c_lo + static_cast<int>(static_cast<int64_t>(c_hi - c_lo) * (warp + 1) / kWpD);
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
    // (expert * H + j) * cp < 2^32 for every supported shape (E <= 512, H <= 8192, I <= 1024)
    const uint8_t* cbase = dn_codes + (lane % CS) * 16;
    const uint8_t* sbase = dn_scales + (lane % CS) * 2;
    auto load_at = [&](int u, int i) -> ItemRows<R> {
        ItemRows<R> it;
#pragma unroll
        for (int k = 0; k < R; ++k) {
            it.r[k].c = make_uint4(0u, 0u, 0u, 0u);
            it.r[k].s = 0u;
        }
        const int r = R * u, t = r >> hsh, j = r & (H - 1);
        if (t != cur_t) set_token(t);
        if (eh[i] >= 0) {
            const uint32_t row = static_cast<uint32_t>(eh[i] + j);
#pragma unroll
            for (int k = 0; k < R; ++k) it.r[k] = load_item(cbase + (row + k) * cp, sbase + (row + k) * sp);
        }
        return it;
    };
    static_assert(CPLD % kDDepth == 0 || kDDepth % CPLD == 0, "ring depth must divide a row or be a multiple of one");
    constexpr int U = kDDepth > CPLD ? kDDepth / CPLD : 1;
    ItemRows<R> buf[kDDepth];
#pragma unroll
    for (int d = 0; d < kDDepth; ++d)
        if (r_lo + d / CPLD < r_hi) buf[d] = load_at(r_lo + d / CPLD, d % CPLD);

    // h' of the CTA's tokens' (token, slot) pairs, token-major, 16 bytes at a
    // time (zero for a missing pair)
    const int q0 = t_first * topk, nq = (t_end - t_first) * topk;
#pragma unroll 4
    for (int i4 = threadIdx.x; i4 < nq * (I / 4); i4 += kThD) {
        const int ql = i4 / (I / 4), k = (i4 - ql * (I / 4)) * 4, q = q0 + ql;
        float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s_eh[q] >= 0) hv = *reinterpret_cast<const float4*>(ws.part + static_cast<int64_t>(q) * I + k);
        const int tl = ql / topk, c = (ql - tl * topk) * CS + k / 32;  // chunk of the token's gathered row
        *reinterpret_cast<float4*>(hs + tl * KC * 32 + c * 32 + (((k / 4 % 8) ^ (c & 7)) << 2)) = hv;
    }
    __syncthreads();

    // piece p of chunk c sits at slot p ^ (c & 7), and c & 7 = lane & 7
    int ho[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) ho[p] = (p ^ (lane & 7)) << 2;
    for (int r0 = r_lo; r0 < r_hi; r0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u;  // unit: rows R r .. R r + R - 1 = t * H + j ..
            if (r < r_hi) {
                const int t = (R * r) >> hsh;
                const float* hrow = hs + (t - t_first) * KC * 32;
                float acc[R];
#pragma unroll
                for (int k = 0; k < R; ++k) acc[k] = 0.f;
#pragma unroll
                for (int i = 0; i < CPLD; ++i) {
                    const int g = u * CPLD + i;
                    const ItemRows<R> it = buf[g % kDDepth];
                    const int rn = r0 + (g + kDDepth) / CPLD;
                    if (rn < r_hi) buf[g % kDDepth] = load_at(rn, (g + kDDepth) % CPLD);
                    const int c = lane + 32 * i;
                    if (c < KC) dn_dot<R>(it, hrow + c * 32, ho, acc);
                    asm volatile("" ::: "memory");
                }
#pragma unroll
                for (int k = 0; k < R; ++k) {
                    const float v = warp_sum(acc[k]);
                    if (lane == 0) y[R * r + k] = v;
                }
            }
        }
    }
    if (!ok)  // malformed CSR: outputs unspecified, written as zero
        for (int i = blockIdx.x * kThD + threadIdx.x; i < T * H; i += gridDim.x * kThD) y[i] = 0.f;
}

size_t small_smem(int64_t bytes) { return static_cast<size_t>(bytes); }

template <int CPL, int NT>
cudaError_t launch_gu(cudaLaunchConfig_t& cfg, int dev, const float* logits, const int32_t* offsets,
                      const int32_t* pair_token, const float* pair_weight, const int32_t* pair_slot,
                      const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts, const uint16_t* x,
                      const float* dn_ts, const MoeWorkspace& ws, int E, int I, int T, int topk)
{
    auto kern = moe_small_gu_kernel<CPL, NT>;
    static OccCache occ;
    cfg.dynamicSmemBytes = small_smem(static_cast<int64_t>(T) * 1024 * CPL * 4);
    cfg.blockDim = dim3(kThG);
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kThG, cfg.dynamicSmemBytes);
    return cudaLaunchKernelEx(&cfg, kern, logits, offsets, pair_token, pair_weight, pair_slot, gu_codes, gu_scales,
                              gu_ts, x, dn_ts, ws, E, I, T, topk);
}

template <int CPLD, int CS, int R>
cudaError_t launch_dn_r(cudaLaunchConfig_t& cfg, int dev, const uint8_t* dn_codes, const uint8_t* dn_scales,
                        float* y, const MoeWorkspace& ws, int H, int T, int topk)
{
    auto kern = moe_small_dn_kernel<CPLD, CS, R>;
    static OccCache occ;
    // a CTA's rows span at most rows_per_cta / H + 2 tokens
    const int64_t rows_per_cta = (static_cast<int64_t>(T) * H + cfg.gridDim.x - 1) / cfg.gridDim.x;
    int64_t tok = rows_per_cta / H + 2;
    if (tok > T) tok = T;
    cfg.dynamicSmemBytes = small_smem(tok * topk * 32 * CS * 4);
    cfg.blockDim = dim3(kThD);
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kThD, cfg.dynamicSmemBytes);
    return cudaLaunchKernelEx(&cfg, kern, dn_codes, dn_scales, y, ws, H, T, topk);
}

// Two rows per warp unit halve the shared-memory reads of h' once there are
// at least as many row pairs as warps (T = 16 with H = 2048: 53.2 against
// 54.8 us a layer back to back); below that, single rows keep more warps
// streaming (T = 1: 15.2 against 16.7 us).
template <int CPLD, int CS>
cudaError_t launch_dn(cudaLaunchConfig_t& cfg, int dev, const uint8_t* dn_codes, const uint8_t* dn_scales, float* y,
                      const MoeWorkspace& ws, int H, int T, int topk)
{
    if (CPLD <= 4 && static_cast<int64_t>(T) * H / 2 >= static_cast<int64_t>(cfg.gridDim.x) * kWpD)
        return launch_dn_r<CPLD, CS, (CPLD <= 4 ? 2 : 1)>(cfg, dev, dn_codes, dn_scales, y, ws, H, T, topk);
    return launch_dn_r<CPLD, CS, 1>(cfg, dev, dn_codes, dn_scales, y, ws, H, T, topk);
}

}  // namespace

bool moe_small_supported(int E, int H, int I, int T, int topk)
{
    const bool h_ok = H == 1024 || H == 2048 || H == 4096 || H == 8192;
    const bool i_ok = I == 256 || I == 512 || I == 1024;
    // h' of all pairs lives in the workspace's partial-output area (P * I <=
    // P * H; the support set keeps H >= 2I); a gathered down row is at most
    // 8 * 1024 elements; the staged activations (T * H f16) at most 64 KiB
    return T >= 1 && T <= kMaxT && T * topk <= kMaxP && topk <= kWarp && E >= 1 && E <= kMaxE && h_ok && i_ok &&
           H >= 2 * I && topk * I <= 8192 && T * H <= kMaxTH;
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
    cfg.blockDim = dim3(kThG);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;

    // rows for one or two tokens, tensor-core tiles (token groups of up to
    // eight) from three on
    const int nt = T == 1 ? 1 : (T == 2 ? 2 : 8);
#define BQD_GU1(CPL_, NT_)                                                                                            \
    launch_gu<CPL_, NT_>(cfg, dev, logits, offsets, pair_token, pair_weight, pair_slot, gu_codes, gu_scales, gu_ts, x, \
                         dn_ts, ws, E, I, T, topk)
#define BQD_GU(CPL_) (nt == 1 ? BQD_GU1(CPL_, 1) : (nt == 2 ? BQD_GU1(CPL_, 2) : BQD_GU1(CPL_, 8)))
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
    (I == 256   ? launch_dn<CPLD_, 8>(cfg, dev, dn_codes, dn_scales, y, ws, H, T, topk)                               \
     : I == 512 ? launch_dn<CPLD_, 16>(cfg, dev, dn_codes, dn_scales, y, ws, H, T, topk)                              \
                : launch_dn<CPLD_, 32>(cfg, dev, dn_codes, dn_scales, y, ws, H, T, topk))
    switch (cpld) {
        case 1: return BQD_DN(1);
        case 2: return BQD_DN(2);
        case 4: return BQD_DN(4);
        default: return BQD_DN(8);
    }
#undef BQD_DN
}

cudaError_t read_and_clear_moe_small_error(unsigned int* out)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_moe_small_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *out = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_moe_small_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace bqd
