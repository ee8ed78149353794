// moe_prefill.cu -- a routed MoE layer for many tokens (prefill) around the
// grouped tensor-core GEMM: the pages' grouped-MoE prefill with a per-expert
// variable-grid NVFP4 GEMM ("Vemloir/LumenLLM" README, Kernels bullet;
// "robertbfuentes7-cloud/bw24" README, MoE bullet: experts decoded once for
// all their tokens).
//
// The layer computes what the small-batch and stream paths compute (softmax
// top-k routing, h = SiLU(gate) * up per (token, slot), y_t = sum over the
// slots of w * (W_dn . h), slots added in order 0 .. topk - 1):
//  1. routing in three kernels that spread the tokens over the GPU: every
//     token's top-k (route_token, the same selection and weights as the
//     decode router) with per-block expert counts; one CTA turning the
//     counts into the CSR offsets and each block's cursors; every block
//     placing its pairs. The list is the decode router's: expert-major,
//     tokens ascending within an expert;
//  2. a gather copies every pair's token row, expert-major, and records the
//     pair of each (token, slot);
//  3. the grouped GEMM gives gate and up of every pair: G [P][2I];
//  4. h = SiLU(g) * u in fp32, split into two bf16 parts hi = bf16(h) and
//     lo = bf16(h - hi), whose sum holds h to ~2^-17 of its size (a single
//     bf16 operand would round h by up to 2^-9, beyond the tolerance),
//     stored side by side: HL [P][2I] = [hi | lo];
//  5. one grouped GEMM of W_dn, its k repeated twice, with HL:
//     D [P][H] = W_dn . hi + W_dn . lo;
//  6. the combine adds each token's slots in order, weighted.
// Every product inside the GEMMs is exact; the sums are fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "gemm.h"
#include "gemv.h"
#include "moe_route.cuh"

namespace bqd {

namespace {

constexpr size_t al256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

constexpr int kRouteThreads = 256;   // eight warps, a token each at a time
constexpr int kScanThreads = 1024;   // >= the largest E
constexpr int kScanBatch = 8;        // block counts loaded together by the scan

// Tokens per routing block: 8 (a token per warp) up to 1024 tokens, then a
// multiple of 8 that keeps the blocks at most 128 (64 at T = 8192).
int route_block_tokens(int T)
{
    const int per = (T + 127) / 128;
    return per <= 8 ? 8 : (per + 7) / 8 * 8;
}
int route_blocks(int T) { return (T + route_block_tokens(T) - 1) / route_block_tokens(T); }

struct PrefillWs {
    int32_t *offsets, *pair_token, *pair_slot, *inv, *sel_e, *blk_cnt;
    float *pair_weight, *sel_w;
    uint16_t *xg, *hl;
    float *gu, *d;
};

PrefillWs carve(void* base, int T, int topk, int H, int I, int E, size_t* total)
{
    const size_t P = static_cast<size_t>(T) * topk;
    uint8_t* p = static_cast<uint8_t*>(base);
    size_t o = 0;
    PrefillWs w{};
    auto take = [&](size_t bytes) {
        uint8_t* r = p ? p + o : nullptr;
        o += al256(bytes);
        return r;
    };
    w.offsets = reinterpret_cast<int32_t*>(take((static_cast<size_t>(E) + 1) * 4));
    w.pair_token = reinterpret_cast<int32_t*>(take(P * 4));
    w.pair_weight = reinterpret_cast<float*>(take(P * 4));
    w.pair_slot = reinterpret_cast<int32_t*>(take(P * 4));
    w.inv = reinterpret_cast<int32_t*>(take(P * 4));
    w.sel_e = reinterpret_cast<int32_t*>(take(P * 4));
    w.sel_w = reinterpret_cast<float*>(take(P * 4));
    w.blk_cnt = reinterpret_cast<int32_t*>(take(static_cast<size_t>(route_blocks(T)) * E * 4));
    w.xg = reinterpret_cast<uint16_t*>(take(P * H * 2));
    w.gu = reinterpret_cast<float*>(take(P * 2 * I * 4));
    w.hl = reinterpret_cast<uint16_t*>(take(P * 2 * I * 2));
    w.d = reinterpret_cast<float*>(take(P * H * 4));
    if (total) *total = o;
    return w;
}

// Routing, pass 1: block b's tokens [tb b, tb b + tb), a warp per token:
// slot s of token t goes to sel_e/sel_w[t * topk + s]; blk_cnt[b][e] counts
// the block's pairs of expert e.
__global__ void __launch_bounds__(kRouteThreads)
    route_select_kernel(const float* __restrict__ logits, int T, int E, int topk, int tb,
                        int32_t* __restrict__ sel_e, float* __restrict__ sel_w, int32_t* __restrict__ blk_cnt)
{
    extern __shared__ int s_cnt[];  // [E]
    for (int e = threadIdx.x; e < E; e += kRouteThreads) s_cnt[e] = 0;
    __syncthreads();
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    const int t0 = blockIdx.x * tb, t1 = min(T, t0 + tb);
    for (int t = t0 + warp; t < t1; t += kRouteThreads / kWarp) {  // warp-uniform
        int e = 0;
        float w = 0.f;
        route_token(logits + static_cast<int64_t>(t) * E, E, topk, lane, &e, &w);
        if (lane < topk) {  // e < E: route_token picks untaken experts only, and topk <= E
            sel_e[t * topk + lane] = e;
            sel_w[t * topk + lane] = w;
            atomicAdd(&s_cnt[e], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kRouteThreads) blk_cnt[static_cast<int64_t>(blockIdx.x) * E + e] = s_cnt[e];
}

// Routing, pass 2 (one CTA, thread e per expert, E <= 1024): blk_cnt[b][e]
// becomes the number of expert e's pairs in blocks before b, and offsets the
// exclusive scan of the experts' totals (offsets[E] = P).
__global__ void __launch_bounds__(kScanThreads)
    route_scan_kernel(int32_t* __restrict__ blk_cnt, int nb, int E, int P, int32_t* __restrict__ offsets)
{
    __shared__ int s_warp[kScanThreads / kWarp];
    const int e = threadIdx.x, lane = e % kWarp, warp = e / kWarp;
    int tot = 0;
    if (e < E) {
        for (int b0 = 0; b0 < nb; b0 += kScanBatch) {  // the loads of a batch in flight together
            int c[kScanBatch];
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j)
                c[j] = b0 + j < nb ? blk_cnt[static_cast<int64_t>(b0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < kScanBatch; ++j) {
                if (b0 + j < nb) blk_cnt[static_cast<int64_t>(b0 + j) * E + e] = tot;
                tot += c[j];
            }
        }
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == kWarp - 1) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = s_warp[lane], vi = v;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, vi, o);
            if (lane >= o) vi += n;
        }
        s_warp[lane] = vi - v;  // exclusive prefix of the warps' totals
    }
    __syncthreads();
    if (e < E) offsets[e] = s_warp[warp] + incl - tot;
    if (e == 0) offsets[E] = P;
}

// Routing, pass 3: one warp per block writes the block's pairs, token by
// token in order, at its experts' cursors (offsets[e] + blk_cnt[b][e]); a
// token's experts are distinct, so its lanes never share a cursor.
__global__ void __launch_bounds__(kWarp)
    route_place_kernel(const int32_t* __restrict__ sel_e, const float* __restrict__ sel_w,
                       const int32_t* __restrict__ blk_cnt, const int32_t* __restrict__ offsets, int T, int E,
                       int topk, int tb, int P, int32_t* __restrict__ pair_token, float* __restrict__ pair_weight,
                       int32_t* __restrict__ pair_slot)
{
    extern __shared__ int s_cur[];  // [E] cursors, then the block's sel_e and sel_w [tb * topk] each
    int* s_sel = s_cur + E;
    float* s_w = reinterpret_cast<float*>(s_sel + tb * topk);
    const int lane = threadIdx.x, b = blockIdx.x;
    const int t0 = b * tb, t1 = min(T, t0 + tb);
    for (int e = lane; e < E; e += kWarp) s_cur[e] = offsets[e] + blk_cnt[static_cast<int64_t>(b) * E + e];
    for (int i = lane; i < (t1 - t0) * topk; i += kWarp) {
        s_sel[i] = sel_e[t0 * topk + i];
        s_w[i] = sel_w[t0 * topk + i];
    }
    __syncwarp();
    for (int t = t0; t < t1; ++t) {
        if (lane < topk) {
            const int e = s_sel[(t - t0) * topk + lane];
            const int pos = s_cur[e];
            s_cur[e] = pos + 1;
            if (pos >= 0 && pos < P) {  // always, as both passes read the same selection; keeps writes in bounds
                pair_token[pos] = t;
                pair_slot[pos] = lane;
                pair_weight[pos] = s_w[(t - t0) * topk + lane];
            }
        }
        __syncwarp();
    }
}

// Pair p's token row, 16 bytes per thread; and inv[(token, slot)] = p.
__global__ void gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ pair_token,
                              const int32_t* __restrict__ pair_slot, uint16_t* __restrict__ xg,
                              int32_t* __restrict__ inv, int P, int H, int T, int topk)
{
    const int per = H / 8;  // 16-byte pieces a row
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < static_cast<int64_t>(P) * per;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int p = static_cast<int>(i / per), c = static_cast<int>(i % per);
        const int t = min(max(pair_token[p], 0), T - 1);
        reinterpret_cast<uint4*>(xg)[i] = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H)[c];
        if (c == 0) {
            const int s = pair_slot[p];
            if (pair_token[p] >= 0 && pair_token[p] < T && s >= 0 && s < topk) inv[pair_token[p] * topk + s] = p;
        }
    }
}

// h = SiLU(g) * u, g = G[p][i], u = G[p][I + i]; HL[p][i] = bf16(h),
// HL[p][I + i] = bf16(h - bf16(h)).
__global__ void silu_split_kernel(const float* __restrict__ gu, uint16_t* __restrict__ hl, int P, int I)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < static_cast<int64_t>(P) * I;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t p = i / I, k = i % I;
        const float g = gu[p * 2 * I + k], u = gu[p * 2 * I + I + k];
        const float h = g / (1.0f + expf(-g)) * u;
        const __nv_bfloat16 hi = __float2bfloat16_rn(h);
        const __nv_bfloat16 lo = __float2bfloat16_rn(h - __bfloat162float(hi));
        hl[p * 2 * I + k] = __bfloat16_as_ushort(hi);
        hl[p * 2 * I + I + k] = __bfloat16_as_ushort(lo);
    }
}

// y[t][j] = sum over s = 0 .. topk - 1 of w(t, s) * D[pair(t, s)][j].
__global__ void combine_kernel(const float* __restrict__ d, const float* __restrict__ pair_weight,
                               const int32_t* __restrict__ inv, float* __restrict__ y, int T, int H, int topk, int P)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < static_cast<int64_t>(T) * H;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / H, j = i % H;
        float acc = 0.f;
        for (int s = 0; s < topk; ++s) {
            const int p = inv[t * topk + s];  // every (token, slot) has one pair; the check keeps reads in bounds
            if (p >= 0 && p < P) acc += pair_weight[p] * d[static_cast<int64_t>(p) * H + j];
        }
        y[i] = acc;
    }
}

unsigned grid_for(int64_t work)
{
    int64_t g = (work + 255) / 256;
    if (g > 152 * 8) g = 152 * 8;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

}  // namespace

size_t moe_prefill_workspace_size(int T, int topk, int H, int I, int E)
{
    size_t total = 0;
    carve(nullptr, T, topk, H, I, E, &total);
    return total;
}

cudaError_t launch_moe_prefill_layer(const float* logits, const uint8_t* gu_codes, const uint8_t* gu_scales,
                                     const float* gu_ts, const uint8_t* dn_codes, const uint8_t* dn_scales,
                                     const float* dn_ts, const uint16_t* x, float* y, void* ws, int E, int H, int I,
                                     int T, int topk, cudaStream_t s)
{
    const int P = T * topk;
    const PrefillWs w = carve(ws, T, topk, H, I, E, nullptr);
    const int tb = route_block_tokens(T), nb = route_blocks(T);
    route_select_kernel<<<nb, kRouteThreads, static_cast<size_t>(E) * 4, s>>>(logits, T, E, topk, tb, w.sel_e,
                                                                             w.sel_w, w.blk_cnt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    route_scan_kernel<<<1, kScanThreads, 0, s>>>(w.blk_cnt, nb, E, P, w.offsets);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    route_place_kernel<<<nb, kWarp, (static_cast<size_t>(E) + 2 * static_cast<size_t>(tb) * topk) * 4, s>>>(
        w.sel_e, w.sel_w, w.blk_cnt, w.offsets, T, E, topk, tb, P, w.pair_token, w.pair_weight, w.pair_slot);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    gather_kernel<<<grid_for(static_cast<int64_t>(P) * H / 8), 256, 0, s>>>(x, w.pair_token, w.pair_slot, w.xg,
                                                                            w.inv, P, H, T, topk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = launch_nvfp4_gemm_grouped(gu_codes, gu_scales, gu_ts, w.offsets, E, w.xg, w.gu, 2 * static_cast<int64_t>(I),
                                  H, P, s);
    if (e != cudaSuccess) return e;
    silu_split_kernel<<<grid_for(static_cast<int64_t>(P) * I), 256, 0, s>>>(w.gu, w.hl, P, I);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = launch_nvfp4_gemm_grouped(dn_codes, dn_scales, dn_ts, w.offsets, E, w.hl, w.d, H, 2 * static_cast<int64_t>(I),
                                  P, s, false, I);
    if (e != cudaSuccess) return e;
    combine_kernel<<<grid_for(static_cast<int64_t>(T) * H), 256, 0, s>>>(w.d, w.pair_weight, w.inv, y, T, H, topk,
                                                                         P);
    return cudaGetLastError();
}

}  // namespace bqd
