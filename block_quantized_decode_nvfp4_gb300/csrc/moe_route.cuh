// moe_route.cuh -- the router of the top-k routed MoE layer, one token per
// warp ("robertbfuentes7-cloud/bw24" README, MoE bullet; the routing rule is
// the workload's: softmax over the experts' logits, keep the topk largest,
// renormalise the kept probabilities).
//
// Shared by the route kernel (moe.cu) and the small-batch MoE kernels
// (moe_small.cu), which route inside every CTA, so that both pick the same
// experts with bit-identical weights.
#pragma once

#include <climits>
#include <cmath>
#include <cstdint>

#include "common.cuh"

namespace bqd {

// Top-k of one token by repeated warp argmax over its E logits (global
// memory, row `logits`): the larger logit first, the lower expert index on
// equal logits; when only NaN logits are left, the lowest index not yet
// taken. Lane l keeps the logits of experts l + 32 j (j < NJ, NJ * 32 >= E)
// in registers and a bit per taken expert. Each round a lane picks its own
// best, then two warp reductions pick the warp's: the largest order-
// preserving key (NaN lowest, -0 counted as +0 so that equal values tie)
// and, among the lanes holding it, the lowest expert index. The weights are
// the softmax of the selected logits (equal to the full softmax renormalised
// over them). Lane s < topk receives the slot-s expert in *e_out and its
// weight in *w_out; topk <= 32. Warp-collective.
__device__ __forceinline__ uint32_t order_key(float v)
{
    if (v != v) return 0u;  // NaN: below every number
    const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int NJ>
__device__ __forceinline__ void route_token_warp(const float* __restrict__ logits, int E, int topk, int lane,
                                                 int* e_out, float* w_out)
{
    float v[NJ];
    uint32_t key[NJ];
    uint32_t taken = 0;  // bit j: expert lane + 32 j is taken (or does not exist)
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const bool in = lane + 32 * j < E;
        v[j] = in ? logits[lane + 32 * j] : 0.f;
        key[j] = order_key(v[j]);
        if (!in) taken |= 1u << j;
    }
    int my_e = 0;
    float my_l = 0.f, lmax = 0.f;
    for (int s = 0; s < topk; ++s) {
        uint32_t bk = 0u;
        int be = INT_MAX;
        float bv = 0.f;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            if (!((taken >> j) & 1u) && (key[j] > bk || (key[j] == bk && e < be))) {
                bk = key[j];
                be = e;
                bv = v[j];
            }
        }
        const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, bk);
        const int we = __reduce_min_sync(0xFFFFFFFFu, bk == wk ? be : INT_MAX);
        const float wv = __shfl_sync(0xFFFFFFFFu, bv, we & 31);
        if ((we & 31) == lane) taken |= 1u << (we >> 5);
        if (lane == s) {
            my_e = we;
            my_l = wv;
        }
        if (s == 0) lmax = wv;
    }
    const float ex = lane < topk ? expf(my_l - lmax) : 0.f;
    const float z = warp_sum(ex);
    *e_out = my_e;
    *w_out = ex / z;
}

// route_token_warp for any E <= 1024 (the register count rounded up to a
// power of two).
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int E, int topk, int lane, int* e_out,
                                            float* w_out)
{
    if (E <= 64)
        route_token_warp<2>(logits, E, topk, lane, e_out, w_out);
    else if (E <= 128)
        route_token_warp<4>(logits, E, topk, lane, e_out, w_out);
    else if (E <= 256)
        route_token_warp<8>(logits, E, topk, lane, e_out, w_out);
    else if (E <= 512)
        route_token_warp<16>(logits, E, topk, lane, e_out, w_out);
    else
        route_token_warp<32>(logits, E, topk, lane, e_out, w_out);
}

}  // namespace bqd
