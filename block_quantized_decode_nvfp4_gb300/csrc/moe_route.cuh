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
// in registers and a bit per taken expert. The weights are the softmax of
// the selected logits (equal to the full softmax renormalised over them).
// Lane s < topk receives the slot-s expert in *e_out and its weight in
// *w_out; topk <= 32. Warp-collective.
template <int NJ>
__device__ __forceinline__ void route_token_warp(const float* __restrict__ logits, int E, int topk, int lane,
                                                 int* e_out, float* w_out)
{
    float v[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) v[j] = lane + 32 * j < E ? logits[lane + 32 * j] : 0.f;
    uint32_t taken = 0;  // bit j: expert lane + 32 j is taken (or does not exist)
#pragma unroll
    for (int j = 0; j < NJ; ++j)
        if (lane + 32 * j >= E) taken |= 1u << j;
    int my_e = 0;
    float my_l = 0.f, lmax = 0.f;
    for (int s = 0; s < topk; ++s) {
        float bv = -INFINITY;
        int be = INT_MAX;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            if (!((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < be))) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if (be == INT_MAX) {  // only NaN logits left: take the lowest free index
            int fe = INT_MAX;
#pragma unroll
            for (int j = 0; j < NJ; ++j)
                if (!((taken >> j) & 1u) && lane + 32 * j < fe) fe = lane + 32 * j;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) fe = min(fe, __shfl_xor_sync(0xFFFFFFFFu, fe, o));
            be = fe;
            float own = 0.f;
#pragma unroll
            for (int j = 0; j < NJ; ++j)
                if (lane + 32 * j == be) own = v[j];
            bv = __shfl_sync(0xFFFFFFFFu, own, be & 31);
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == s) {
            my_e = be;
            my_l = bv;
        }
        if (s == 0) lmax = bv;
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
