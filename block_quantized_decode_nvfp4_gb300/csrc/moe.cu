// moe.cu -- top-k routed MoE layer on NVFP4 experts for decode (sm_103a).
//
// What is computed ("robertbfuentes7-cloud/bw24" README, MoE bullet: routed
// tokens batched expert-major, every selected expert's weights decoded once
// for all of its tokens; the routing rule and the SiLU(gate) * up activation
// are the workload's):
//   router:  p = softmax(logits[t]); keep the topk largest; w = p / sum(kept)
//   list:    (token, slot) pairs grouped by expert (CSR offsets), tokens in
//            increasing order inside an expert
//   gate_up: g = W_gu[e][0:I] . x_t, u = W_gu[e][I:2I] . x_t, h = SiLU(g) * u
//   down:    d = W_dn[e] . h
//   combine: y_t = sum over slots s = 0..topk-1 (in that order) of w_s * d_s
//
// Kernels: one route kernel (a single CTA builds the list without atomics on
// global memory), a gate_up kernel and a down kernel whose CTAs each take one
// active expert and a slice of its rows (an expert's rows are streamed once
// for all of its tokens), and a combine kernel with a fixed summation order.
// The result is deterministic run to run.
//
// Device-side faults in a caller-supplied list set bits in the workspace's
// status word (never a trap): 1 = offsets not a valid CSR, 2 = a token or
// slot id out of range, 4 = a (token, slot) produced zero or several times.
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

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
constexpr int kStatusBadOffsets = 1;
constexpr int kStatusBadPair = 2;
constexpr int kStatusCoverage = 4;

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// Exclusive prefix sum over the CTA (kThreads threads); scratch holds
// kWarps + 1 ints. Returns the exclusive prefix; *total gets the sum.
__device__ int block_exclusive_scan(int v, int* scratch, int* total)
{
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    int incl = v;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == kWarp - 1) scratch[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int c = scratch[w];
            scratch[w] = run;
            run += c;
        }
        scratch[kWarps] = run;
    }
    __syncthreads();
    const int r = scratch[warp] + incl - v;
    *total = scratch[kWarps];
    __syncthreads();
    return r;
}

// ------------------------------------------------------------------ route
// One CTA. Warp w routes tokens [T*w/8, T*(w+1)/8) with route_token
// (moe_route.cuh): top-k by repeated warp argmax over logits held in
// registers, weights as the softmax of the selected logits (equal to
// renormalising the full softmax).
// Then a counting sort by expert: per-warp counts, a CTA-wide scan, and each
// warp placing its own tokens in order, so a segment lists tokens ascending.
__global__ void __launch_bounds__(kThreads) moe_route_kernel(const float* __restrict__ logits, int T, int E,
                                                             int topk, int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ pair_token,
                                                             float* __restrict__ pair_weight,
                                                             int32_t* __restrict__ pair_slot)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int P = T * topk;
    int* wc = reinterpret_cast<int*>(smem);               // [kWarps][E] counts, then write cursors
    int* sel_e = wc + kWarps * E;                         // [P]
    float* sel_w = reinterpret_cast<float*>(sel_e + P);   // [P]
    int* scratch = reinterpret_cast<int*>(sel_w + P);     // [kWarps + 1]

    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    for (int i = threadIdx.x; i < kWarps * E; i += kThreads) wc[i] = 0;
    __syncthreads();

    const int t_lo = static_cast<int>(static_cast<int64_t>(T) * warp / kWarps);
    const int t_hi = static_cast<int>(static_cast<int64_t>(T) * (warp + 1) / kWarps);
    int* cnt = wc + warp * E;
    for (int t = t_lo; t < t_hi; ++t) {
        int my_e = 0;
        float my_w = 0.f;
        route_token(logits + static_cast<int64_t>(t) * E, E, topk, lane, &my_e, &my_w);
        if (lane < topk) {
            sel_e[t * topk + lane] = my_e;
            sel_w[t * topk + lane] = my_w;
            cnt[my_e] += 1;  // the topk experts of one token are distinct
        }
        __syncwarp();
    }
    __syncthreads();

    // CSR offsets: each thread owns a run of consecutive experts.
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = threadIdx.x * per;
    int mine = 0;
    for (int e = e0; e < e0 + per && e < E; ++e)
        for (int w = 0; w < kWarps; ++w) mine += wc[w * E + e];
    int total = 0;
    int run = block_exclusive_scan(mine, scratch, &total);
    for (int e = e0; e < e0 + per && e < E; ++e) {
        offsets[e] = run;
        for (int w = 0; w < kWarps; ++w) {  // counts -> per-warp write cursors
            const int c = wc[w * E + e];
            wc[w * E + e] = run;
            run += c;
        }
    }
    if (threadIdx.x == 0) offsets[E] = P;
    __syncthreads();

    for (int t = t_lo; t < t_hi; ++t) {
        if (lane < topk) {
            const int e = sel_e[t * topk + lane];
            const int pos = cnt[e];
            cnt[e] = pos + 1;
            pair_token[pos] = t;
            pair_slot[pos] = lane;
            pair_weight[pos] = sel_w[t * topk + lane];
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------------ helpers
// The expert of active-expert index `a` (experts with a non-empty segment,
// in increasing order), or -1. Reads offsets[0..E]. CTA-wide.
__device__ int find_active_expert(const int32_t* __restrict__ offsets, int E, int a, int* scratch)
{
    __shared__ int s_e;
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = threadIdx.x * per;
    int mine = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) mine += offsets[e + 1] > offsets[e] ? 1 : 0;
    if (threadIdx.x == 0) s_e = -1;
    int total = 0;
    int run = block_exclusive_scan(mine, scratch, &total);
    if (a < total && a >= run && a < run + mine) {
        for (int e = e0; e < e0 + per && e < E; ++e) {
            if (offsets[e + 1] > offsets[e]) {
                if (run == a) s_e = e;
                ++run;
            }
        }
    }
    __syncthreads();
    return s_e;
}

// CTA (0,0) of the gate_up kernel checks the CSR and clears the per-(token,
// slot) counters and weights the later kernels fill.
__device__ void moe_validate_and_clear(const int32_t* __restrict__ offsets, int E, int P, const MoeWorkspace& ws)
{
    bool bad = false;
    for (int e = threadIdx.x; e < E; e += kThreads)
        if (offsets[e + 1] < offsets[e]) bad = true;
    if (threadIdx.x == 0 && (offsets[0] != 0 || offsets[E] != P)) bad = true;
    if (bad) atomicOr(ws.status, kStatusBadOffsets);
    for (int i = threadIdx.x; i < P; i += kThreads) {
        ws.count[i] = 0;
        ws.wts[i] = 0.f;
    }
}

// ------------------------------------------------------------------ gate_up
// Row pointers of PAIRS (gate, up) pairs starting at pair ib of an expert's
// gate_up weight: slots (2p, 2p+1) = rows (ib+p, I+ib+p). Returns the number
// of valid pairs; unused slots repeat a valid row.
template <int PAIRS>
__device__ __forceinline__ int pair_rows(const uint8_t* codes_e, const uint8_t* scales_e, int64_t cpitch,
                                         int64_t spitch, int I, int ib, int i_hi, const uint8_t* (&crow)[2 * PAIRS],
                                         const uint8_t* (&srow)[2 * PAIRS])
{
    const int npairs = ib >= i_hi ? 0 : (i_hi - ib >= PAIRS ? PAIRS : i_hi - ib);
#pragma unroll
    for (int r = 0; r < 2 * PAIRS; ++r) {
        const int pr = r / 2 < npairs ? r / 2 : 0;
        const int64_t row = (r % 2 == 0 ? 0 : I) + (npairs ? ib + pr : 0);
        crow[r] = codes_e + row * cpitch;
        srow[r] = scales_e + row * spitch;
    }
    return npairs;
}

// Row pointers of RPW consecutive rows starting at jb (< j_hi valid).
template <int RPW>
__device__ __forceinline__ int block_rows(const uint8_t* codes_e, const uint8_t* scales_e, int64_t cpitch,
                                          int64_t spitch, int jb, int j_hi, const uint8_t* (&crow)[RPW],
                                          const uint8_t* (&srow)[RPW])
{
    const int nrows = jb >= j_hi ? 0 : (j_hi - jb >= RPW ? RPW : j_hi - jb);
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int64_t row = nrows ? jb + (r < nrows ? r : 0) : 0;
        crow[r] = codes_e + row * cpitch;
        srow[r] = scales_e + row * spitch;
    }
    return nrows;
}

// Rows of one expert's gate_up weight against NC staged token columns. The
// first row group's loads are issued before `stage` fills the activations
// (CTA-wide, followed by a barrier), so that staging hides under HBM latency.
template <int LG, int NC, class Stage>
__device__ __forceinline__ void gate_up_rows(const uint8_t* codes_e, const uint8_t* scales_e, float ts, int H, int I,
                                             int i_lo, int i_hi, const float* xs, int g0, int ng, float* h_ws,
                                             Stage stage)
{
    constexpr int PAIRS = NC <= 4 ? 2 : 1;      // (gate, up) row pairs per lane group
    constexpr int RPW = 2 * PAIRS;
    constexpr int kGroups = kWarp / LG;          // lane groups per warp
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    const int grp = lane / LG, g = lane % LG;
    const int64_t cpitch = H / 2, spitch = H / 16;
    const int chunks = H / Nvfp4Vec::kElems;
    const int mine = (warp * kGroups + grp) * PAIRS;
    const int step = kWarps * kGroups * PAIRS;
    RowStream<Nvfp4Vec, RPW, 2, LG> rs;
    const uint8_t* crow[RPW];
    const uint8_t* srow[RPW];
    int npairs = pair_rows<PAIRS>(codes_e, scales_e, cpitch, spitch, I, i_lo + mine, i_hi, crow, srow);
    if (npairs) rs.start(crow, srow, 0, chunks, g);
    stage();
    __syncthreads();
    for (int ib = i_lo + mine; ib - mine < i_hi; ib += step) {
        if (ib != i_lo + mine) {
            npairs = pair_rows<PAIRS>(codes_e, scales_e, cpitch, spitch, I, ib, i_hi, crow, srow);
            if (npairs) rs.start(crow, srow, 0, chunks, g);
        }
        float2 acc[RPW][NC];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[r][n] = make_float2(0.f, 0.f);
        if (npairs) rs.template run<NC>(xs, H, acc);
#pragma unroll
        for (int p = 0; p < PAIRS; ++p)
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float gs = group_sum<LG>(acc[2 * p][n].x + acc[2 * p][n].y) * ts;
                const float us = group_sum<LG>(acc[2 * p + 1][n].x + acc[2 * p + 1][n].y) * ts;
                if (g == n && n < ng && p < npairs) {
                    const float hv = gs / (1.0f + expf(-gs)) * us;
                    h_ws[static_cast<int64_t>(g0 + n) * I + ib + p] = hv;
                }
            }
    }
}

template <int LG, int NCG>
__global__ void __launch_bounds__(kThreads, 1) moe_gate_up_kernel(
    const uint8_t* __restrict__ gu_codes, const uint8_t* __restrict__ gu_scales, const float* __restrict__ gu_ts,
    const uint16_t* __restrict__ x, const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_token,
    MoeWorkspace ws, int E, int H, int I, int T, int topk)
{
    extern __shared__ __align__(16) float xs[];  // [NCG][H]
    __shared__ int scratch[kWarps + 1];
    const int P = T * topk;
    if (blockIdx.x == 0 && blockIdx.y == 0) moe_validate_and_clear(offsets, E, P, ws);
    const int e = find_active_expert(offsets, E, blockIdx.x, scratch);
    if (e < 0) return;
    const int p0 = offsets[e], p1 = offsets[e + 1];
    if (p0 < 0 || p1 > P || p0 > p1) {
        if (threadIdx.x == 0) atomicOr(ws.status, kStatusBadOffsets);
        return;
    }
    const int i_lo = static_cast<int>(static_cast<int64_t>(I) * blockIdx.y / gridDim.y);
    const int i_hi = static_cast<int>(static_cast<int64_t>(I) * (blockIdx.y + 1) / gridDim.y);
    const uint8_t* codes_e = gu_codes + static_cast<int64_t>(e) * 2 * I * (H / 2);
    const uint8_t* scales_e = gu_scales + static_cast<int64_t>(e) * 2 * I * (H / 16);
    const float ts = gu_ts[e];
    for (int g0 = p0; g0 < p1; g0 += NCG) {
        const int ng = p1 - g0 < NCG ? p1 - g0 : NCG;
        __syncthreads();
        auto stage = [&]() {
            // the ng token columns, 8 bf16 per 16-byte load; columns past ng
            // are never written back, so they are left unstaged
            const int vecs = H / 8;
            for (int i = threadIdx.x; i < ng * vecs; i += kThreads) {
                const int n = i / vecs, v = i - n * vecs;
                const int t = pair_token[g0 + n];
                uint4 u = make_uint4(0, 0, 0, 0);
                if (t >= 0 && t < T)
                    u = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * H + 8 * v);
                else if (v == 0)
                    atomicOr(ws.status, kStatusBadPair);
                put_piece<Nvfp4Vec>(xs + n * H, 2 * v, make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y)));
                put_piece<Nvfp4Vec>(xs + n * H, 2 * v + 1,
                                    make_float4(bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)));
            }
        };
        if (ng == 1)
            gate_up_rows<LG, 1>(codes_e, scales_e, ts, H, I, i_lo, i_hi, xs, g0, ng, ws.h, stage);
        else if (ng == 2)
            gate_up_rows<LG, 2>(codes_e, scales_e, ts, H, I, i_lo, i_hi, xs, g0, ng, ws.h, stage);
        else if (ng <= 4)
            gate_up_rows<LG, 4>(codes_e, scales_e, ts, H, I, i_lo, i_hi, xs, g0, ng, ws.h, stage);
        else
            gate_up_rows<LG, NCG>(codes_e, scales_e, ts, H, I, i_lo, i_hi, xs, g0, ng, ws.h, stage);
    }
}

// ------------------------------------------------------------------ down
template <int LG, int NC, class Stage>
__device__ __forceinline__ void down_rows(const uint8_t* codes_e, const uint8_t* scales_e, float ts, int H, int I,
                                          int j_lo, int j_hi, const float* xs, const int* slot_of, int ng,
                                          float* part, Stage stage)
{
    constexpr int RPW = NC <= 4 ? 4 : 2;
    constexpr int kGroups = kWarp / LG;
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    const int grp = lane / LG, g = lane % LG;
    const int64_t cpitch = I / 2, spitch = I / 16;
    const int chunks = I / Nvfp4Vec::kElems;
    const int mine = (warp * kGroups + grp) * RPW;
    const int step = kWarps * kGroups * RPW;
    RowStream<Nvfp4Vec, RPW, 2, LG> rs;
    const uint8_t* crow[RPW];
    const uint8_t* srow[RPW];
    int nrows = block_rows<RPW>(codes_e, scales_e, cpitch, spitch, j_lo + mine, j_hi, crow, srow);
    if (nrows) rs.start(crow, srow, 0, chunks, g);
    stage();
    __syncthreads();
    for (int jb = j_lo + mine; jb - mine < j_hi; jb += step) {
        if (jb != j_lo + mine) {
            nrows = block_rows<RPW>(codes_e, scales_e, cpitch, spitch, jb, j_hi, crow, srow);
            if (nrows) rs.start(crow, srow, 0, chunks, g);
        }
        float2 acc[RPW][NC];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[r][n] = make_float2(0.f, 0.f);
        if (nrows) rs.template run<NC>(xs, I, acc);
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                const float v = group_sum<LG>(acc[r][n].x + acc[r][n].y) * ts;
                if (g == n && n < ng && r < nrows && slot_of[n] >= 0)
                    part[static_cast<int64_t>(slot_of[n]) * H + jb + r] = v;
            }
    }
}

template <int LG>
__global__ void __launch_bounds__(kThreads, 1) moe_down_kernel(
    const uint8_t* __restrict__ dn_codes, const uint8_t* __restrict__ dn_scales, const float* __restrict__ dn_ts,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_token,
    const float* __restrict__ pair_weight, const int32_t* __restrict__ pair_slot, MoeWorkspace ws, int E, int H,
    int I, int T, int topk)
{
    constexpr int NCG = 8;
    extern __shared__ __align__(16) float xs[];  // [NCG][I]
    __shared__ int scratch[kWarps + 1];
    __shared__ int slot_of[NCG];  // flat (token * topk + slot) of each staged pair, -1 if invalid
    const int P = T * topk;
    const int e = find_active_expert(offsets, E, blockIdx.x, scratch);
    if (e < 0) return;
    const int p0 = offsets[e], p1 = offsets[e + 1];
    if (p0 < 0 || p1 > P || p0 > p1) return;  // reported by the gate_up kernel
    const int j_lo = static_cast<int>(static_cast<int64_t>(H) * blockIdx.y / gridDim.y);
    const int j_hi = static_cast<int>(static_cast<int64_t>(H) * (blockIdx.y + 1) / gridDim.y);
    const uint8_t* codes_e = dn_codes + static_cast<int64_t>(e) * H * (I / 2);
    const uint8_t* scales_e = dn_scales + static_cast<int64_t>(e) * H * (I / 16);
    const float ts = dn_ts[e];
    for (int g0 = p0; g0 < p1; g0 += NCG) {
        const int ng = p1 - g0 < NCG ? p1 - g0 : NCG;
        __syncthreads();
        auto stage = [&]() {
            if (threadIdx.x < NCG) {
                int flat = -1;
                if (static_cast<int>(threadIdx.x) < ng) {
                    const int t = pair_token[g0 + threadIdx.x], s = pair_slot[g0 + threadIdx.x];
                    if (t >= 0 && t < T && s >= 0 && s < topk) {
                        flat = t * topk + s;
                        if (blockIdx.y == 0) {
                            ws.wts[flat] = pair_weight[g0 + threadIdx.x];
                            atomicAdd(ws.count + flat, 1);
                        }
                    } else {
                        atomicOr(ws.status, kStatusBadPair);
                    }
                }
                slot_of[threadIdx.x] = flat;
            }
            const int vecs = I / 4;
            for (int i = threadIdx.x; i < ng * vecs; i += kThreads) {
                const int n = i / vecs, v = i - n * vecs;
                put_piece<Nvfp4Vec>(xs + n * I, v,
                                    reinterpret_cast<const float4*>(ws.h + static_cast<int64_t>(g0 + n) * I)[v]);
            }
        };
        if (ng == 1)
            down_rows<LG, 1>(codes_e, scales_e, ts, H, I, j_lo, j_hi, xs, slot_of, ng, ws.part, stage);
        else if (ng == 2)
            down_rows<LG, 2>(codes_e, scales_e, ts, H, I, j_lo, j_hi, xs, slot_of, ng, ws.part, stage);
        else if (ng <= 4)
            down_rows<LG, 4>(codes_e, scales_e, ts, H, I, j_lo, j_hi, xs, slot_of, ng, ws.part, stage);
        else
            down_rows<LG, 8>(codes_e, scales_e, ts, H, I, j_lo, j_hi, xs, slot_of, ng, ws.part, stage);
    }
}

// ------------------------------------------------------------------ combine
__global__ void __launch_bounds__(kThreads) moe_combine_kernel(MoeWorkspace ws, float* __restrict__ y, int H,
                                                               int topk)
{
    const int t = blockIdx.y;
    const int j = blockIdx.x * kThreads + threadIdx.x;
    if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < topk && ws.count[t * topk + threadIdx.x] != 1)
        atomicOr(ws.status, kStatusCoverage);
    if (j >= H) return;
    // slots in order 0..topk-1; loads of up to eight slots in flight at once
    float acc = 0.f;
    for (int s0 = 0; s0 < topk; s0 += 8) {
        int cnt[8];
        float wv[8], pv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int f = t * topk + s0 + i;
            const bool in = s0 + i < topk;
            cnt[i] = in ? ws.count[f] : 0;
            wv[i] = in ? ws.wts[f] : 0.f;
            pv[i] = in ? ws.part[static_cast<int64_t>(f) * H + j] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (cnt[i] > 0) acc = fmaf(wv[i], pv[i], acc);
    }
    y[static_cast<int64_t>(t) * H + j] = acc;
}

int lanes_for(int chunks) { return chunks >= 32 ? 32 : (chunks >= 16 ? 16 : 8); }

template <int LG, int NCG>
cudaError_t launch_gate_up(dim3 grid, size_t smem, cudaStream_t s, const uint8_t* c, const uint8_t* sc,
                           const float* ts, const uint16_t* x, const int32_t* off, const int32_t* pt,
                           const MoeWorkspace& ws, int E, int H, int I, int T, int topk)
{
    static OccCache occ;
    auto kern = moe_gate_up_kernel<LG, NCG>;
    int dev = 0;
    cudaGetDevice(&dev);
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kThreads, smem);  // sets the smem opt-in
    kern<<<grid, kThreads, smem, s>>>(c, sc, ts, x, off, pt, ws, E, H, I, T, topk);
    return cudaGetLastError();
}

template <int LG>
cudaError_t launch_down(dim3 grid, size_t smem, cudaStream_t s, const uint8_t* c, const uint8_t* sc, const float* ts,
                        const int32_t* off, const int32_t* pt, const float* pw, const int32_t* ps,
                        const MoeWorkspace& ws, int E, int H, int I, int T, int topk)
{
    static OccCache occ;
    auto kern = moe_down_kernel<LG>;
    int dev = 0;
    cudaGetDevice(&dev);
    blocks_per_sm(occ, reinterpret_cast<const void*>(kern), dev, kThreads, smem);
    kern<<<grid, kThreads, smem, s>>>(c, sc, ts, off, pt, pw, ps, ws, E, H, I, T, topk);
    return cudaGetLastError();
}

}  // namespace

size_t moe_workspace_size(int T, int topk, int H, int I)
{
    const size_t P = static_cast<size_t>(T) * topk;
    return 256 + align256(P * 4) + align256(P * 4) + align256(P * I * 4) + align256(P * H * 4);
}

MoeWorkspace moe_workspace_carve(void* base, int T, int topk, int H, int I)
{
    const size_t P = static_cast<size_t>(T) * topk;
    char* p = static_cast<char*>(base);
    MoeWorkspace ws;
    ws.status = reinterpret_cast<int32_t*>(p);
    p += 256;
    ws.count = reinterpret_cast<int32_t*>(p);
    p += align256(P * 4);
    ws.wts = reinterpret_cast<float*>(p);
    p += align256(P * 4);
    ws.h = reinterpret_cast<float*>(p);
    p += align256(P * I * 4);
    ws.part = reinterpret_cast<float*>(p);
    return ws;
}

cudaError_t launch_moe_route(const float* logits, int T, int E, int topk, int32_t* offsets, int32_t* pair_token,
                             float* pair_weight, int32_t* pair_slot, cudaStream_t s)
{
    const int P = T * topk;
    const size_t smem = static_cast<size_t>(kWarps) * E * 4 + static_cast<size_t>(P) * 8 + (kWarps + 1) * 4;
    static OccCache occ;
    int dev = 0;
    cudaGetDevice(&dev);
    blocks_per_sm(occ, reinterpret_cast<const void*>(moe_route_kernel), dev, kThreads, smem);
    moe_route_kernel<<<1, kThreads, smem, s>>>(logits, T, E, topk, offsets, pair_token, pair_weight, pair_slot);
    return cudaGetLastError();
}

cudaError_t launch_moe_grouped(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                               const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts,
                               const uint16_t* x, const int32_t* offsets, const int32_t* pair_token,
                               const float* pair_weight, const int32_t* pair_slot, float* y,
                               const MoeWorkspace& ws, int E, int H, int I, int T, int topk, cudaStream_t s)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int sms = dev_info(dev).sms;
    const int P = T * topk;
    const int max_active = P < E ? P : E;
    if (moe_small_supported(E, H, I, T, topk))  // writes the status word itself
        return launch_moe_small_layer(nullptr, gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x, offsets,
                                      pair_token, pair_weight, pair_slot, y, ws, E, H, I, T, topk, s);
    err = cudaMemsetAsync(ws.status, 0, sizeof(int32_t), s);
    if (err != cudaSuccess) return err;
    const dim3 grid_c((H + kThreads - 1) / kThreads, T);

    if (moe_stream_supported(E, H, I)) {
        err = launch_moe_stream_layer(gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x, offsets, pair_token,
                                      pair_weight, pair_slot, ws, E, H, I, T, topk, s);
        if (err != cudaSuccess) return err;
        moe_combine_kernel<<<grid_c, kThreads, 0, s>>>(ws, y, H, topk);
        return cudaGetLastError();
    }

    // gate_up: one CTA per (active expert, slice of its I row pairs)
    int gy = (2 * sms + max_active - 1) / max_active;
    if (gy > I / 2) gy = I / 2;
    if (gy < 1) gy = 1;
    const int ncg_a = H <= 4096 ? 8 : 4;
    const size_t smem_a = static_cast<size_t>(ncg_a) * H * sizeof(float);
    const dim3 grid_a(max_active, gy);
    const int lg_a = lanes_for(H / 32);
#define BQD_GU(LG)                                                                                                   \
    (ncg_a == 8 ? launch_gate_up<LG, 8>(grid_a, smem_a, s, gu_codes, gu_scales, gu_ts, x, offsets, pair_token, ws, \
                                        E, H, I, T, topk)                                                            \
                : launch_gate_up<LG, 4>(grid_a, smem_a, s, gu_codes, gu_scales, gu_ts, x, offsets, pair_token, ws, \
                                        E, H, I, T, topk))
    err = lg_a == 32 ? BQD_GU(32) : (lg_a == 16 ? BQD_GU(16) : BQD_GU(8));
#undef BQD_GU
    if (err != cudaSuccess) return err;

    // down: one CTA per (active expert, slice of its H rows)
    int gz = (2 * sms + max_active - 1) / max_active;
    if (gz > H / 8) gz = H / 8;
    if (gz < 1) gz = 1;
    const size_t smem_b = static_cast<size_t>(8) * I * sizeof(float);
    const dim3 grid_b(max_active, gz);
    const int lg_b = lanes_for(I / 32);
#define BQD_DN(LG) \
    launch_down<LG>(grid_b, smem_b, s, dn_codes, dn_scales, dn_ts, offsets, pair_token, pair_weight, pair_slot, ws, E, \
                    H, I, T, topk)
    err = lg_b == 32 ? BQD_DN(32) : (lg_b == 16 ? BQD_DN(16) : BQD_DN(8));
#undef BQD_DN
    if (err != cudaSuccess) return err;

    moe_combine_kernel<<<grid_c, kThreads, 0, s>>>(ws, y, H, topk);
    return cudaGetLastError();
}

}  // namespace bqd
