// gemv.h -- internal launchers behind the C ABI (not part of the public API).
// Each enqueues work on `s` and returns the launch status; none allocates,
// synchronises or validates arguments (the C ABI layer does that first).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace bqd {

// Records the name of a failed CUDA call as the calling thread's last CUDA
// error (what bqd_last_cuda_error returns); cudaSuccess records nothing.
void record_cuda_error(cudaError_t e);

cudaError_t launch_nvfp4_gemv_cuda_core(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                        float* y, int64_t M, int64_t K, int N, cudaStream_t s);
cudaError_t launch_q8_0_gemv_cuda_core(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M,
                                       int64_t K, int N, cudaStream_t s);
cudaError_t launch_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float ts, float* w, int64_t M,
                                 int64_t K, cudaStream_t s);
cudaError_t launch_q8_0_dequant(const int8_t* q, const uint16_t* d, float* w, int64_t M, int64_t K, cudaStream_t s);

// Register-streaming GEMV (gemv_direct.cu): N == 1, K a multiple of 1024
// with K / 1024 in {1, 2, 3, 4, 6, 8, 12, 16}.
bool direct_gemv_supported(int64_t M, int64_t K, int N);
cudaError_t launch_nvfp4_gemv_direct(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                     float* y, int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_q8_0_gemv_direct(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M,
                                    int64_t K, cudaStream_t s);
cudaError_t launch_q4_0_gemv_direct(const uint8_t* codes, const uint16_t* d, const uint16_t* x, float* y,
                                    int64_t M, int64_t K, cudaStream_t s);
// Q4_0 on the CUDA-core path (any M, K % 32 == 0, 1 <= N <= 16) and its
// dequantisation.
cudaError_t launch_q4_0_gemv_cuda_core(const uint8_t* codes, const uint16_t* d, const uint16_t* x, float* y,
                                       int64_t M, int64_t K, int N, cudaStream_t s);
cudaError_t launch_q4_0_dequant(const uint8_t* codes, const uint16_t* d, float* w, int64_t M, int64_t K,
                                cudaStream_t s);
// FP8 block-128 (E4M3 codes [M][K], fp32 scales [ceil(M/128)][ceil(K/128)]):
// the direct kernel (N == 1, the K above), the CUDA-core path (any M,
// K % 32 == 0, 1 <= N <= 16) and the dequantisation.
cudaError_t launch_fp8_b128_gemv_direct(const uint8_t* codes, const float* scales, const uint16_t* x, float* y,
                                        int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_fp8_b128_gemv_cuda_core(const uint8_t* codes, const float* scales, const uint16_t* x, float* y,
                                           int64_t M, int64_t K, int N, cudaStream_t s);
cudaError_t launch_fp8_b128_dequant(const uint8_t* codes, const float* scales, float* w, int64_t M, int64_t K,
                                    cudaStream_t s);
// The same kernel with a fused epilogue: y = W x + r (y may be r); and, on a
// gate_up weight of 2I rows (gate rows 0..I-1, up rows I..2I-1),
// h = SiLU(gate . x) * (up . x).
cudaError_t launch_nvfp4_gemv_direct_add(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                         const float* r, float* y, int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_q8_0_gemv_direct_add(const int8_t* q, const uint16_t* d, const uint16_t* x, const float* r,
                                        float* y, int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_nvfp4_gemv_direct_silu_mul(const uint8_t* codes, const uint8_t* scales, float ts,
                                              const uint16_t* x, float* h, int64_t I, int64_t K, cudaStream_t s);
cudaError_t launch_q8_0_gemv_direct_silu_mul(const int8_t* q, const uint16_t* d, const uint16_t* x, float* h,
                                             int64_t I, int64_t K, cudaStream_t s);

// Warp-tile tensor-core GEMV for a few tokens (gemv_tiles.cu): 2 <= N <= 16,
// K a multiple of 1024, N * K <= 32768 (the activations pass through
// registers once per CTA).
bool tiles_gemv_supported(int64_t M, int64_t K, int N);
cudaError_t launch_nvfp4_gemv_tiles(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                    float* y, int64_t M, int64_t K, int N, cudaStream_t s);

// bf16 -> NVFP4 / Q8_0 encoders (encode.cu).
cudaError_t launch_nvfp4_encode(const uint16_t* w, float ts, uint8_t* codes, uint8_t* scales, int64_t M, int64_t K,
                                cudaStream_t s);
cudaError_t launch_q8_0_encode(const uint16_t* w, int8_t* q, uint16_t* d, int64_t M, int64_t K, cudaStream_t s);

// Bulk-copy streaming GEMV (gemv_stream.cu): N == 1, K % 256 == 0.
bool stream_gemv_supported(int64_t M, int64_t K, int N);
cudaError_t launch_nvfp4_gemv_stream(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                     float* y, int64_t M, int64_t K, cudaStream_t s);
cudaError_t launch_q8_0_gemv_stream(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M,
                                    int64_t K, cudaStream_t s);
// Reads and clears the device error word of the streaming kernels (synchronous).
cudaError_t read_and_clear_stream_error(unsigned int* out);
// Failure-path test setting of the streaming kernel (bqd_debug_stream_fault).
void set_stream_fault(int withhold_last, long long wait_limit);

// Tensor-core GEMV (gemv_mma.cu): NVFP4, 1 <= N <= 16, K % 256 == 0.
bool mma_gemv_supported(int64_t M, int64_t K, int N);
cudaError_t launch_nvfp4_gemv_mma(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x,
                                  float* y, int64_t M, int64_t K, int N, cudaStream_t s);
cudaError_t read_and_clear_mma_error(unsigned int* out);

// MoE (moe.cu). Limits checked by the ABI layer: E <= 1024, topk <= 32,
// T * topk <= 8192.
constexpr int kMoeMaxExperts = 1024;
constexpr int kMoeMaxTopk = 32;
constexpr int kMoeMaxPairs = 8192;

cudaError_t launch_moe_route(const float* logits, int T, int E, int topk, int32_t* offsets, int32_t* pair_token,
                             float* pair_weight, int32_t* pair_slot, cudaStream_t s);

struct MoeWorkspace {
    int32_t* status;  // device error bits (see bqd.h)
    int32_t* count;   // [T*topk] times each (token, slot) was produced
    float* wts;       // [T*topk] routing weight of (token, slot)
    float* h;         // [T*topk][I] SiLU(gate) * up, pair (expert-major) order
    float* part;      // [T*topk][H] down projection of (token, slot)
};
size_t moe_workspace_size(int T, int topk, int H, int I);
MoeWorkspace moe_workspace_carve(void* base, int T, int topk, int H, int I);

// Streaming gate_up and down kernels (moe_stream.cu) for H % 256 == 0 and
// I % 256 == 0; the combine kernel of moe.cu runs after them.
bool moe_stream_supported(int E, int H, int I);
cudaError_t launch_moe_stream_layer(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                                    const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts,
                                    const uint16_t* x, const int32_t* offsets, const int32_t* pair_token,
                                    const float* pair_weight, const int32_t* pair_slot, const MoeWorkspace& ws, int E,
                                    int H, int I, int T, int topk, cudaStream_t stream);
cudaError_t read_and_clear_moe_stream_error(unsigned int* out);
cudaError_t read_and_clear_moe_small_error(unsigned int* out);

// Small-batch MoE kernels (moe_small.cu): the limits of moe_small_supported
// (T <= 16, T * topk <= 128, E <= 512, H in {1024, ..., 8192}, I in {256,
// 512, 1024}). With logits != nullptr every gate_up CTA routes the tokens
// itself (the list arguments are ignored); otherwise the caller's
// expert-major list is checked and used. Writes the workspace's status
// word, per-(token, slot) list, h and h' (for the down kernel), and y (the
// combine is part of the down kernel).
bool moe_small_supported(int E, int H, int I, int T, int topk);
cudaError_t launch_moe_small_layer(const float* logits, const uint8_t* gu_codes, const uint8_t* gu_scales,
                                   const float* gu_ts, const uint8_t* dn_codes, const uint8_t* dn_scales,
                                   const float* dn_ts, const uint16_t* x, const int32_t* offsets,
                                   const int32_t* pair_token, const float* pair_weight, const int32_t* pair_slot,
                                   float* y, const MoeWorkspace& ws, int E, int H, int I, int T, int topk,
                                   cudaStream_t stream);

cudaError_t launch_moe_grouped(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                               const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts,
                               const uint16_t* x, const int32_t* offsets, const int32_t* pair_token,
                               const float* pair_weight, const int32_t* pair_slot, float* y,
                               const MoeWorkspace& ws, int E, int H, int I, int T, int topk, cudaStream_t s);

}  // namespace bqd
