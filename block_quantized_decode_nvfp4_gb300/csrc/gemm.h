// gemm.h -- internal launcher of the prefill GEMM (gemm_prefill.cu): NVFP4
// weights [M][K] times bf16 tokens [T][K] on the tensor cores, Y [T][M].
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace bqd {

// K a multiple of 64, M >= 1, T >= 1 (and the grid limits).
bool gemm_supported(int64_t M, int64_t K, int64_t T);
cudaError_t launch_nvfp4_gemm(const uint8_t* codes, const uint8_t* scales, float ts, const uint16_t* x, float* y,
                              int64_t M, int64_t K, int64_t T, cudaStream_t s);
// Grouped form: E experts' weights [E][M][K] and scales, fp32 tensor scales
// ts [E] (device), tokens [P][K] gathered expert-major, expert e's rows
// [offsets[e], offsets[e + 1]) (device int32 [E + 1]), Y [P][M].
bool gemm_grouped_supported(int64_t E, int64_t M, int64_t K, int64_t P);
// accumulate: Y += instead of Y =. weight_k (default K): the weights' k; a
// smaller divisor of K repeats them along the tokens' k, so that tokens
// [P][r * weight_k] holding r parts of each activation row (side by side)
// give W . (part 0 + ... + part r-1) in one call.
cudaError_t launch_nvfp4_gemm_grouped(const uint8_t* codes, const uint8_t* scales, const float* ts,
                                      const int32_t* offsets, int E, const uint16_t* x, float* y, int64_t M,
                                      int64_t K, int64_t P, cudaStream_t s, bool accumulate = false,
                                      int64_t weight_k = 0);

// MoE prefill layer (moe_prefill.cu): route, gather, grouped gate_up GEMM,
// SiLU(gate) * up split into two bf16 parts, grouped down GEMM of both
// parts, fixed-order combine. T * topk <= 8192 (the route kernel's limit),
// H % 64 == 0, I % 64 == 0.
size_t moe_prefill_workspace_size(int T, int topk, int H, int I, int E);
cudaError_t launch_moe_prefill_layer(const float* logits, const uint8_t* gu_codes, const uint8_t* gu_scales,
                                     const float* gu_ts, const uint8_t* dn_codes, const uint8_t* dn_scales,
                                     const float* dn_ts, const uint16_t* x, float* y, void* ws, int E, int H, int I,
                                     int T, int topk, cudaStream_t s);
cudaError_t read_and_clear_gemm_error(unsigned int* out);

}  // namespace bqd
