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
cudaError_t launch_nvfp4_gemm_grouped(const uint8_t* codes, const uint8_t* scales, const float* ts,
                                      const int32_t* offsets, int E, const uint16_t* x, float* y, int64_t M,
                                      int64_t K, int64_t P, cudaStream_t s);
cudaError_t read_and_clear_gemm_error(unsigned int* out);

}  // namespace bqd
