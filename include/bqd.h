/*
 * bqd.h -- C ABI of libbqd.so, the GB300 (sm_103a) block-quantized decode
 * matvec library: y = W . x with NVFP4 or Q8_0 weights (also Q4_0, Q4_1 and
 * FP8 block-128), for N = 1 token (plain decode) up to N = 16 (speculative
 * verify), and a top-k routed MoE layer whose experts are NVFP4; around
 * them, decode-path epilogue fusions, bf16 -> NVFP4 / Q8_0 encoders, and
 * NVFP4 prefill GEMMs on the tensor cores with a MoE prefill layer.
 *
 * Sources (what each call computes):
 *  - "Vemloir/LumenLLM" README, Quantization and Kernels bullets: weights in
 *    NVFP4, a block-scaled 4-bit floating-point format; decode runs GEMVs
 *    reduced with warp shuffles.
 *  - "robertbfuentes7-cloud/bw24" README, feature list: the NVFP4 (W4) decode
 *    path is a block-scaled FP4 matvec; speculative decoding verifies K+1
 *    draft tokens in one batched target forward (a matvec with N = K+1
 *    columns); MoE batches routed tokens expert-major and decodes each
 *    selected expert's weights once.
 *  - "avifenesh/memra" README, Decode kernels bullet: NVFP4, Q4_0 and Q8_0
 *    matvecs; Loaders bullet: FP8 checkpoints quantised in blocks of 128.
 *  - "robertbfuentes7-cloud/bw24" README, GGUF bullet: Q4_0 and Q4_1 among
 *    the file formats; safetensors loader bullet: large tensors re-encoded
 *    to Q8_0 / NVFP4 at load.
 * The pages do not print the formats' bit layouts. Elements follow the
 * public closed forms (E2M1 per OCP MX v1.0, E4M3 per OCP OFP8 v1.0, fp16
 * per IEEE 754 binary16, bf16 = upper half of binary32); the block structure
 * is the workload's: NVFP4 has one E4M3 scale per 16 consecutive k of a row
 * plus one FP32 tensor scale, two E2M1 codes per byte with the low nibble
 * holding the lower k; Q8_0 has one fp16 scale per 32 consecutive k.
 *
 * Conventions for every call:
 *  - All array pointers are DEVICE pointers owned by the caller. The library
 *    never allocates, frees or prints, and never synchronises except in
 *    the two status readers, bqd_moe_read_status and bqd_device_error. Work
 *    is enqueued on `stream` (0 = legacy default stream) in stream order;
 *    calls return before the GPU finishes.
 *  - Arrays are dense, row-major, innermost index contiguous, and every base
 *    pointer must be 16-byte aligned.
 *  - Activations are bf16 bit patterns, token-major: x[n][k], row pitch K.
 *    Outputs are fp32, token-major: y[n][m], row pitch M.
 *  - Argument errors are detected on the host before any CUDA call and
 *    return BQD_ERR_NULL / BQD_ERR_SHAPE / BQD_ERR_ALIGN / BQD_ERR_WORKSPACE
 *    / BQD_ERR_PATH without enqueueing anything. BQD_ERR_ARCH means the
 *    current device is not compute capability 10.3. BQD_ERR_LAUNCH reports a
 *    CUDA error from the launch itself (cudaGetLastError).
 *  - Results are deterministic: the same inputs give bit-identical outputs.
 *  - Accuracy: fp32 accumulation; |y - y_exact| <= 1e-3 * sum_k |w x| + 1e-6
 *    per output, where y_exact is the real-valued definition. Dequantised
 *    weights are bit-exact.
 */
#ifndef BQD_H
#define BQD_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int bqd_status;

enum {
    BQD_OK = 0,
    BQD_ERR_NULL = 1,      /* a required pointer is NULL */
    BQD_ERR_SHAPE = 2,     /* a size is out of range or breaks a divisibility rule */
    BQD_ERR_ALIGN = 3,     /* a base pointer is not 16-byte aligned */
    BQD_ERR_ARCH = 4,      /* no current CUDA device, or it is not sm_103 */
    BQD_ERR_LAUNCH = 5,    /* the CUDA launch failed */
    BQD_ERR_WORKSPACE = 6, /* MoE workspace missing or smaller than moe_workspace_bytes() */
    BQD_ERR_PATH = 7,      /* unknown path, or the path does not support these arguments */
    BQD_ERR_DEVICE = 8     /* bqd_moe_read_status found device-side error bits */
};

/* Compute paths of the GEMVs (nvfp4_gemv_path, q8_0_gemv_path). */
enum {
    BQD_PATH_AUTO = 0,      /* the library's choice for the shape (what nvfp4_gemv / q8_0_gemv use) */
    BQD_PATH_CUDA_CORE = 1, /* register-prefetch loads, in-register decode, fp32 FMA; any shape */
    BQD_PATH_STREAM = 2,    /* bulk-copy (TMA) stream into a shared-memory ring, decode on the CUDA
                               cores; N == 1 and K % 256 == 0 (K <= 16384) only, else BQD_ERR_PATH */
    BQD_PATH_DIRECT = 4,    /* weights streamed from HBM straight into registers by fully coalesced 16-byte
                               loads, compile-time unrolled over a row, decode and mixed-precision FMAs on the
                               CUDA cores; N == 1 and K a multiple of 1024 with K / 1024 one of 1, 2, 3, 4, 6,
                               8, 12, 16, else BQD_ERR_PATH */
    BQD_PATH_TILES = 5,     /* NVFP4 only: warp tiles of 8 weight rows x 16 token slots on the tensor cores
                               (mma.sync m16n8k16, exact f16 or bf16 operands, fp32 accumulation), weights
                               streamed straight into registers as for BQD_PATH_DIRECT, a CTA's tiles shared
                               by its warps with a fixed-order sum; 2 <= N <= 16, K a multiple of 1024 and
                               N * K <= 32768, else BQD_ERR_PATH. q8_0_gemv_path returns BQD_ERR_PATH */
    BQD_PATH_MMA = 3        /* NVFP4 only: weights decoded exactly to f16 (or bf16) in tensor memory and
                               multiplied on the tensor cores (tcgen05.mma, fp32 accumulation), the
                               (row tile, k) work split over thread-block clusters with a fixed-order
                               sum, so results are deterministic; 1 <= N <= 16,
                               K % 256 == 0, M < 2^30, K <= 2^20 (smaller if shared memory runs
                               short), else BQD_ERR_PATH. q8_0_gemv_path returns BQD_ERR_PATH */
};

/* Launch options (bqd_set_launch_flags). */
enum {
    /* Programmatic dependent launch for the streaming and tensor-core GEMVs
     * (BQD_PATH_STREAM, BQD_PATH_MMA) and the MoE stream kernels: a call may
     * start while the previous kernel in the same stream is still finishing.
     * A GEMV call may begin reading its WEIGHTS (codes, scales, q, d) then;
     * its activations are read, and its output written, only after that
     * previous kernel has completed, so chaining layers is safe. The MoE
     * kernels read nothing before the previous kernel has completed. Do not
     * enable it if a call's weights can be written by the kernel immediately
     * before it in the stream. Off by default. */
    BQD_LAUNCH_PDL = 1
};

/* Sets the process-wide launch options (BQD_LAUNCH_* bits); returns the
 * previous value. Thread-safe; affects calls made after it returns. */
unsigned int bqd_set_launch_flags(unsigned int flags);
unsigned int bqd_get_launch_flags(void);

/* Device-side status bits written by moe_grouped_gemv into its workspace. */
enum {
    BQD_MOE_BAD_OFFSETS = 1, /* expert_offsets is not a CSR of T*topk pairs */
    BQD_MOE_BAD_PAIR = 2,    /* a pair_token or pair_slot is out of range */
    BQD_MOE_COVERAGE = 4     /* some (token, slot) appears zero or several times */
};

/* Text of a status code (static storage; never NULL). */
const char* bqd_status_string(bqd_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int bqd_version(void);

/* Name of the CUDA error behind the calling thread's last BQD_ERR_LAUNCH
 * (static storage; "cudaSuccess" if there was none). */
const char* bqd_last_cuda_error(void);

/*
 * nvfp4_gemv -- y[n][m] = ts * sum_k e2m1(c[m][k]) * e4m3(s[m][k/16]) * x[n][k]
 * ("robertbfuentes7-cloud/bw24" README, NVFP4 (W4) decode path; the N > 1
 * case is the speculative verify of K+1 tokens).
 *   codes   u8 [M][K/2]: two E2M1 codes per byte, low nibble = even k.
 *   scales  u8 [M][K/16]: E4M3 block scales (signed; NaN codes give NaN).
 *   tensor_scale: the FP32 tensor scale ts.
 *   x       bf16 bits [N][K];   y  fp32 [N][M] (written, never read).
 *   M >= 0, K >= 0 with K % 16 == 0, 1 <= N <= 16, M * K < 2^62.
 *   M == 0: returns BQD_OK without touching the GPU (pointers may be NULL).
 *   K == 0: y is set to zero (codes, scales and x may be NULL).
 */
bqd_status nvfp4_gemv(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x, float* y,
                      int64_t M, int64_t K, int N, cudaStream_t stream);

/* nvfp4_gemv with an explicit compute path (BQD_PATH_*), to compare paths.
 * AUTO takes, for N == 1, BQD_PATH_DIRECT where it applies, else
 * BQD_PATH_STREAM where it applies; for N >= 2 BQD_PATH_MMA where it
 * applies; else BQD_PATH_CUDA_CORE (BQD_PATH_TILES only when asked for:
 * on the verify shapes it is slower than BQD_PATH_MMA). q8_0_gemv_path's
 * AUTO is the same without the tensor-core paths. */
bqd_status nvfp4_gemv_path(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x,
                           float* y, int64_t M, int64_t K, int N, int path, cudaStream_t stream);

/*
 * q8_0_gemv -- y[n][m] = sum_k fp16(d[m][k/32]) * q[m][k] * x[n][k]
 * ("avifenesh/memra" README, Decode kernels bullet: Q8_0 matvec).
 *   q  int8 [M][K] (any value, -128 included);  d  fp16 bits [M][K/32].
 *   The planes are separate (planar), not GGUF's interleaved 34-byte blocks.
 *   x bf16 bits [N][K]; y fp32 [N][M]. K % 32 == 0, 1 <= N <= 16; M == 0 and
 *   K == 0 behave as in nvfp4_gemv.
 */
bqd_status q8_0_gemv(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M, int64_t K, int N,
                     cudaStream_t stream);

/*
 * nvfp4_gemv_add -- y[m] = ts * sum_k e2m1(c[m][k]) * e4m3(s[m][k/16]) * x[k]
 *                   + residual[m]: the GEMV with the residual add of a decode
 * layer fused into its epilogue ("Vemloir/LumenLLM" README, Kernels bullet:
 * the decode path's fused epilogues, next to the warp-shuffle GEMVs).
 *   Arguments as nvfp4_gemv plus residual fp32 [M] (device, 16-byte aligned;
 *   it may be y itself: each output is read, then written, by one thread).
 *   The sum is rounded to fp32 once, then the residual added (one more fp32
 *   rounding). N == 1 (the decode path), M >= 1, K a multiple of 1024 with
 *   K / 1024 in {1, 2, 3, 4, 6, 8, 12, 16}; else BQD_ERR_SHAPE. Runs the
 *   direct kernel (BQD_PATH_DIRECT) with its launch options.
 */
bqd_status nvfp4_gemv_add(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x,
                          const float* residual, float* y, int64_t M, int64_t K, int N, cudaStream_t stream);

/* q8_0_gemv_add -- q8_0_gemv plus residual[m], as nvfp4_gemv_add. */
bqd_status q8_0_gemv_add(const int8_t* q, const uint16_t* d, const uint16_t* x, const float* residual, float* y,
                         int64_t M, int64_t K, int N, cudaStream_t stream);

/*
 * nvfp4_gemv_silu_mul -- h[i] = SiLU(g[i]) * u[i], g = W[i] . x (gate),
 * u = W[I + i] . x (up): a dense MLP's gate_up projection with its
 * activation fused, so g and u never reach memory ("Vemloir/LumenLLM"
 * README, Kernels bullet). W is NVFP4 [2I][K] (codes [2I][K/2], scales
 * [2I][K/16], rows 0..I-1 gate, I..2I-1 up, as the MoE experts' gate_up);
 * h fp32 [I]. g and u are the GEMV's fp32 outputs; SiLU(g) = g / (1 +
 * e^-g) in fp32. N == 1, I >= 1, K as nvfp4_gemv_add; else BQD_ERR_SHAPE.
 */
bqd_status nvfp4_gemv_silu_mul(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x,
                               float* h, int64_t I, int64_t K, int N, cudaStream_t stream);

/* q8_0_gemv_silu_mul -- the same on a Q8_0 gate_up weight (q [2I][K], d [2I][K/32]). */
bqd_status q8_0_gemv_silu_mul(const int8_t* q, const uint16_t* d, const uint16_t* x, float* h, int64_t I, int64_t K,
                              int N, cudaStream_t stream);

/*
 * nvfp4_encode -- NVFP4 codes and block scales of a bf16 weight, on the GPU
 * (re-encoding large tensors at load: "robertbfuentes7-cloud/bw24" README,
 * safetensors loader bullet). Per 16-element block b of a row:
 *   s_b = E4M3(amax_b / 6 / ts),  code_k = E2M1(w_k / (e4m3(s_b) * ts)),
 * every value an IEEE fp32 operation rounded to nearest even, E4M3 and E2M1
 * rounded to nearest even and saturated (448, 6); a zero s_b gives zero
 * codes; a negative w that rounds to zero is -0 (code 8). The integer
 * outputs are a function of the input bits alone (deterministic).
 *   w bf16 bits [M][K]; tensor_scale ts in [2^-100, 2^100] (the caller's
 *   choice, e.g. amax(W) / (6 * 448)); codes u8 [M][K/2] (low nibble = even
 *   k); scales u8 [M][K/16]. K % 16 == 0; w and codes 16-byte aligned.
 *   NaN weights are outside the contract.
 */
bqd_status nvfp4_encode(const uint16_t* w, float tensor_scale, uint8_t* codes, uint8_t* scales, int64_t M, int64_t K,
                        cudaStream_t stream);

/*
 * q8_0_encode -- Q8_0 of a bf16 weight, per 32-element block:
 *   d_b = fp16(amax_b / 127),  q_k = rint(w_k / d_b) clamped to [-127, 127],
 * fp32 operations and conversions rounded to nearest even; d_b = 0 gives
 * q = 0. w bf16 bits [M][K]; q int8 [M][K]; d fp16 bits [M][K/32] (planar,
 * as q8_0_gemv takes them). K % 32 == 0; w and q 16-byte aligned, d 2-byte
 * aligned. Blocks with amax above 65504 * 127, and NaN weights, are outside
 * the contract.
 */
bqd_status q8_0_encode(const uint16_t* w, int8_t* q, uint16_t* d, int64_t M, int64_t K, cudaStream_t stream);

/* q8_0_gemv with an explicit compute path (BQD_PATH_*). */
bqd_status q8_0_gemv_path(const int8_t* q, const uint16_t* d, const uint16_t* x, float* y, int64_t M, int64_t K,
                          int N, int path, cudaStream_t stream);

/*
 * bqd_device_error -- waits for the device, copies the device error words of
 * the streaming and tensor-core GEMV kernels (BQD_PATH_STREAM, BQD_PATH_MMA),
 * of the MoE stream kernels, of the small-batch MoE kernels (the
 * activations' copy in moe_layer / moe_grouped_gemv at T <= 16) and of the
 * prefill GEMM (nvfp4_gemm) to *bits_out (OR of the five) and clears them. Bit 0: a wait ran out
 * (the kernel gave up instead of hanging; its outputs are unspecified).
 * Returns BQD_ERR_DEVICE if any bit was set. Synchronising: do not call it
 * inside a stream capture.
 */
bqd_status bqd_device_error(unsigned int* bits_out);

/*
 * bqd_debug_stream_fault -- a switch for testing the failure path of the
 * streaming GEMV kernel (BQD_PATH_STREAM), not for production use. With
 * withhold_last_stage != 0, each CTA's producer stops before issuing the
 * copy of its last ring stage, so the consumer warps' wait for it can only
 * run out: they give up after wait_limit_cycles SM clock cycles, set bit 0
 * of the device error word (bqd_device_error) and leave that stage's rows
 * unwritten. No copy is in flight when they give up. wait_limit_cycles = 0
 * restores the default limit (2^31 cycles, about one second);
 * withhold_last_stage = 0 restores normal operation. Process-wide; affects
 * calls made after it returns. Returns BQD_ERR_SHAPE for a negative limit.
 */
bqd_status bqd_debug_stream_fault(int withhold_last_stage, long long wait_limit_cycles);

/*
 * nvfp4_dequant -- w[m][k] = fl32(e2m1(c[m][k]) * e4m3(s[m][k/16]) * ts),
 * the dequantised weight rounded once to fp32 (bit-exact). Uses the same
 * device decoders as the GEMV. w fp32 [M][K]. Shape rules as nvfp4_gemv.
 */
bqd_status nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, float tensor_scale, float* w, int64_t M,
                         int64_t K, cudaStream_t stream);

/* q8_0_dequant -- w[m][k] = fp16(d[m][k/32]) * q[m][k] (exact in fp32). */
bqd_status q8_0_dequant(const int8_t* q, const uint16_t* d, float* w, int64_t M, int64_t K, cudaStream_t stream);

/*
 * q4_0_gemv -- y[n][m] = sum_k fp16(d[m][k/32]) * (q[m][k] - 8) * x[n][k]
 * ("avifenesh/memra" README, Decode kernels bullet: NVFP4 / Q4_0 / Q8_0
 * matvecs; "robertbfuentes7-cloud/bw24" README, GGUF bullet: Q4_0 among the
 * file formats).
 *   codes u8 [M][K/2]: 16 bytes per 32-element block; byte j of a block
 *         holds element j (low nibble) and element j + 16 (high nibble), the
 *         order of a GGUF Q4_0 block, whose fp16 field is the d plane:
 *   d     fp16 bits [M][K/32]. The planes are a GGUF block's two fields,
 *         split (planar), so a loader copies them byte for byte.
 *   x bf16 bits [N][K]; y fp32 [N][M]. K % 32 == 0, 1 <= N <= 16; M == 0 and
 *   K == 0 behave as in nvfp4_gemv. codes, d, x, y 16-byte aligned.
 *   AUTO: BQD_PATH_DIRECT for N == 1 and the K it takes (K a multiple of
 *   1024 with K / 1024 in {1, 2, 3, 4, 6, 8, 12, 16}), else
 *   BQD_PATH_CUDA_CORE. Products are exact (q - 8 and the prescaled
 *   activations are f16 values, or fp32 FMAs outside that range); sums fp32.
 */
bqd_status q4_0_gemv(const uint8_t* codes, const uint16_t* d, const uint16_t* x, float* y, int64_t M, int64_t K,
                     int N, cudaStream_t stream);

/* q4_0_gemv with an explicit compute path: BQD_PATH_AUTO, BQD_PATH_DIRECT or
 * BQD_PATH_CUDA_CORE (others: BQD_ERR_PATH). */
bqd_status q4_0_gemv_path(const uint8_t* codes, const uint16_t* d, const uint16_t* x, float* y, int64_t M,
                          int64_t K, int N, int path, cudaStream_t stream);

/*
 * q4_1_gemv -- y[n][m] = sum_k (fp16(d[m][k/32]) * q[m][k] + fp16(mn[m][k/32])) * x[n][k]
 * ("robertbfuentes7-cloud/bw24" README, GGUF bullet: Q4_1 among the file
 * formats).
 *   codes u8 [M][K/2]: 16 bytes per 32-element block in the Q4_0 order
 *         (byte j holds element j in its low and element j + 16 in its
 *         high nibble), q in 0..15.
 *   dm    fp16 bits [M][K/32][2]: each block's (d, mn), the two fp16 fields
 *         of a GGUF Q4_1 block side by side, so a loader copies them byte
 *         for byte.
 *   x bf16 bits [N][K]; y fp32 [N][M]. K % 32 == 0, 1 <= N <= 16; M == 0 and
 *   K == 0 behave as in nvfp4_gemv. codes, dm, x, y 16-byte aligned.
 *   One path (the CUDA-core GEMV): per block, d * sum q x + mn * sum x, the
 *   products q x exact in fp32, the sums fp32.
 */
bqd_status q4_1_gemv(const uint8_t* codes, const uint16_t* dm, const uint16_t* x, float* y, int64_t M, int64_t K,
                     int N, cudaStream_t stream);

/* q4_1_dequant -- w[m][k] = fp16(d) * q + fp16(mn) rounded once to fp32;
 * layout and shape rules as q4_1_gemv. */
bqd_status q4_1_dequant(const uint8_t* codes, const uint16_t* dm, float* w, int64_t M, int64_t K,
                        cudaStream_t stream);

/*
 * fp8_b128_gemv -- y[n][m] = sum_k e4m3(c[m][k]) * s[m/128][k/128] * x[n][k]
 * ("Vemloir/LumenLLM" README, Quantization bullet: FP8 E4M3 weights beside
 * NVFP4; "avifenesh/memra" README, Loaders bullet: FP8 checkpoints
 * quantised in blocks of 128, one scale per 128 x 128 tile).
 *   codes  u8 [M][K]: E4M3 bytes (OCP 8-bit FP, E4M3FN; 0x7f and 0xff are
 *          NaN and give NaN), row-major.
 *   scales fp32 [ceil(M/128)][ceil(K/128)], row-major: the tile scale that
 *          multiplies the E4M3 values (a checkpoint's "scale_inv").
 *   x bf16 bits [N][K]; y fp32 [N][M]. K % 32 == 0, 1 <= N <= 16; M == 0 and
 *   K == 0 behave as in nvfp4_gemv. codes, scales, x, y 16-byte aligned.
 *   AUTO: BQD_PATH_DIRECT for N == 1 and the K it takes (K a multiple of
 *   1024 with K / 1024 in {1, 2, 3, 4, 6, 8, 12, 16}), else
 *   BQD_PATH_CUDA_CORE. Products are exact (E4M3 values are f16 values, the
 *   activations f16 after an exact per-call power-of-two prescale, or fp32
 *   FMAs outside that range); the sums and the scale multiply are fp32.
 */
bqd_status fp8_b128_gemv(const uint8_t* codes, const float* scales, const uint16_t* x, float* y, int64_t M,
                         int64_t K, int N, cudaStream_t stream);

/* fp8_b128_gemv with an explicit compute path: BQD_PATH_AUTO, BQD_PATH_DIRECT
 * or BQD_PATH_CUDA_CORE (others: BQD_ERR_PATH). */
bqd_status fp8_b128_gemv_path(const uint8_t* codes, const float* scales, const uint16_t* x, float* y, int64_t M,
                              int64_t K, int N, int path, cudaStream_t stream);

/*
 * nvfp4_gemm -- Y[t][m] = ts * sum_k e2m1(c[m][k]) * e4m3(s[m][k/16]) * x[t][k]
 * for many tokens (prefill) on the tensor cores ("Vemloir/LumenLLM" README,
 * Kernels bullet: NVFP4 grouped-MoE prefill, a per-expert variable-grid
 * NVFP4 GEMM; this is the GEMM of one weight matrix, which a grouped MoE
 * prefill runs per expert on its gathered tokens).
 *   codes, scales, tensor_scale as nvfp4_gemv; x bf16 bits [T][K]; y fp32
 *   [T][M] (written, never read). K % 64 == 0, T >= 0, M >= 0; M == 0 or
 *   T == 0: BQD_OK without touching the GPU; K == 0: y set to zero. All
 *   pointers 16-byte aligned. Every product is exact (the dequantised
 *   weight and x are bf16 values); the sums are fp32 in the tensor cores'
 *   order, so |y - y_exact| stays within the GEMV tolerance. Tiles of 128
 *   weight rows x 256 tokens, one CTA each (up to 65535 token tiles).
 */
bqd_status nvfp4_gemm(const uint8_t* codes, const uint8_t* scales, float tensor_scale, const uint16_t* x, float* y,
                      int64_t M, int64_t K, int64_t T, cudaStream_t stream);

/*
 * nvfp4_gemm_grouped -- the per-expert variable-grid form of nvfp4_gemm for
 * a MoE prefill ("Vemloir/LumenLLM" README, Kernels bullet): for every
 * expert e and every gathered token p in [offsets[e], offsets[e + 1]),
 *   Y[p][m] = ts[e] * sum_k e2m1(c[e][m][k]) * e4m3(s[e][m][k/16]) * x[p][k].
 *   codes u8 [E][M][K/2]; scales u8 [E][M][K/16]; tensor_scales fp32 [E]
 *   (device); x bf16 bits [P][K], the routed tokens gathered expert-major;
 *   expert_offsets int32 [E + 1] (device), 0 = offsets[0] <= ... <=
 *   offsets[E] = P; y fp32 [P][M]. K % 64 == 0, E >= 1; M == 0 or P == 0:
 *   BQD_OK without touching the GPU; K == 0: y set to zero. codes, scales,
 *   x, y 16-byte aligned; tensor_scales and expert_offsets 4-byte aligned.
 *   One launch: tiles of 256 weight rows x BN of an expert's tokens, BN =
 *   32, 64 or 128 for a mean of at most 16, at most 48, or more tokens per
 *   expert (P / E rounded up), wider where the tile count would exceed the
 *   grid's 65535 rows (P / 128 + E <= 65535 is required). Offsets
 *   outside [0, P] are clamped (no access leaves the arrays; the outputs of
 *   such a call are unspecified).
 */
bqd_status nvfp4_gemm_grouped(const uint8_t* codes, const uint8_t* scales, const float* tensor_scales,
                              const uint16_t* x, const int32_t* expert_offsets, float* y, int E, int64_t M, int64_t K,
                              int64_t P, cudaStream_t stream);

/*
 * moe_prefill_layer -- the routed MoE layer of moe_layer for many tokens
 * (prefill), on the tensor cores: routing as moe_route_topk, the routed
 * tokens gathered expert-major, gate/up of every (token, slot) pair by
 * nvfp4_gemm_grouped, h = SiLU(gate) * up in fp32, the down projection by
 * nvfp4_gemm_grouped on h split into two bf16 parts (bf16(h) and the bf16
 * of the rest, so h is kept to ~2^-17 of its size), and y_t = sum over the
 * slots s = 0 .. topk - 1 of w(t, s) * down (in slot order; deterministic).
 * ("Vemloir/LumenLLM" README, Kernels bullet: NVFP4 grouped-MoE prefill.)
 *   Layout and meaning of logits, the weights, tensor scales, x and y as
 *   moe_layer; workspace of moe_prefill_workspace_bytes(T, topk, H, I, E)
 *   bytes, 16-byte aligned (about T * topk * (6 H + 12 I) bytes).
 *   T * topk <= 8192, topk <= min(E, 32), E <= 1024, H and I multiples of 64
 *   (up to 65536); else BQD_ERR_SHAPE. A too small workspace:
 *   BQD_ERR_WORKSPACE. Pointers 16-byte aligned (the tensor scales 4).
 */
size_t moe_prefill_workspace_bytes(int T, int topk, int H, int I, int E);
bqd_status moe_prefill_layer(const float* logits, const uint8_t* gu_codes, const uint8_t* gu_scales,
                             const float* gu_ts, const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts,
                             const uint16_t* x, float* y, void* workspace, size_t workspace_bytes, int E, int H, int I,
                             int T, int topk, cudaStream_t stream);

/* q4_0_dequant -- w[m][k] = fp16(d[m][k/32]) * (q[m][k] - 8) (exact in
 * fp32); layout and shape rules as q4_0_gemv. */
bqd_status q4_0_dequant(const uint8_t* codes, const uint16_t* d, float* w, int64_t M, int64_t K,
                        cudaStream_t stream);

/* fp8_b128_dequant -- w[m][k] = e4m3(c[m][k]) * s[m/128][k/128] in fp32 (the
 * exact product rounded once to nearest); layout and shape rules as
 * fp8_b128_gemv. */
bqd_status fp8_b128_dequant(const uint8_t* codes, const float* scales, float* w, int64_t M, int64_t K,
                            cudaStream_t stream);

/*
 * moe_route_topk -- router and expert-major list of a top-k routed MoE layer
 * ("robertbfuentes7-cloud/bw24" README, MoE bullet: expert-major batching).
 *   logits fp32 [T][E]. For each token: softmax over the E logits, keep the
 *   topk largest (equal logits: lower expert index first), renormalise the
 *   kept probabilities to sum to 1. Slot s of a token is its s-th largest.
 *   Outputs, P = T * topk pairs grouped by expert (a CSR):
 *     expert_offsets int32 [E+1]: expert e owns pairs [off[e], off[e+1]).
 *     pair_token  int32 [P], pair_slot int32 [P], pair_weight fp32 [P];
 *     inside an expert's segment tokens are in increasing order.
 *   1 <= T, 1 <= topk <= min(E, 32), E <= 1024, T * topk <= 8192.
 *   NaN logits are outside the contract (they are selected last).
 */
bqd_status moe_route_topk(const float* logits, int T, int E, int topk, int32_t* expert_offsets, int32_t* pair_token,
                          float* pair_weight, int32_t* pair_slot, cudaStream_t stream);

/* Bytes of device workspace moe_grouped_gemv needs for these sizes. */
size_t moe_workspace_bytes(int T, int topk, int H, int I);

/*
 * moe_grouped_gemv -- one routed MoE FFN layer over T tokens, given the
 * expert-major list (from moe_route_topk or the caller):
 *   g = W_gu[e][0:I] . x_t,  u = W_gu[e][I:2I] . x_t,  h = SiLU(g) * u,
 *   y_t = sum_{s = 0..topk-1, in order} w_{t,s} * (W_dn[e_{t,s}] . h)
 * Each active expert's weights are streamed once for all of its tokens.
 *   gu_codes u8 [E][2I][H/2], gu_scales u8 [E][2I][H/16], gu_ts fp32 [E]
 *     (rows 0..I-1 of an expert are the gate projection, I..2I-1 the up one);
 *   dn_codes u8 [E][H][I/2], dn_scales u8 [E][H][I/16], dn_ts fp32 [E];
 *   x bf16 bits [T][H]; y fp32 [T][H];
 *   workspace: device memory of at least moe_workspace_bytes(T, topk, H, I)
 *   bytes, 256-byte aligned, owned by the caller, not shared by calls that
 *   may overlap. Its first int32 is the status word (BQD_MOE_* bits, cleared
 *   at the start of each call); h (fp32 [T*topk][I], pair order) starts at
 *   byte 256 + 2 * align256(4 * T * topk).
 *   H % 32 == 0, I % 32 == 0, 32 <= H <= 8192, 32 <= I <= 4096,
 *   1 <= topk <= min(E, 32), E <= 1024, T * topk <= 8192.
 *   Malformed lists never fault: the status word records them (read it with
 *   bqd_moe_read_status) and the affected outputs are unspecified.
 */
bqd_status moe_grouped_gemv(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                            const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts, const uint16_t* x,
                            const int32_t* expert_offsets, const int32_t* pair_token, const float* pair_weight,
                            const int32_t* pair_slot, float* y, void* workspace, size_t workspace_bytes, int E,
                            int H, int I, int T, int topk, cudaStream_t stream);

/*
 * moe_layer -- the routed MoE layer from router logits: the same results as
 * moe_route_topk followed by moe_grouped_gemv ("robertbfuentes7-cloud/bw24"
 * README, MoE bullet), in fewer launches.
 *   logits fp32 [T][E]; the other arguments as in moe_grouped_gemv;
 *   workspace: at least moe_layer_workspace_bytes(T, topk, H, I, E) bytes,
 *   256-byte aligned, owned by the caller, not shared by calls that may
 *   overlap. Its first int32 is the status word, h starts where
 *   moe_grouped_gemv puts it.
 *   For decode and verify batches (T <= 16, T * topk <= 128, topk <= 32,
 *   E <= 512, H one of 1024, 2048, 4096, 8192, I one of 256, 512, 1024,
 *   H >= 2 I, topk * I <= 8192, T * H <= 32768) the layer is two kernels:
 *   the gate_up kernel routes the tokens in every CTA (no route kernel) and
 *   leaves the per-(token, slot) list and h for the down kernel, which
 *   folds in the weighted combine; otherwise moe_route_topk writes the list
 *   into the workspace and moe_grouped_gemv follows. Limits as
 *   moe_grouped_gemv plus those of moe_route_topk. NaN logits are outside
 *   the contract.
 */
bqd_status moe_layer(const float* logits, const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                     const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts, const uint16_t* x,
                     float* y, void* workspace, size_t workspace_bytes, int E, int H, int I, int T, int topk,
                     cudaStream_t stream);

/* Bytes of device workspace moe_layer needs for these sizes (0 if a size is < 1). */
size_t moe_layer_workspace_bytes(int T, int topk, int H, int I, int E);

/*
 * moe_grouped_gemv_noalloc -- moe_grouped_gemv for callers that cannot
 * allocate device memory (no counterpart on the source pages; it exists for
 * programs whose host owns every device allocation and gives plug-ins no
 * allocator, and for loops that must not allocate once running).
 * Same arguments and results as moe_grouped_gemv, without the workspace:
 * the scratch is a 4 MiB array inside libbqd.so, held on every GPU that
 * loads the library until the process exits. Calls whose
 * moe_workspace_bytes(T, topk, H, I) exceeds 4 MiB return BQD_ERR_WORKSPACE
 * before touching the GPU. The library allocates nothing on this path.
 * The first call on each device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * The address is cached per CUDA context: after cudaDeviceReset (or any
 * other way the context is destroyed and created again) the next call looks
 * it up again, so that call too should come before any stream capture.
 * A failed lookup or launch returns BQD_ERR_LAUNCH and records the CUDA
 * error's name for bqd_last_cuda_error().
 * Every call shares the one array: calls that may run at the same time on
 * the GPU (other streams, other threads) race and give unspecified results.
 * The array keeps the last call's contents; whatever a call needs zeroed it
 * clears itself. Device-side list checks still run, but their status word
 * lives in the shared array and is not reported.
 */
bqd_status moe_grouped_gemv_noalloc(const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_ts,
                                    const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_ts,
                                    const uint16_t* x, const int32_t* expert_offsets, const int32_t* pair_token,
                                    const float* pair_weight, const int32_t* pair_slot, float* y, int E, int H,
                                    int I, int T, int topk, cudaStream_t stream);

/*
 * bqd_moe_read_status -- waits for `stream`, copies the workspace's status
 * word to *status_out and returns BQD_ERR_DEVICE if it is non-zero, else
 * BQD_OK. Synchronising: do not call it inside a stream capture.
 */
bqd_status bqd_moe_read_status(const void* workspace, int32_t* status_out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BQD_H */
