"""Block-quantized decode matvec for GB300 (sm_103a).

y = W . x with NVFP4 or Q8_0 weights for N = 1..16 tokens, and a top-k routed
MoE layer over NVFP4 experts, computed by the CUDA kernels of libbqd.so
behind the C ABI in include/bqd.h. This package holds the ctypes binding
(same names as the C ABI), the in-tree build and the seeded workload
generator.
"""
from ._binding import (  # noqa: F401
    BQD_PATH_AUTO,
    BQD_PATH_CUDA_CORE,
    BQD_LAUNCH_PDL,
    BQD_PATH_STREAM,
    BQD_PATH_MMA,
    BQD_PATH_DIRECT,
    BQD_PATH_TILES,
    get_launch_flags,
    set_launch_flags,
    bqd_device_error,
    debug_stream_fault,
    BqdError,
    bqd_moe_read_status,
    lib,
    moe_grouped_gemv,
    moe_grouped_gemv_noalloc,
    moe_layer,
    moe_layer_workspace_bytes,
    moe_prefill_layer,
    moe_prefill_workspace_bytes,
    moe_route_topk,
    moe_workspace_bytes,
    nvfp4_dequant,
    nvfp4_encode,
    nvfp4_gemm,
    nvfp4_gemm_grouped,
    nvfp4_gemv,
    nvfp4_gemv_add,
    nvfp4_gemv_path,
    nvfp4_gemv_silu_mul,
    q8_0_dequant,
    q8_0_encode,
    q8_0_gemv,
    q8_0_gemv_add,
    q8_0_gemv_path,
    q4_0_gemv,
    q4_0_gemv_path,
    q4_0_dequant,
    fp8_b128_gemv,
    fp8_b128_gemv_path,
    fp8_b128_dequant,
    q8_0_gemv_silu_mul,
    version,
)
