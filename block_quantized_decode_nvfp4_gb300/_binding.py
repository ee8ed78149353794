"""ctypes binding of libbqd.so: the C ABI of include/bqd.h, same names.

Argument marshalling only. Array arguments are torch tensors (device memory)
or raw integer device addresses; sizes are passed through unchanged; the
stream defaults to torch's current stream. A non-zero status raises BqdError.
There is no fallback: if libbqd.so is missing every call raises.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbqd.so")

BQD_OK = 0
STATUS_NAMES = {0: "BQD_OK", 1: "BQD_ERR_NULL", 2: "BQD_ERR_SHAPE", 3: "BQD_ERR_ALIGN", 4: "BQD_ERR_ARCH",
                5: "BQD_ERR_LAUNCH", 6: "BQD_ERR_WORKSPACE", 7: "BQD_ERR_PATH", 8: "BQD_ERR_DEVICE"}
BQD_PATH_AUTO = 0
BQD_PATH_CUDA_CORE = 1
BQD_PATH_STREAM = 2
BQD_PATH_MMA = 3
BQD_PATH_DIRECT = 4
BQD_PATH_TILES = 5
BQD_LAUNCH_PDL = 1

_lib = None


class BqdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().bqd_status_string(status).decode() if _lib is not None else "?"
        if status == 5 and _lib is not None:
            msg += ": " + lib().bqd_last_cuda_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({msg})")


_vp, _i64, _i32, _f32, _sz = C.c_void_p, C.c_int64, C.c_int, C.c_float, C.c_size_t
SIGNATURES = {
    "bqd_status_string": (C.c_char_p, [_i32]),
    "bqd_version": (_i32, []),
    "bqd_last_cuda_error": (C.c_char_p, []),
    "bqd_set_launch_flags": (C.c_uint, [C.c_uint]),
    "bqd_get_launch_flags": (C.c_uint, []),
    "nvfp4_gemv": (_i32, [_vp, _vp, _f32, _vp, _vp, _i64, _i64, _i32, _vp]),
    "nvfp4_gemv_path": (_i32, [_vp, _vp, _f32, _vp, _vp, _i64, _i64, _i32, _i32, _vp]),
    "q8_0_gemv": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "q8_0_gemv_path": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp]),
    "nvfp4_gemm": (_i32, [_vp, _vp, _f32, _vp, _vp, _i64, _i64, _i64, _vp]),
    "moe_prefill_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "moe_prefill_layer": (_i32, [_vp] * 10 + [_sz, _i32, _i32, _i32, _i32, _i32, _vp]),
    "nvfp4_gemm_grouped": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _vp]),
    "q4_0_gemv": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "q4_0_gemv_path": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp]),
    "q4_0_dequant": (_i32, [_vp, _vp, _vp, _i64, _i64, _vp]),
    "q4_1_gemv": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "q4_1_dequant": (_i32, [_vp, _vp, _vp, _i64, _i64, _vp]),
    "fp8_b128_gemv": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "fp8_b128_gemv_path": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _vp]),
    "fp8_b128_dequant": (_i32, [_vp, _vp, _vp, _i64, _i64, _vp]),
    "nvfp4_gemv_add": (_i32, [_vp, _vp, _f32, _vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "nvfp4_encode": (_i32, [_vp, _f32, _vp, _vp, _i64, _i64, _vp]),
    "q8_0_encode": (_i32, [_vp, _vp, _vp, _i64, _i64, _vp]),
    "q8_0_gemv_add": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "nvfp4_gemv_silu_mul": (_i32, [_vp, _vp, _f32, _vp, _vp, _i64, _i64, _i32, _vp]),
    "q8_0_gemv_silu_mul": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "bqd_device_error": (_i32, [C.POINTER(C.c_uint)]),
    "bqd_debug_stream_fault": (_i32, [_i32, C.c_longlong]),
    "nvfp4_dequant": (_i32, [_vp, _vp, _f32, _vp, _i64, _i64, _vp]),
    "q8_0_dequant": (_i32, [_vp, _vp, _vp, _i64, _i64, _vp]),
    "moe_route_topk": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "moe_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "moe_grouped_gemv": (_i32, [_vp] * 13 + [_sz, _i32, _i32, _i32, _i32, _i32, _vp]),
    "bqd_moe_read_status": (_i32, [_vp, C.POINTER(C.c_int32), _vp]),
    "moe_grouped_gemv_noalloc": (_i32, [_vp] * 12 + [_i32, _i32, _i32, _i32, _i32, _vp]),
    "moe_layer": (_i32, [_vp] * 10 + [_sz, _i32, _i32, _i32, _i32, _i32, _vp]),
    "moe_layer_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
}


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                               "g.build()'); there is no CPU fallback")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> None:
    if status != BQD_OK:
        raise BqdError(status, where)


def version() -> int:
    return lib().bqd_version()


def set_launch_flags(flags: int) -> int:
    """Process-wide launch options (BQD_LAUNCH_*); returns the previous value."""
    return lib().bqd_set_launch_flags(flags)


def get_launch_flags() -> int:
    return lib().bqd_get_launch_flags()


def nvfp4_gemv(codes, scales, tensor_scale, x, y, M, K, N, stream=None):
    _check(lib().nvfp4_gemv(_ptr(codes), _ptr(scales), tensor_scale, _ptr(x), _ptr(y), M, K, N, _stream(stream)),
           "nvfp4_gemv")


def nvfp4_gemv_path(codes, scales, tensor_scale, x, y, M, K, N, path, stream=None):
    _check(lib().nvfp4_gemv_path(_ptr(codes), _ptr(scales), tensor_scale, _ptr(x), _ptr(y), M, K, N, path,
                                 _stream(stream)), "nvfp4_gemv_path")


def q8_0_gemv(q, d, x, y, M, K, N, stream=None):
    _check(lib().q8_0_gemv(_ptr(q), _ptr(d), _ptr(x), _ptr(y), M, K, N, _stream(stream)), "q8_0_gemv")


def q8_0_gemv_path(q, d, x, y, M, K, N, path, stream=None):
    _check(lib().q8_0_gemv_path(_ptr(q), _ptr(d), _ptr(x), _ptr(y), M, K, N, path, _stream(stream)),
           "q8_0_gemv_path")


def nvfp4_gemv_add(codes, scales, tensor_scale, x, residual, y, M, K, N=1, stream=None):
    _check(lib().nvfp4_gemv_add(_ptr(codes), _ptr(scales), tensor_scale, _ptr(x), _ptr(residual), _ptr(y), M, K, N,
                                _stream(stream)), "nvfp4_gemv_add")


def q8_0_gemv_add(q, d, x, residual, y, M, K, N=1, stream=None):
    _check(lib().q8_0_gemv_add(_ptr(q), _ptr(d), _ptr(x), _ptr(residual), _ptr(y), M, K, N, _stream(stream)),
           "q8_0_gemv_add")


def nvfp4_gemv_silu_mul(codes, scales, tensor_scale, x, h, I, K, N=1, stream=None):
    _check(lib().nvfp4_gemv_silu_mul(_ptr(codes), _ptr(scales), tensor_scale, _ptr(x), _ptr(h), I, K, N,
                                     _stream(stream)), "nvfp4_gemv_silu_mul")


def q8_0_gemv_silu_mul(q, d, x, h, I, K, N=1, stream=None):
    _check(lib().q8_0_gemv_silu_mul(_ptr(q), _ptr(d), _ptr(x), _ptr(h), I, K, N, _stream(stream)),
           "q8_0_gemv_silu_mul")


def nvfp4_encode(w, tensor_scale, codes, scales, M, K, stream=None):
    _check(lib().nvfp4_encode(_ptr(w), tensor_scale, _ptr(codes), _ptr(scales), M, K, _stream(stream)),
           "nvfp4_encode")


def q8_0_encode(w, q, d, M, K, stream=None):
    _check(lib().q8_0_encode(_ptr(w), _ptr(q), _ptr(d), M, K, _stream(stream)), "q8_0_encode")


def bqd_device_error() -> int:
    """Device error bits of the streaming kernels (synchronising; clears them)."""
    out = C.c_uint(0)
    st = lib().bqd_device_error(C.byref(out))
    if st not in (BQD_OK, 8):
        raise BqdError(st, "bqd_device_error")
    return out.value


def debug_stream_fault(withhold_last_stage: bool, wait_limit_cycles: int = 0) -> None:
    """Failure-path test switch of the streaming GEMV kernel (see bqd.h)."""
    _check(lib().bqd_debug_stream_fault(1 if withhold_last_stage else 0, wait_limit_cycles),
           "bqd_debug_stream_fault")


def nvfp4_dequant(codes, scales, tensor_scale, w, M, K, stream=None):
    _check(lib().nvfp4_dequant(_ptr(codes), _ptr(scales), tensor_scale, _ptr(w), M, K, _stream(stream)),
           "nvfp4_dequant")


def q8_0_dequant(q, d, w, M, K, stream=None):
    _check(lib().q8_0_dequant(_ptr(q), _ptr(d), _ptr(w), M, K, _stream(stream)), "q8_0_dequant")


def nvfp4_gemm(codes, scales, tensor_scale, x, y, M, K, T, stream=None):
    _check(lib().nvfp4_gemm(_ptr(codes), _ptr(scales), tensor_scale, _ptr(x), _ptr(y), M, K, T, _stream(stream)),
           "nvfp4_gemm")


def nvfp4_gemm_grouped(codes, scales, tensor_scales, x, expert_offsets, y, E, M, K, P, stream=None):
    _check(lib().nvfp4_gemm_grouped(_ptr(codes), _ptr(scales), _ptr(tensor_scales), _ptr(x), _ptr(expert_offsets),
                                    _ptr(y), E, M, K, P, _stream(stream)), "nvfp4_gemm_grouped")


def moe_prefill_workspace_bytes(T, topk, H, I, E):
    return int(lib().moe_prefill_workspace_bytes(T, topk, H, I, E))


def moe_prefill_layer(logits, gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x, y, workspace,
                      workspace_bytes, E, H, I, T, topk, stream=None):
    _check(lib().moe_prefill_layer(_ptr(logits), _ptr(gu_codes), _ptr(gu_scales), _ptr(gu_ts), _ptr(dn_codes),
                                   _ptr(dn_scales), _ptr(dn_ts), _ptr(x), _ptr(y), _ptr(workspace), workspace_bytes,
                                   E, H, I, T, topk, _stream(stream)), "moe_prefill_layer")


def q4_0_gemv(codes, d, x, y, M, K, N, stream=None):
    _check(lib().q4_0_gemv(_ptr(codes), _ptr(d), _ptr(x), _ptr(y), M, K, N, _stream(stream)), "q4_0_gemv")


def q4_0_gemv_path(codes, d, x, y, M, K, N, path, stream=None):
    _check(lib().q4_0_gemv_path(_ptr(codes), _ptr(d), _ptr(x), _ptr(y), M, K, N, path, _stream(stream)),
           "q4_0_gemv_path")


def q4_0_dequant(codes, d, w, M, K, stream=None):
    _check(lib().q4_0_dequant(_ptr(codes), _ptr(d), _ptr(w), M, K, _stream(stream)), "q4_0_dequant")


def q4_1_gemv(codes, dm, x, y, M, K, N, stream=None):
    """Q4_1 GEMV: codes [M][K/2] (Q4_0 nibble order), dm [M][K/32][2] fp16 (d, m)."""
    _check(lib().q4_1_gemv(_ptr(codes), _ptr(dm), _ptr(x), _ptr(y), M, K, N, _stream(stream)), "q4_1_gemv")


def q4_1_dequant(codes, dm, w, M, K, stream=None):
    _check(lib().q4_1_dequant(_ptr(codes), _ptr(dm), _ptr(w), M, K, _stream(stream)), "q4_1_dequant")


def fp8_b128_gemv(codes, scales, x, y, M, K, N, stream=None):
    """FP8 block-128 GEMV: E4M3 codes [M][K], fp32 tile scales [ceil(M/128)][ceil(K/128)]."""
    _check(lib().fp8_b128_gemv(_ptr(codes), _ptr(scales), _ptr(x), _ptr(y), M, K, N, _stream(stream)),
           "fp8_b128_gemv")


def fp8_b128_gemv_path(codes, scales, x, y, M, K, N, path, stream=None):
    _check(lib().fp8_b128_gemv_path(_ptr(codes), _ptr(scales), _ptr(x), _ptr(y), M, K, N, path, _stream(stream)),
           "fp8_b128_gemv_path")


def fp8_b128_dequant(codes, scales, w, M, K, stream=None):
    _check(lib().fp8_b128_dequant(_ptr(codes), _ptr(scales), _ptr(w), M, K, _stream(stream)), "fp8_b128_dequant")


def moe_route_topk(logits, T, E, topk, expert_offsets, pair_token, pair_weight, pair_slot, stream=None):
    _check(lib().moe_route_topk(_ptr(logits), T, E, topk, _ptr(expert_offsets), _ptr(pair_token),
                                _ptr(pair_weight), _ptr(pair_slot), _stream(stream)), "moe_route_topk")


def moe_workspace_bytes(T, topk, H, I) -> int:
    return lib().moe_workspace_bytes(T, topk, H, I)


def moe_grouped_gemv(gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x, expert_offsets, pair_token,
                     pair_weight, pair_slot, y, workspace, workspace_bytes, E, H, I, T, topk, stream=None):
    _check(lib().moe_grouped_gemv(_ptr(gu_codes), _ptr(gu_scales), _ptr(gu_ts), _ptr(dn_codes), _ptr(dn_scales),
                                  _ptr(dn_ts), _ptr(x), _ptr(expert_offsets), _ptr(pair_token), _ptr(pair_weight),
                                  _ptr(pair_slot), _ptr(y), _ptr(workspace), workspace_bytes, E, H, I, T, topk,
                                  _stream(stream)), "moe_grouped_gemv")


def moe_grouped_gemv_noalloc(gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x, expert_offsets,
                             pair_token, pair_weight, pair_slot, y, E, H, I, T, topk, stream=None):
    """moe_grouped_gemv without a caller workspace (scratch inside the library)."""
    _check(lib().moe_grouped_gemv_noalloc(_ptr(gu_codes), _ptr(gu_scales), _ptr(gu_ts), _ptr(dn_codes),
                                          _ptr(dn_scales), _ptr(dn_ts), _ptr(x), _ptr(expert_offsets),
                                          _ptr(pair_token), _ptr(pair_weight), _ptr(pair_slot), _ptr(y), E, H, I, T,
                                          topk, _stream(stream)), "moe_grouped_gemv_noalloc")


def moe_layer(logits, gu_codes, gu_scales, gu_ts, dn_codes, dn_scales, dn_ts, x, y, workspace, workspace_bytes,
              E, H, I, T, topk, stream=None):
    """Router and routed MoE layer from logits (moe_route_topk + moe_grouped_gemv in one call)."""
    _check(lib().moe_layer(_ptr(logits), _ptr(gu_codes), _ptr(gu_scales), _ptr(gu_ts), _ptr(dn_codes),
                           _ptr(dn_scales), _ptr(dn_ts), _ptr(x), _ptr(y), _ptr(workspace), workspace_bytes, E, H, I,
                           T, topk, _stream(stream)), "moe_layer")


def moe_layer_workspace_bytes(T, topk, H, I, E) -> int:
    return lib().moe_layer_workspace_bytes(T, topk, H, I, E)


def bqd_moe_read_status(workspace, stream=None) -> int:
    """Device status word of a MoE workspace (synchronising). Returns the bits."""
    out = C.c_int32(0)
    st = lib().bqd_moe_read_status(_ptr(workspace), C.byref(out), _stream(stream))
    if st not in (BQD_OK, 8):
        raise BqdError(st, "bqd_moe_read_status")
    return out.value
