"""fp64 CPU oracle for the block-quantized decode matvec (test infrastructure).

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg may import this package. It wraps oracle.c (built by oracle/build.py) with
ctypes and numpy arrays; it shares nothing with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        u8p, i8p, u16p = C.POINTER(C.c_uint8), C.POINTER(C.c_int8), C.POINTER(C.c_uint16)
        f32p, f64p, i32p, i64p = (C.POINTER(C.c_float), C.POINTER(C.c_double),
                                  C.POINTER(C.c_int32), C.POINTER(C.c_int64))
        i64 = C.c_int64
        for name, res, args in [
            ("oracle_e2m1", C.c_double, [C.c_uint8]),
            ("oracle_e4m3", C.c_double, [C.c_uint8]),
            ("oracle_fp16", C.c_double, [C.c_uint16]),
            ("oracle_bf16", C.c_double, [C.c_uint16]),
            ("oracle_nvfp4_dequant_f64", None, [u8p, u8p, C.c_float, i64, i64, f64p]),
            ("oracle_nvfp4_dequant_f32", None, [u8p, u8p, C.c_float, i64, i64, f32p]),
            ("oracle_q8_0_dequant_f64", None, [i8p, u16p, i64, i64, f64p]),
            ("oracle_q8_0_dequant_f32", None, [i8p, u16p, i64, i64, f32p]),
            ("oracle_nvfp4_gemv", None, [u8p, u8p, C.c_float, u16p, i64, i64, i64, i64p, i64, f64p, f64p]),
            ("oracle_nvfp4_gemv_f64x", None, [u8p, u8p, C.c_float, f64p, i64, i64, i64, f64p, f64p]),
            ("oracle_q8_0_gemv", None, [i8p, u16p, u16p, i64, i64, i64, i64p, i64, f64p, f64p]),
            ("oracle_q4_0_dequant_f64", None, [u8p, u16p, i64, i64, f64p]),
            ("oracle_q4_0_dequant_f32", None, [u8p, u16p, i64, i64, f32p]),
            ("oracle_q4_0_gemv", None, [u8p, u16p, u16p, i64, i64, i64, i64p, i64, f64p, f64p]),
            ("oracle_q4_1_dequant_f64", None, [u8p, u16p, i64, i64, f64p]),
            ("oracle_q4_1_dequant_f32", None, [u8p, u16p, i64, i64, f32p]),
            ("oracle_q4_1_gemv", None, [u8p, u16p, u16p, i64, i64, i64, i64p, i64, f64p, f64p]),
            ("oracle_fp8_b128_dequant_f64", None, [u8p, f32p, i64, i64, f64p]),
            ("oracle_fp8_b128_dequant_f32", None, [u8p, f32p, i64, i64, f32p]),
            ("oracle_fp8_b128_gemv", None, [u8p, f32p, u16p, i64, i64, i64, i64p, i64, f64p, f64p]),
            ("oracle_moe_route", None, [f32p, i64, i64, i64, i32p, f64p]),
            ("oracle_moe_layer", None, [u8p, u8p, f32p, u8p, u8p, f32p, u16p, i32p, f64p,
                                        i64, i64, i64, i64] + [f64p] * 8),
        ]:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(C.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- decoders
def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def e4m3(b: int) -> float:
    return lib().oracle_e4m3(b)


def fp16(h: int) -> float:
    return lib().oracle_fp16(h)


def bf16(b: int) -> float:
    return lib().oracle_bf16(b)


# ---------------------------------------------------------------- dequant
def nvfp4_dequant(codes, scales, ts, M, K, dtype=np.float64):
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    w = np.empty((M, K), dtype=dtype)
    if dtype == np.float64:
        lib().oracle_nvfp4_dequant_f64(_p(codes, C.c_uint8), _p(scales, C.c_uint8), ts, M, K, _p(w, C.c_double))
    else:
        lib().oracle_nvfp4_dequant_f32(_p(codes, C.c_uint8), _p(scales, C.c_uint8), ts, M, K, _p(w, C.c_float))
    return w


def q8_0_dequant(q, d, M, K, dtype=np.float64):
    q, d = _c(q, np.int8), _c(d, np.uint16)
    w = np.empty((M, K), dtype=dtype)
    if dtype == np.float64:
        lib().oracle_q8_0_dequant_f64(_p(q, C.c_int8), _p(d, C.c_uint16), M, K, _p(w, C.c_double))
    else:
        lib().oracle_q8_0_dequant_f32(_p(q, C.c_int8), _p(d, C.c_uint16), M, K, _p(w, C.c_float))
    return w


def q4_0_dequant(codes, d, M, K, dtype=np.float64):
    """Q4_0 weight [M][K]: fp16(d) * (q - 8), q from the GGUF block order
    (element j < 16 of a 32-block: low nibble of code byte j; j >= 16: high
    nibble of byte j - 16)."""
    codes, d = _c(codes, np.uint8), _c(d, np.uint16)
    w = np.empty((M, K), dtype=dtype)
    if dtype == np.float64:
        lib().oracle_q4_0_dequant_f64(_p(codes, C.c_uint8), _p(d, C.c_uint16), M, K, _p(w, C.c_double))
    else:
        lib().oracle_q4_0_dequant_f32(_p(codes, C.c_uint8), _p(d, C.c_uint16), M, K, _p(w, C.c_float))
    return w


def q4_1_dequant(codes, dm, M, K, dtype=np.float64):
    """Q4_1 weight [M][K]: fp16(d) * q + fp16(m) per 32-block, q in the
    Q4_0 block order, dm [M][K/32][2] = the block's (d, m) fp16 bits."""
    codes, dm = _c(codes, np.uint8), _c(dm, np.uint16)
    w = np.empty((M, K), dtype=dtype)
    if dtype == np.float64:
        lib().oracle_q4_1_dequant_f64(_p(codes, C.c_uint8), _p(dm, C.c_uint16), M, K, _p(w, C.c_double))
    else:
        lib().oracle_q4_1_dequant_f32(_p(codes, C.c_uint8), _p(dm, C.c_uint16), M, K, _p(w, C.c_float))
    return w


def fp8_b128_dequant(codes, scales, M, K, dtype=np.float64):
    """FP8 block-128 weight [M][K]: e4m3(code) * the fp32 scale of the
    128 x 128 tile holding the element (scales [ceil(M/128)][ceil(K/128)])."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.float32)
    w = np.empty((M, K), dtype=dtype)
    if dtype == np.float64:
        lib().oracle_fp8_b128_dequant_f64(_p(codes, C.c_uint8), _p(scales, C.c_float), M, K, _p(w, C.c_double))
    else:
        lib().oracle_fp8_b128_dequant_f32(_p(codes, C.c_uint8), _p(scales, C.c_float), M, K, _p(w, C.c_float))
    return w


# ---------------------------------------------------------------- GEMV
def nvfp4_gemv(codes, scales, ts, x, M, K, rows=None):
    """(y, a) as fp64 arrays [N][len(rows) or M]; x is bf16 bits [N][K]."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    x = _c(x, np.uint16).reshape(-1, K)
    N = x.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    R = M if r is None else len(r)
    y = np.empty((N, R)); a = np.empty((N, R))
    lib().oracle_nvfp4_gemv(_p(codes, C.c_uint8), _p(scales, C.c_uint8), ts, _p(x, C.c_uint16),
                            M, K, N, _p(r, C.c_int64), 0 if r is None else len(r),
                            _p(y, C.c_double), _p(a, C.c_double))
    return y, a


def nvfp4_gemv_f64x(codes, scales, ts, x, M, K):
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    x = _c(x, np.float64).reshape(-1, K)
    N = x.shape[0]
    y = np.empty((N, M)); a = np.empty((N, M))
    lib().oracle_nvfp4_gemv_f64x(_p(codes, C.c_uint8), _p(scales, C.c_uint8), ts, _p(x, C.c_double),
                                 M, K, N, _p(y, C.c_double), _p(a, C.c_double))
    return y, a


def q8_0_gemv(q, d, x, M, K, rows=None):
    q, d = _c(q, np.int8), _c(d, np.uint16)
    x = _c(x, np.uint16).reshape(-1, K)
    N = x.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    R = M if r is None else len(r)
    y = np.empty((N, R)); a = np.empty((N, R))
    lib().oracle_q8_0_gemv(_p(q, C.c_int8), _p(d, C.c_uint16), _p(x, C.c_uint16), M, K, N,
                           _p(r, C.c_int64), 0 if r is None else len(r),
                           _p(y, C.c_double), _p(a, C.c_double))
    return y, a


def q4_0_gemv(codes, d, x, M, K, rows=None):
    codes, d = _c(codes, np.uint8), _c(d, np.uint16)
    x = _c(x, np.uint16).reshape(-1, K)
    N = x.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    R = M if r is None else len(r)
    y = np.empty((N, R)); a = np.empty((N, R))
    lib().oracle_q4_0_gemv(_p(codes, C.c_uint8), _p(d, C.c_uint16), _p(x, C.c_uint16), M, K, N,
                           _p(r, C.c_int64), 0 if r is None else len(r),
                           _p(y, C.c_double), _p(a, C.c_double))
    return y, a


def q4_1_gemv(codes, dm, x, M, K, rows=None):
    codes, dm = _c(codes, np.uint8), _c(dm, np.uint16)
    x = _c(x, np.uint16).reshape(-1, K)
    N = x.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    R = M if r is None else len(r)
    y = np.empty((N, R)); a = np.empty((N, R))
    lib().oracle_q4_1_gemv(_p(codes, C.c_uint8), _p(dm, C.c_uint16), _p(x, C.c_uint16), M, K, N,
                           _p(r, C.c_int64), 0 if r is None else len(r),
                           _p(y, C.c_double), _p(a, C.c_double))
    return y, a


def fp8_b128_gemv(codes, scales, x, M, K, rows=None):
    codes, scales = _c(codes, np.uint8), _c(scales, np.float32)
    x = _c(x, np.uint16).reshape(-1, K)
    N = x.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    R = M if r is None else len(r)
    y = np.empty((N, R)); a = np.empty((N, R))
    lib().oracle_fp8_b128_gemv(_p(codes, C.c_uint8), _p(scales, C.c_float), _p(x, C.c_uint16), M, K, N,
                               _p(r, C.c_int64), 0 if r is None else len(r),
                               _p(y, C.c_double), _p(a, C.c_double))
    return y, a


# ---------------------------------------------------------------- decode-path epilogues
def _gemv(fmt, w, x, M, K, rows):
    if fmt == "nvfp4":
        codes, scales, ts = w
        return nvfp4_gemv(codes, scales, ts, x, M, K, rows=rows)
    q, d = w
    return q8_0_gemv(q, d, x, M, K, rows=rows)


def gemv_add(fmt, w, x, r, M, K, rows=None):
    """y = W x + r for a residual r (fp32 [N][M]), the dense GEMV's residual
    epilogue ("Vemloir/LumenLLM" README, Kernels bullet: the decode path's
    fused epilogues). fmt "nvfp4" with w = (codes, scales, ts) or "q8_0" with
    w = (q, d). Returns (y, a): y fp64 [N][len(rows) or M], a = sum|w x|."""
    y, a = _gemv(fmt, w, x, M, K, rows)
    r = np.asarray(r, dtype=np.float32).reshape(y.shape[0], -1).astype(np.float64)
    if rows is not None:
        r = r[:, np.asarray(rows)]
    return y + r, a


def silu(g):
    """SiLU(g) = g / (1 + e^-g), fp64."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def gemv_silu_mul(fmt, w, x, I, K, rows=None):
    """h_i = SiLU(g_i) u_i with g = rows 0..I-1 and u = rows I..2I-1 of the
    gate_up weight times x: a dense MLP's first projection with its
    activation fused ("Vemloir/LumenLLM" README, Kernels bullet). Returns
    (h, g, u, ag, au), fp64 [N][len(rows) or I]."""
    rows = np.arange(I) if rows is None else np.asarray(rows, dtype=np.int64)
    g, ag = _gemv(fmt, w, x, 2 * I, K, rows)
    u, au = _gemv(fmt, w, x, 2 * I, K, rows + I)
    return silu(g) * u, g, u, ag, au


# ---------------------------------------------------------------- MoE
def moe_route(logits, topk):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    if not 0 < topk <= E:
        raise ValueError("need 0 < topk <= E")
    sel = np.empty((T, topk), dtype=np.int32)
    w = np.empty((T, topk))
    lib().oracle_moe_route(_p(logits, C.c_float), T, E, topk, _p(sel, C.c_int32), _p(w, C.c_double))
    return sel, w


def moe_layer(layer: dict, sel=None, weights=None, want_parts: bool = False):
    """Routed MoE FFN of a layer dict (synthetic.moe_layer layout).

    Returns y [T][H] (fp64) and, with want_parts, a dict of the stage values
    g, u, h, ag, au [T][topk][I] and d, ad [T][topk][H].
    """
    T, H, I, topk = layer["T"], layer["H"], layer["I"], layer["topk"]
    if sel is None:
        sel, weights = moe_route(layer["logits"], topk)
    sel = _c(sel, np.int32); weights = _c(weights, np.float64)
    y = np.empty((T, H))
    parts = {k: (np.empty((T, topk, I)) if want_parts else None) for k in ("g", "u", "h", "ag", "au")}
    parts.update({k: (np.empty((T, topk, H)) if want_parts else None) for k in ("d", "ad")})
    arr = [_c(layer[k], t) for k, t in (("gu_codes", np.uint8), ("gu_scales", np.uint8), ("gu_ts", np.float32),
                                        ("dn_codes", np.uint8), ("dn_scales", np.uint8), ("dn_ts", np.float32),
                                        ("x", np.uint16))]
    lib().oracle_moe_layer(_p(arr[0], C.c_uint8), _p(arr[1], C.c_uint8), _p(arr[2], C.c_float),
                           _p(arr[3], C.c_uint8), _p(arr[4], C.c_uint8), _p(arr[5], C.c_float),
                           _p(arr[6], C.c_uint16), _p(sel, C.c_int32), _p(weights, C.c_double),
                           T, H, I, topk, _p(y, C.c_double),
                           *[_p(parts[k], C.c_double) for k in ("g", "u", "h", "ag", "au", "d", "ad")])
    if want_parts:
        return y, parts
    return y


# ---------------------------------------------------------------- encoders (bf16 -> NVFP4 / Q8_0)
# Re-encoding bf16 weights at load ("robertbfuentes7-cloud/bw24" README,
# safetensors loader bullet: large tensors re-encode to Q8_0 / NVFP4 at
# load). Every decision is taken on fp32 values computed with IEEE fp32
# operations (round to nearest even), as the GPU encoder takes them; the
# conversions to E4M3, E2M1 and fp16 round to nearest, ties to even, and
# saturate (E4M3 at 448, E2M1 at 6).

def _rn_grid(v, grid):
    """Index of the nearest grid value to |v| (grid ascending, nonnegative),
    ties to the even index; |v| above the grid's top saturates to it."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    g = np.asarray(grid, dtype=np.float64)
    d = np.abs(a[..., None] - g)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    idx = np.argmax(cand, axis=-1)  # the lowest index at the minimum distance
    two = cand.sum(axis=-1) > 1  # a tie (two grid values at the same distance)
    idx = np.where(two & (idx % 2 == 1), idx + 1, idx)
    return np.where(a >= g[-1], len(g) - 1, idx)


def e4m3_positive_grid():
    """The 127 nonnegative finite E4M3 values, code order (code = index)."""
    return np.array([e4m3(c) for c in range(0x7F)])


def e2m1_positive_grid():
    return np.array([e2m1(c) for c in range(8)])


def e4m3_encode(v):
    """E4M3 codes of nonnegative fp32 values (RN-even, saturating at 448)."""
    return _rn_grid(v, e4m3_positive_grid()).astype(np.uint8)


def e2m1_encode(v):
    """E2M1 codes of fp32 values (RN-even, saturating at 6; the sign bit
    follows the value's sign, so a negative value that rounds to zero is -0)."""
    v = np.asarray(v, dtype=np.float32)
    mag = _rn_grid(v, e2m1_positive_grid()).astype(np.uint8)
    return (np.signbit(v).astype(np.uint8) << 3) | mag


def nvfp4_encode(w, ts, M, K):
    """(codes u8 [M][K/2], scales u8 [M][K/16]) of bf16 bits w [M][K]:
    per 16-element block, s = E4M3(amax / 6 / ts) and element code =
    E2M1(w / (e4m3(s) * ts)), all in fp32; a zero scale gives zero codes."""
    x = np.asarray(w, dtype=np.uint16).reshape(M, K // 16, 16)
    wf = (x.astype(np.uint32) << 16).view(np.float32)
    ts = np.float32(ts)
    amax = np.abs(wf).max(axis=-1)
    s32 = (amax / np.float32(6)) / ts
    sc = e4m3_encode(s32)
    sdec = np.array([e4m3(c) for c in range(256)], dtype=np.float64).astype(np.float32)[sc]
    den = (sdec * ts).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (wf / den[..., None]).astype(np.float32)
    codes = np.where(sdec[..., None] == 0, np.uint8(0), e2m1_encode(q))
    codes = codes.reshape(M, K // 2, 2)
    packed = (codes[..., 0] | (codes[..., 1] << 4)).astype(np.uint8)
    return packed, sc.astype(np.uint8)


def q8_0_encode(w, M, K):
    """(q i8 [M][K], d fp16 bits [M][K/32]) of bf16 bits w [M][K]: per
    32-element block d = fp16(amax / 127) and q = rint(w / d) in [-127, 127],
    all in fp32; a zero d gives q = 0."""
    x = np.asarray(w, dtype=np.uint16).reshape(M, K // 32, 32)
    wf = (x.astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(wf).max(axis=-1)
    d16 = (amax / np.float32(127)).astype(np.float16)
    d32 = d16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(wf / d32[..., None])
    q = np.where(d32[..., None] == 0, 0, np.clip(q, -127, 127)).astype(np.int8)
    return q.reshape(M, K), d16.view(np.uint16).reshape(M, K // 32)
