"""C ABI checks that need no GPU: the library loads, exports every function
declared in include/bqd.h, and rejects bad arguments on the host before any
CUDA call (the documented status codes)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from block_quantized_decode_nvfp4_gb300 import build
    build.build()
    import block_quantized_decode_nvfp4_gb300 as bqd
    return bqd.lib()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "bqd.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("nvfp4_gemv", "q8_0_gemv", "moe_grouped_gemv", "moe_route_topk", "nvfp4_dequant",
                     "q8_0_dequant", "moe_workspace_bytes", "bqd_status_string", "bqd_moe_read_status"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    import block_quantized_decode_nvfp4_gb300._binding as b
    for name in _declared_functions():
        assert hasattr(L, name), name
        assert name in b.SIGNATURES, f"binding lacks {name}"


def test_status_strings(L):
    for code in range(9):
        assert L.bqd_status_string(code)
    assert L.bqd_status_string(99) == b"unknown status"
    assert L.bqd_version() >= 100


A = 0x10000  # a 16-byte aligned fake address: never dereferenced (every call below fails validation first)
U = 0x10008  # misaligned


def test_nvfp4_gemv_validation(L):
    s = None
    assert L.nvfp4_gemv(None, A, 1.0, A, A, 4, 32, 1, s) == 1          # NULL codes
    assert L.nvfp4_gemv(A, A, 1.0, A, None, 4, 32, 1, s) == 1          # NULL y
    assert L.nvfp4_gemv(A, A, 1.0, A, A, 4, 24, 1, s) == 2             # K % 16
    assert L.nvfp4_gemv(A, A, 1.0, A, A, -1, 32, 1, s) == 2            # M < 0
    assert L.nvfp4_gemv(A, A, 1.0, A, A, 4, 32, 0, s) == 2             # N < 1
    assert L.nvfp4_gemv(A, A, 1.0, A, A, 4, 32, 17, s) == 2            # N > 16
    assert L.nvfp4_gemv(U, A, 1.0, A, A, 4, 32, 1, s) == 3             # misaligned codes
    assert L.nvfp4_gemv(A, A, 1.0, U, A, 4, 32, 1, s) == 3             # misaligned x
    assert L.nvfp4_gemv(A, A, 1.0, A, U, 4, 32, 1, s) == 3             # misaligned y
    assert L.nvfp4_gemv(None, None, 1.0, None, None, 0, 32, 1, s) == 0  # M == 0: no work, no CUDA call
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 4, 32, 1, 99, s) == 7    # unknown path
    assert L.nvfp4_gemv(A, A, 1.0, A, A, 1 << 40, 1 << 30, 1, s) == 2  # M * K overflow


def test_compute_path_restrictions(L):
    # a path that does not take the arguments answers BQD_ERR_PATH (7) on
    # the host, before any CUDA call
    s, MMA, STREAM = None, 3, 2
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 256, 4112, 8, MMA, s) == 7      # K % 256 != 0
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 256, 128, 8, MMA, s) == 7       # K < 256
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 4, (1 << 20) + 256, 2, MMA, s) == 7  # K > 2^20
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 256, 65536, 16, MMA, s) == 7    # activations exceed shared memory
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 256, 4096, 2, STREAM, s) == 7   # stream path is N = 1 only
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 256, 16640, 1, STREAM, s) == 7  # K > 16384
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 256, 4112, 1, STREAM, s) == 7   # K % 256 != 0
    assert L.q8_0_gemv_path(A, A, A, A, 256, 4096, 4, MMA, s) == 7            # no tensor-core Q8_0 path
    assert L.q8_0_gemv_path(A, A, A, A, 256, 4096, 2, STREAM, s) == 7
    assert L.q8_0_gemv_path(A, A, A, A, 256, 4096, 1, 99, s) == 7
    # argument errors come before path errors
    assert L.nvfp4_gemv_path(A, A, 1.0, A, A, 256, 4096, 17, MMA, s) == 2


def test_q8_0_and_dequant_validation(L):
    s = None
    assert L.q8_0_gemv(A, A, A, A, 4, 48, 1, s) == 2                   # K % 32
    assert L.q8_0_gemv(A, None, A, A, 4, 64, 1, s) == 1
    assert L.q8_0_gemv(A, A, A, A, 4, 64, 17, s) == 2
    assert L.q8_0_gemv(A, U, A, A, 4, 64, 1, s) == 3
    assert L.nvfp4_dequant(A, A, 1.0, None, 4, 32, s) == 1
    assert L.nvfp4_dequant(A, A, 1.0, A, 4, 8, s) == 2
    assert L.q8_0_dequant(A, A, U, 4, 32, s) == 3
    assert L.q8_0_dequant(None, None, None, 0, 32, s) == 0


def test_moe_validation(L):
    s = None
    assert L.moe_route_topk(A, 1, 8, 9, A, A, A, A, s) == 2            # topk > E
    assert L.moe_route_topk(A, 1, 2000, 8, A, A, A, A, s) == 2         # E too large
    assert L.moe_route_topk(A, 2000, 256, 8, A, A, A, A, s) == 2       # T * topk > 8192
    assert L.moe_route_topk(A, 1, 256, 33, A, A, A, A, s) == 2         # topk > 32
    assert L.moe_route_topk(None, 1, 256, 8, A, A, A, A, s) == 1
    assert L.moe_route_topk(A, 1, 256, 8, A, U, A, A, s) == 3
    ws = L.moe_workspace_bytes(16, 8, 2048, 512)
    P = 128
    align = lambda n: (n + 255) // 256 * 256
    assert ws == 256 + 2 * align(4 * P) + align(4 * P * 512) + align(4 * P * 2048)
    args = [A] * 12
    assert L.moe_grouped_gemv(*args, None, ws, 256, 2048, 512, 16, 8, s) == 6      # no workspace
    assert L.moe_grouped_gemv(*args, A, ws - 1, 256, 2048, 512, 16, 8, s) == 6     # too small
    assert L.moe_grouped_gemv(*args, A + 16, ws, 256, 2048, 512, 16, 8, s) == 6    # not 256-aligned
    assert L.moe_grouped_gemv(*args, A, ws, 256, 2047, 512, 16, 8, s) == 2         # H % 32
    assert L.moe_grouped_gemv(*args, A, ws, 256, 2048, 500, 16, 8, s) == 2         # I % 32
    bad = list(args)
    bad[7] = None
    assert L.moe_grouped_gemv(*bad, A, ws, 256, 2048, 512, 16, 8, s) == 1
    bad[7] = U
    assert L.moe_grouped_gemv(*bad, A, ws, 256, 2048, 512, 16, 8, s) == 3
    out = C.c_int32(0)
    assert L.bqd_moe_read_status(None, C.byref(out), s) == 1


def test_binding_raises_on_error():
    import block_quantized_decode_nvfp4_gb300 as bqd
    with pytest.raises(bqd.BqdError) as ei:
        bqd.nvfp4_gemv(None, A, 1.0, A, A, 4, 32, 1, stream=0)
    assert ei.value.status == 1


def test_moe_layer_validation(L):
    s = None
    a = [A] * 9
    wsb = L.moe_layer_workspace_bytes(1, 8, 2048, 512, 256)
    assert wsb >= L.moe_workspace_bytes(1, 8, 2048, 512) + 257 * 4
    assert L.moe_layer(None, *a[1:], A, wsb, 256, 2048, 512, 1, 8, s) == 1          # NULL logits
    assert L.moe_layer(*a, A, wsb, 256, 2048, 512, 1, 0, s) == 2                    # topk < 1
    assert L.moe_layer(*a, A, wsb, 256, 2040, 512, 1, 8, s) == 2                    # H % 32
    assert L.moe_layer(*a, A, wsb - 1, 256, 2048, 512, 1, 8, s) == 6                # workspace too small
    assert L.moe_layer(*a, A + 16, wsb, 256, 2048, 512, 1, 8, s) == 6               # workspace misaligned
    assert L.moe_layer(*a[:8], U, A, wsb, 256, 2048, 512, 1, 8, s) == 3             # misaligned y
    assert L.moe_layer_workspace_bytes(0, 8, 2048, 512, 256) == 0


def test_format_entry_points_validation(L):
    # Q4_0, Q4_1 and FP8 block-128: shape, NULL, alignment and path errors on
    # the host, before any CUDA call
    s, CORE, MMA, DIRECT = None, 1, 3, 4
    for gemv in (L.q4_0_gemv, L.q4_1_gemv, L.fp8_b128_gemv):
        assert gemv(A, A, A, A, 4, 48, 1, s) == 2                        # K % 32
        assert gemv(A, A, A, A, 4, 64, 17, s) == 2                       # N > 16
        assert gemv(A, None, A, A, 4, 64, 1, s) == 1                     # NULL scales
        assert gemv(A, A, U, A, 4, 64, 1, s) == 3                        # misaligned x
        assert gemv(None, None, None, None, 0, 64, 1, s) == 0            # M == 0
    for path in (L.q4_0_gemv_path, L.fp8_b128_gemv_path):
        assert path(A, A, A, A, 4, 1024, 1, MMA, s) == 7                 # no tensor-core path
        assert path(A, A, A, A, 4, 96, 1, DIRECT, s) == 7                # K the direct kernel does not take
        assert path(A, A, A, A, 4, 1024, 2, DIRECT, s) == 7              # direct is N = 1 only
        assert path(A, A, A, A, 4, 48, 1, CORE, s) == 2                  # argument errors first
    for deq in (L.q4_0_dequant, L.q4_1_dequant, L.fp8_b128_dequant):
        assert deq(A, A, U, 4, 32, s) == 3
        assert deq(A, A, None, 4, 32, s) == 1
        assert deq(A, A, A, 4, 48, s) == 2
        assert deq(None, None, None, 0, 32, s) == 0


def test_fusion_and_encoder_validation(L):
    s = None
    assert L.nvfp4_gemv_add(A, A, 1.0, A, A, A, 4, 1536, 1, s) == 2     # K the direct kernel does not take
    assert L.nvfp4_gemv_add(A, A, 1.0, A, A, A, 4, 1024, 2, s) == 2     # N = 1 only
    assert L.nvfp4_gemv_add(A, A, 1.0, A, None, A, 4, 1024, 1, s) == 1  # no residual
    assert L.nvfp4_gemv_add(A, A, 1.0, A, U, A, 4, 1024, 1, s) == 3     # misaligned residual
    assert L.q8_0_gemv_add(A, A, A, A, A, 4, 1000, 1, s) == 2           # K % 32
    assert L.nvfp4_gemv_silu_mul(A, A, 1.0, A, A, 0, 1024, 1, s) == 2   # I = 0
    assert L.q8_0_gemv_silu_mul(A, A, A, A, 8, 1536, 1, s) == 2
    assert L.nvfp4_encode(A, 1.0, A, A, 4, 24, s) == 2                  # K % 16
    assert L.nvfp4_encode(A, float("nan"), A, A, 4, 32, s) == 2         # tensor scale NaN
    assert L.nvfp4_encode(A, 0.0, A, A, 4, 32, s) == 2                  # tensor scale 0
    assert L.nvfp4_encode(A, 1.0, None, A, 4, 32, s) == 1
    assert L.nvfp4_encode(U, 1.0, A, A, 4, 32, s) == 3
    assert L.nvfp4_encode(None, 1.0, None, None, 0, 32, s) == 0
    assert L.q8_0_encode(A, A, A, 4, 48, s) == 2
    assert L.q8_0_encode(A, A, A + 1, 4, 64, s) == 3                    # odd fp16 plane


def test_prefill_entry_points_validation(L):
    s = None
    assert L.nvfp4_gemm(A, A, 1.0, A, A, 4, 32, 8, s) == 2              # K % 64
    assert L.nvfp4_gemm(A, A, 1.0, A, A, -1, 64, 8, s) == 2
    assert L.nvfp4_gemm(A, A, 1.0, A, None, 4, 64, 8, s) == 1           # NULL y
    assert L.nvfp4_gemm(A, A, 1.0, A, U, 4, 64, 8, s) == 3
    assert L.nvfp4_gemm(None, None, 1.0, None, None, 4, 64, 0, s) == 0  # T == 0
    g = L.nvfp4_gemm_grouped
    assert g(A, A, A, A, A, A, 0, 32, 64, 8, s) == 2                    # E < 1
    assert g(A, A, A, A, A, A, 2, 32, 96, 8, s) == 2                    # K % 64
    assert g(A, A, A, A, A, None, 2, 32, 64, 8, s) == 1
    assert g(A, A, A, A, A, U, 2, 32, 64, 8, s) == 3
    assert g(None, None, None, None, None, None, 2, 0, 64, 8, s) == 0   # M == 0
    wsb = L.moe_prefill_workspace_bytes(1024, 8, 2048, 512, 256)
    assert wsb >= 8192 * (6 * 2048 + 12 * 512)
    assert L.moe_prefill_workspace_bytes(0, 8, 2048, 512, 256) == 0
    a = [A] * 9
    lay = L.moe_prefill_layer
    assert lay(*a, A, wsb, 256, 2048, 512, 1025, 8, s) == 2             # T * topk > 8192
    assert lay(*a, A, wsb, 256, 2000, 512, 16, 8, s) == 2               # H % 64
    assert lay(*a, A, wsb, 256, 2048, 32, 16, 8, s) == 2                # I < 64
    assert lay(*a, A, wsb, 2048, 2048, 512, 16, 8, s) == 2              # E > 1024
    assert lay(*a, A, wsb, 4, 2048, 512, 16, 8, s) == 2                 # topk > E
    assert lay(None, *a[1:], A, wsb, 256, 2048, 512, 16, 8, s) == 1     # NULL logits
    small = L.moe_prefill_workspace_bytes(16, 8, 2048, 512, 256)
    assert lay(*a, A, small - 1, 256, 2048, 512, 16, 8, s) == 6         # workspace too small
    assert lay(*a, A + 8, small, 256, 2048, 512, 16, 8, s) == 3         # misaligned workspace
    bad = list(a)
    bad[3] = A + 2                                                      # gate/up tensor scales not 4-byte aligned
    assert lay(*bad, A, small, 256, 2048, 512, 16, 8, s) == 3
