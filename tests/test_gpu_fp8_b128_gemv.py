"""FP8 block-128 GEMV and dequantisation on the GPU against the fp64 oracle,
through the C ABI (tolerance as for NVFP4: |y - y_ref| <= 1e-3 * sum|w x| +
1e-6; dequantisation and exact invariants bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.gpu_util import Guarded, assert_within, dev, need_gpu
from tests.test_oracle_fp8_b128 import _build_worked

pytestmark = pytest.mark.gpu

DIRECT, CUDA_CORE = "direct", "cuda_core"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert bqd.bqd_device_error() == 0, "a pipeline wait ran out"


def _path(p):
    return {None: None, DIRECT: bqd.BQD_PATH_DIRECT, CUDA_CORE: bqd.BQD_PATH_CUDA_CORE}[p]


def run(w, codes=None, scales=None, x=None, path=None):
    M, K = w["M"], w["K"]
    xx = w["x"] if x is None else x
    N = xx.shape[0]
    out = Guarded(N * M)
    c = dev(w["codes"] if codes is None else codes)
    s = dev(w["scales"] if scales is None else scales)
    if path is None:
        bqd.fp8_b128_gemv(c, s, dev(xx), out.ptr, M, K, N)
    else:
        bqd.fp8_b128_gemv_path(c, s, dev(xx), out.ptr, M, K, N, _path(path))
    return out.get().reshape(N, M)


def check(w, rows=None, what="", path=None):
    y = run(w, path=path)
    ref, a = oracle.fp8_b128_gemv(w["codes"], w["scales"], w["x"], w["M"], w["K"], rows=rows)
    assert_within(y if rows is None else y[:, rows], ref, a, what)
    return y


def _worked(golden, K=None):
    M, K0, codes, scales, x = _build_worked(golden("fp8_b128_worked_example.txt"))
    if K is not None and K > K0:  # zero codes and activations past K0, unit scales for the new tiles
        codes = np.concatenate([codes, np.zeros((M, K - K0), dtype=np.uint8)], axis=1)
        x = np.concatenate([x, np.zeros((1, K - K0), dtype=np.uint16)], axis=1)
        scales = np.concatenate([scales, np.ones((scales.shape[0], (K - K0) // 128), dtype=np.float32)], axis=1)
    else:
        K = K0
    return {"M": M, "K": K, "codes": codes, "scales": scales, "x": x}


@pytest.mark.parametrize("K,path", [(None, None), (1024, DIRECT), (1024, CUDA_CORE)])
def test_worked_example(golden, K, path):
    # the hand-worked rows across both tile boundaries (rows 127 / 128, k 127 / 128)
    g = golden("fp8_b128_worked_example.txt")
    w = _worked(golden, K)
    y = run(w, path=path)
    want_y, want_a = np.zeros(w["M"]), np.zeros(w["M"])
    for m, yv, av in g["y"]:
        want_y[int(m)], want_a[int(m)] = float(yv), float(av)
    assert_within(y[0], want_y, want_a, f"worked K={w['K']} {path}")


def test_dequant_bit_exact():
    M, K = 300, 1056  # a partial last tile row and tile column
    w = syn.dense_fp8_b128(M, K, seed=3)
    w["codes"][0, :6] = [0x01, 0x7E, 0x80, 0xFE, 0x08, 0x07]  # smallest subnormal, 448, -0, -448, 2^-6, 7 * 2^-9
    w["scales"][0, 0] = 2.0 ** -126                            # results in fp32's subnormal range
    out = torch.full((M * K,), float("nan"), dtype=torch.float32, device="cuda")
    bqd.fp8_b128_dequant(dev(w["codes"]), dev(w["scales"]), out, M, K)
    ref = oracle.fp8_b128_dequant(w["codes"], w["scales"], M, K, dtype=np.float32)
    assert np.array_equal(out.cpu().numpy().reshape(M, K).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("M,K,N", [
    (1, 32, 1), (127, 128, 3), (129, 160, 5), (300, 4096, 1), (513, 1024, 8), (64, 2048, 16),
    (200, 8192, 9), (90, 12288, 16), (1000, 96, 2), (7, 1024, 1), (333, 3072, 1), (77, 16384, 1),
    (257, 4128, 1),
])
def test_edge_shapes(M, K, N):
    check(syn.dense_fp8_b128(M, K, N=N, seed=M + K + N), what=f"{M}x{K} N={N}")


@pytest.mark.parametrize("M,K", syn.FP8_B128_SHAPES)
def test_full_size_n1(M, K):
    check(syn.dense_fp8_b128(M, K, N=1, seed=0), what=f"{M}x{K}")


def test_full_size_verify_sampled_rows():
    M, K = 12288, 4096
    w = syn.dense_fp8_b128(M, K, N=8, seed=1)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, M - 1], np.random.default_rng(5).choice(M, 1024, replace=False)]))
    check(w, rows=rows, what=f"{M}x{K} N=8")


@pytest.mark.parametrize("M,K", [(1, 1024), (700, 4096), (4864, 4096), (33, 12288), (70, 3072), (9, 6144)])
def test_direct_and_cuda_core_paths_match_oracle(M, K):
    w = syn.dense_fp8_b128(M, K, N=1, seed=M + 2 * K)
    ref, a = oracle.fp8_b128_gemv(w["codes"], w["scales"], w["x"], M, K)
    for path in (DIRECT, CUDA_CORE):
        assert_within(run(w, path=path), ref, a, f"{M}x{K} {path}")


@pytest.mark.parametrize("path", [DIRECT, CUDA_CORE])
def test_exact_invariants(path):
    """One-hot x gives the dequantised column bit for bit; zero codes give
    zero; the sign bit negates y exactly; a NaN code spoils its row only."""
    M, K = 700, 4096
    w = syn.dense_fp8_b128(M, K, N=1, seed=13)
    W = oracle.fp8_b128_dequant(w["codes"], w["scales"], M, K, dtype=np.float32)
    for k in (0, 31, 32, 127, 128, 2047, 2048, 4095):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80
        assert np.array_equal(run(w, x=x, path=path)[0], W[:, k]), f"one-hot k={k}"
    assert np.all(run(w, codes=np.zeros_like(w["codes"]), path=path) == 0)
    assert np.array_equal(run(w, codes=w["codes"] ^ np.uint8(0x80), path=path), -run(w, path=path))
    c = w["codes"].copy()
    c[5, 100] = 0x7F
    y = run(w, codes=c, path=path)[0]
    assert np.isnan(y[5]) and np.all(np.isfinite(np.delete(y, 5)))


def test_scales_shared_by_row_tiles():
    # one tile's scale doubled (a power of two): rows outside its 128-row
    # tile are unchanged bit for bit, rows inside stay within the bound
    M, K = 384, 4096
    w = syn.dense_fp8_b128(M, K, N=1, seed=17)
    s2 = w["scales"].copy()
    s2[1, 5] *= 2.0
    y0, y1 = run(w), run(w, scales=s2)
    out = np.r_[0:128, 256:384]
    assert np.array_equal(y0[0, out].view(np.uint32), y1[0, out].view(np.uint32))
    ref, a = oracle.fp8_b128_gemv(w["codes"], s2, w["x"], M, K)
    assert_within(y1, ref, a, "doubled tile")


def test_wide_activation_range_and_determinism():
    M, K = 512, 4096
    w = syn.dense_fp8_b128(M, K, N=1, seed=21)
    x = w["x"].copy()
    x[0, 10] = 0x7000  # 2^97: far outside the others' f16-exact range
    x[0, 11] = 0x0001  # a bf16 subnormal
    check(dict(w, x=x), what="wide range")
    assert np.array_equal(run(w).view(np.uint32), run(w).view(np.uint32))


def test_rejections():
    w = syn.dense_fp8_b128(16, 1024, seed=1)
    out = Guarded(16)
    c, s = dev(w["codes"]), dev(w["scales"])
    with pytest.raises(bqd.BqdError):  # K % 32 != 0
        bqd.fp8_b128_gemv(c, s, dev(w["x"]), out.ptr, 16, 1000, 1)
    with pytest.raises(bqd.BqdError):  # direct path at a K it does not take
        bqd.fp8_b128_gemv_path(c, s, dev(w["x"][:, :96]), out.ptr, 16, 96, 1, bqd.BQD_PATH_DIRECT)
    with pytest.raises(bqd.BqdError):  # no tensor-core path for FP8 block-128
        bqd.fp8_b128_gemv_path(c, s, dev(w["x"]), out.ptr, 16, 1024, 1, bqd.BQD_PATH_MMA)
    with pytest.raises(bqd.BqdError):  # N = 17
        bqd.fp8_b128_gemv(c, s, dev(np.repeat(w["x"], 17, 0)), out.ptr, 16, 1024, 17)
    e = Guarded(6, fill=5.0)
    bqd.fp8_b128_gemv(None, None, None, e.ptr, 3, 0, 2)  # K == 0: zeros
    assert np.all(e.get() == 0)
