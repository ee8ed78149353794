"""Q4_0 GEMV and dequantisation on the GPU against the fp64 oracle, through
the C ABI (tolerance as for NVFP4: |y - y_ref| <= 1e-3 * sum|w x| + 1e-6;
dequantisation and exact invariants bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.gpu_util import Guarded, assert_within, dev, need_gpu
from tests.test_oracle_q4_0 import _build_worked

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert bqd.bqd_device_error() == 0, "a pipeline wait ran out"


def run(w, codes=None, x=None, path=None):
    M, K = w["M"], w["K"]
    xx = w["x"] if x is None else x
    N = xx.shape[0]
    out = Guarded(N * M)
    c = dev(w["codes"] if codes is None else codes)
    if path is None:
        bqd.q4_0_gemv(c, dev(w["d"]), dev(xx), out.ptr, M, K, N)
    else:
        bqd.q4_0_gemv_path(c, dev(w["d"]), dev(xx), out.ptr, M, K, N, path)
    return out.get().reshape(N, M)


def check(w, rows=None, what="", path=None):
    y = run(w, path=path)
    ref, a = oracle.q4_0_gemv(w["codes"], w["d"], w["x"], w["M"], w["K"], rows=rows)
    assert_within(y if rows is None else y[:, rows], ref, a, what)
    return y


def test_worked_example(golden):
    g = golden("q4_0_worked_example.txt")
    M, K, codes, d, x = _build_worked(g)
    y = run({"M": M, "K": K, "codes": codes, "d": d, "x": x})
    assert_within(y[0], np.array([float(v) for v in g["y"][0]]), np.array([float(v) for v in g["a"][0]]), "worked")


def test_dequant_bit_exact():
    M, K = 300, 1024
    w = syn.dense_q4_0(M, K, seed=3)
    w["d"][0, :4] = [0x0001, 0x7BFF, 0x8000, 0xBC00]  # subnormal, largest, -0, -1
    out = torch.full((M * K,), float("nan"), dtype=torch.float32, device="cuda")
    bqd.q4_0_dequant(dev(w["codes"]), dev(w["d"]), out, M, K)
    ref = oracle.q4_0_dequant(w["codes"], w["d"], M, K, dtype=np.float32)
    assert np.array_equal(out.cpu().numpy().reshape(M, K).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("M,K,N", [
    (1, 32, 1), (127, 64, 3), (129, 512, 5), (300, 4096, 1), (513, 1024, 8), (64, 2048, 16),
    (200, 8192, 9), (90, 12288, 16), (1000, 96, 2), (7, 1024, 1), (333, 3072, 1), (77, 16384, 1),
])
def test_edge_shapes(M, K, N):
    check(syn.dense_q4_0(M, K, N=N, seed=M + K + N), what=f"{M}x{K} N={N}")


@pytest.mark.parametrize("M,K", syn.Q4_0_SHAPES)
def test_full_size_n1(M, K):
    check(syn.dense_q4_0(M, K, N=1, seed=0), what=f"{M}x{K}")


@pytest.mark.parametrize("M,K", [(4096, 4096), (12288, 4096)])
def test_full_size_verify_sampled_rows(M, K):
    w = syn.dense_q4_0(M, K, N=8, seed=1)
    rows = np.unique(np.concatenate([[0, 1, M - 1], np.random.default_rng(5).choice(M, 1024, replace=False)]))
    check(w, rows=rows, what=f"{M}x{K} N=8")


@pytest.mark.parametrize("M,K", [(1, 1024), (700, 4096), (4864, 4096), (33, 12288), (70, 3072), (9, 6144)])
def test_direct_and_cuda_core_paths_match_oracle(M, K):
    w = syn.dense_q4_0(M, K, N=1, seed=M + 2 * K)
    ref, a = oracle.q4_0_gemv(w["codes"], w["d"], w["x"], M, K)
    for path in (bqd.BQD_PATH_DIRECT, bqd.BQD_PATH_CUDA_CORE):
        assert_within(run(w, path=path), ref, a, f"{M}x{K} path {path}")


@pytest.mark.parametrize("path", ["direct", "cuda_core"])
def test_exact_invariants(path):
    """One-hot x gives the dequantised column bit for bit; code 8 everywhere
    gives zero; q -> 16 - q negates y exactly."""
    M, K = 700, 4096
    P = bqd.BQD_PATH_DIRECT if path == "direct" else bqd.BQD_PATH_CUDA_CORE
    w = syn.dense_q4_0(M, K, N=1, seed=13)
    W = oracle.q4_0_dequant(w["codes"], w["d"], M, K, dtype=np.float32)
    for k in (0, 15, 16, 31, 32, 47, 48, 2048, 4095):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80
        assert np.array_equal(run(w, x=x, path=P)[0], W[:, k]), f"one-hot k={k}"
    assert np.all(run(w, codes=np.full_like(w["codes"], 0x88), path=P) == 0)
    lo, hi = np.maximum(w["codes"] & 0x0F, 1), np.maximum(w["codes"] >> 4, 1)
    c1 = (lo | (hi << 4)).astype(np.uint8)
    c2 = ((16 - lo) | ((16 - hi) << 4)).astype(np.uint8)
    assert np.array_equal(run(w, codes=c2, path=P), -run(w, codes=c1, path=P))


def test_wide_activation_range_and_determinism():
    M, K = 512, 4096
    w = syn.dense_q4_0(M, K, N=1, seed=21)
    x = w["x"].copy()
    x[0, 10] = 0x7000  # 2^97: far outside the others' f16-exact range
    x[0, 11] = 0x0001  # a bf16 subnormal
    check(dict(w, x=x), what="wide range")
    assert np.array_equal(run(w).view(np.uint32), run(w).view(np.uint32))


def test_rejections():
    w = syn.dense_q4_0(16, 1024, seed=1)
    out = Guarded(16)
    with pytest.raises(bqd.BqdError):  # K % 32 != 0
        bqd.q4_0_gemv(dev(w["codes"]), dev(w["d"]), dev(w["x"]), out.ptr, 16, 1000, 1)
    with pytest.raises(bqd.BqdError):  # direct path at a K it does not take
        bqd.q4_0_gemv_path(dev(w["codes"]), dev(w["d"]), dev(w["x"][:, :96]), out.ptr, 16, 96, 1,
                           bqd.BQD_PATH_DIRECT)
    with pytest.raises(bqd.BqdError):  # no tensor-core path for Q4_0
        bqd.q4_0_gemv_path(dev(w["codes"]), dev(w["d"]), dev(w["x"]), out.ptr, 16, 1024, 1, bqd.BQD_PATH_MMA)
    with pytest.raises(bqd.BqdError):  # N = 17
        bqd.q4_0_gemv(dev(w["codes"]), dev(w["d"]), dev(np.repeat(w["x"], 17, 0)), out.ptr, 16, 1024, 17)
    e = Guarded(6, fill=5.0)
    bqd.q4_0_gemv(None, None, None, e.ptr, 3, 0, 2)  # K == 0: zeros
    assert np.all(e.get() == 0)
