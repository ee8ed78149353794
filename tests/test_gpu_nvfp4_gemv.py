"""NVFP4 GEMV on the GPU against the fp64 oracle: the method's tolerance
|y - y_ref| <= 1e-3 * sum|w x| + 1e-6 per output, plus exact invariants."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.gpu_util import Guarded, assert_within, dev, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run(w, N=None, path=None):
    M, K = w["M"], w["K"]
    N = N or w["x"].shape[0]
    out = Guarded(N * M)
    args = (dev(w["codes"]), dev(w["scales"]), w["ts"], dev(w["x"]), out.ptr, M, K, N)
    if path is None:
        bqd.nvfp4_gemv(*args)
    else:
        bqd.nvfp4_gemv_path(*args, path)
    return out.get().reshape(N, M)


def check(w, rows=None, what=""):
    y = run(w)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], w["M"], w["K"], rows=rows)
    got = y if rows is None else y[:, rows]
    assert_within(got, ref, a, what)
    return y


def test_tiny_workload():
    check(syn.tiny_nvfp4(seed=0), what="256x512 N=1")


def test_worked_example(golden):
    g = golden("nvfp4_worked_example.txt")
    h = lambda v: [int(t, 16) for t in v]
    w = {"M": 2, "K": 32, "ts": float(g["ts"][0][0]),
         "codes": np.array([h(g["codes_row0"][0]), h(g["codes_row1"][0])], dtype=np.uint8),
         "scales": np.array([h(g["scales_row0"][0]), h(g["scales_row1"][0])], dtype=np.uint8),
         "x": np.array([h(g["x_col0"][0]), h(g["x_col1"][0])], dtype=np.uint16)}
    y = run(w)
    want = np.array([[float(v) for v in g["y_col0"][0]], [float(v) for v in g["y_col1"][0]]])
    a = np.array([[float(v) for v in g["a_col0"][0]], [float(v) for v in g["a_col1"][0]]])
    assert_within(y, want, a, "worked example")


@pytest.mark.parametrize("M,K,N", [
    (1, 16, 1), (1, 32, 1), (127, 48, 3), (129, 512, 5), (300, 4096, 1), (77, 4112, 2),
    (513, 1024, 8), (64, 2048, 16), (200, 8192, 9), (100, 12288, 16), (33, 16, 16), (1000, 96, 4),
])
def test_edge_shapes(M, K, N):
    check(syn.dense_nvfp4(M, K, N=N, seed=M * 7 + K + N), what=f"{M}x{K} N={N}")


@pytest.mark.parametrize("M,K", syn.NVFP4_SHAPES)
def test_full_size_n1(M, K):
    check(syn.dense_nvfp4(M, K, N=1, seed=0), what=f"{M}x{K} N=1")


@pytest.mark.parametrize("M,K", syn.VERIFY_SHAPES)
@pytest.mark.parametrize("N", [4, 8])
def test_full_size_verify_sampled_rows(M, K, N):
    w = syn.dense_nvfp4(M, K, N=N, seed=0)
    rng = np.random.default_rng(M + N)
    rows = np.unique(np.concatenate([[0, 1, M - 2, M - 1], rng.choice(M, 512, replace=False)]))
    check(w, rows=rows, what=f"{M}x{K} N={N}")


def test_deterministic_and_path_equivalence():
    w = syn.dense_nvfp4(12288, 4096, N=1, seed=1)
    y1, y2 = run(w), run(w)
    y3 = run(w, path=bqd.BQD_PATH_CUDA_CORE)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert np.array_equal(y1.view(np.uint32), y3.view(np.uint32))


def test_one_hot_selects_dequantised_column_exactly():
    w = syn.dense_nvfp4(300, 1024, N=4, seed=5)
    x = np.zeros((4, 1024), dtype=np.uint16)
    for n, k in enumerate((0, 1, 511, 1023)):
        x[n, k] = 0x3F80
    w["x"] = x
    y = run(w)
    W = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], 300, 1024, dtype=np.float32)
    for n, k in enumerate((0, 1, 511, 1023)):
        assert np.array_equal(y[n], W[:, k])


def test_sign_flip_zero_codes_and_tensor_scale_are_exact():
    w = syn.dense_nvfp4(500, 2048, N=2, seed=6)
    y = run(w)
    neg = dict(w, codes=w["codes"] ^ 0x88)
    assert np.array_equal(run(neg), -y)
    zero = dict(w, codes=np.zeros_like(w["codes"]))
    assert np.all(run(zero) == 0)
    y1 = run(dict(w, ts=1.0))
    y2 = run(dict(w, ts=2.0))
    assert np.array_equal(y2, 2 * y1)


def test_empty_shapes():
    out = Guarded(8, fill=5.0)
    bqd.nvfp4_gemv(None, None, 1.0, None, out.ptr, 4, 0, 2)  # K == 0: y = 0
    assert np.all(out.get() == 0)
    bqd.nvfp4_gemv(None, None, 1.0, None, None, 0, 64, 1)  # M == 0: nothing
    torch.cuda.synchronize()
