"""Q8_0 GEMV on the GPU against the fp64 oracle (tolerance as for NVFP4)."""
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


def run(w, q=None):
    M, K = w["M"], w["K"]
    N = w["x"].shape[0]
    out = Guarded(N * M)
    bqd.q8_0_gemv(dev(w["q"] if q is None else q), dev(w["d"]), dev(w["x"]), out.ptr, M, K, N)
    return out.get().reshape(N, M)


def check(w, rows=None, what=""):
    y = run(w)
    ref, a = oracle.q8_0_gemv(w["q"], w["d"], w["x"], w["M"], w["K"], rows=rows)
    assert_within(y if rows is None else y[:, rows], ref, a, what)
    return y


def test_worked_example(golden):
    g = golden("q8_0_worked_example.txt")
    M, K = 2, 64
    q = np.zeros((M, K), dtype=np.int8)
    for item in g["row0_q_nonzero"][0]:
        k, v = item.split(":")
        q[0, int(k)] = int(v)
    q[1, :] = 1
    d = np.array([[int(v, 16) for v in g["d_row0"][0]], [int(v, 16) for v in g["d_row1"][0]]], dtype=np.uint16)
    x = np.full((1, K), 0x3F80, dtype=np.uint16)
    for item in g["x_special"][0]:
        k, v = item.split(":")
        x[0, int(k)] = int(v, 16)
    y = run({"M": M, "K": K, "q": q, "d": d, "x": x})
    assert_within(y[0], np.array([float(v) for v in g["y"][0]]), np.array([float(v) for v in g["a"][0]]), "worked")


@pytest.mark.parametrize("M,K,N", [
    (1, 32, 1), (127, 64, 3), (129, 512, 5), (300, 4096, 1), (513, 1024, 8), (64, 2048, 16),
    (200, 8192, 9), (90, 12288, 16), (1000, 96, 2),
])
def test_edge_shapes(M, K, N):
    check(syn.dense_q8_0(M, K, N=N, seed=M + K + N), what=f"{M}x{K} N={N}")


@pytest.mark.parametrize("M,K", syn.Q8_0_SHAPES[:2])
def test_full_size_n1(M, K):
    check(syn.dense_q8_0(M, K, N=1, seed=0), what=f"{M}x{K}")


def test_lm_head_sampled_rows():
    M, K = syn.Q8_0_SHAPES[2]
    w = syn.dense_q8_0(M, K, N=1, seed=0)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, 1, M - 2, M - 1], rng.choice(M, 4096, replace=False)]))
    check(w, rows=rows, what="LM head")


def test_extremes_and_exact_invariants():
    w = syn.dense_q8_0(256, 1024, N=2, seed=9)
    w["q"][:, :64] = -128
    w["q"][:, 64:128] = 127
    check(w, what="int8 extremes")
    y = run(w)
    q2 = w["q"].astype(np.int16)
    q2 = np.clip(-q2, -127, 127).astype(np.int8)  # negation, exact except -128 -> 127
    w2 = dict(w, q=q2)
    w2["q"][:, :64] = 0
    w3 = dict(w, q=w["q"].copy())
    w3["q"][:, :64] = 0
    assert np.array_equal(run(w2), -run(w3))
    x = np.zeros((2, 1024), dtype=np.uint16)
    x[0, 5] = 0x3F80
    x[1, 1000] = 0x3F80
    yo = run(dict(w, x=x))
    W = oracle.q8_0_dequant(w["q"], w["d"], 256, 1024, dtype=np.float32)
    assert np.array_equal(yo[0], W[:, 5]) and np.array_equal(yo[1], W[:, 1000])


def test_deterministic():
    w = syn.dense_q8_0(4096, 12288, N=1, seed=2)
    assert np.array_equal(run(w).view(np.uint32), run(w).view(np.uint32))


def test_empty_shapes():
    out = Guarded(6, fill=5.0)
    bqd.q8_0_gemv(None, None, None, out.ptr, 3, 0, 2)
    assert np.all(out.get() == 0)
    torch.cuda.synchronize()


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert bqd.bqd_device_error() == 0, "a pipeline wait ran out"


@pytest.mark.parametrize("M,K", syn.Q8_0_SHAPES[:2] + [(1, 256), (33, 768), (500, 16384), (4864, 4096), (70, 3072),
                                                      (9, 6144), (1, 1024)])
def test_stream_and_cuda_core_paths_match_oracle(M, K):
    w = syn.dense_q8_0(M, K, N=1, seed=M + K)
    ref, a = oracle.q8_0_gemv(w["q"], w["d"], w["x"], M, K)
    for path in (bqd.BQD_PATH_STREAM, bqd.BQD_PATH_CUDA_CORE) + ((bqd.BQD_PATH_DIRECT,) if K % 1024 == 0 else ()):
        out = Guarded(M)
        bqd.q8_0_gemv_path(dev(w["q"]), dev(w["d"]), dev(w["x"]), out.ptr, M, K, 1, path)
        assert_within(out.get()[None], ref, a, f"{M}x{K} path {path}")


# ---------------------------------------------------------------- N = 1 stream kernel, exact invariants
def _run_path(w, path, q=None, x=None):
    M, K = w["M"], w["K"]
    xx = w["x"] if x is None else x
    out = Guarded(M)
    bqd.q8_0_gemv_path(dev(w["q"] if q is None else q), dev(w["d"]), dev(xx), out.ptr, M, K, 1, path)
    return out.get()


@pytest.mark.parametrize("path", ["stream", "direct"])
def test_n1_extremes_and_exact_invariants(path):
    """Through the N = 1 paths: blocks of q = -128 and 127 within the
    tolerance; a one-hot x gives the dequantised column bit for bit;
    negating q negates y exactly."""
    M, K = 700, 4096
    P = bqd.BQD_PATH_STREAM if path == "stream" else bqd.BQD_PATH_DIRECT
    w = syn.dense_q8_0(M, K, N=1, seed=13)
    w["q"][:, :64] = -128
    w["q"][:, 64:128] = 127
    ref, a = oracle.q8_0_gemv(w["q"], w["d"], w["x"], M, K)
    assert_within(_run_path(w, P)[None], ref, a, "stream int8 extremes")
    W = oracle.q8_0_dequant(w["q"], w["d"], M, K, dtype=np.float32)
    for k in (0, 31, 32, 63, 64, 100, 2048, 4095):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80
        assert np.array_equal(_run_path(w, P, x=x), W[:, k]), f"one-hot k={k}"
    q3 = w["q"].copy()
    q3[:, :64] = 0  # -128 has no int8 negation
    q2 = (-q3.astype(np.int16)).astype(np.int8)
    assert np.array_equal(_run_path(w, P, q=q2), -_run_path(w, P, q=q3))
