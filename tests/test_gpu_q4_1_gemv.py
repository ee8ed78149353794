"""Q4_1 GEMV (CUDA-core path) and dequantisation on the GPU against the fp64
oracle, through the C ABI (tolerance as for NVFP4: |y - y_ref| <= 1e-3 *
sum|w x| + 1e-6; dequantisation and one-hot columns bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.gpu_util import Guarded, assert_within, dev, need_gpu
from tests.test_oracle_q4_1 import _build_worked

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run(w, x=None, codes=None):
    M, K = w["M"], w["K"]
    xx = w["x"] if x is None else x
    N = xx.shape[0]
    out = Guarded(N * M)
    bqd.q4_1_gemv(dev(w["codes"] if codes is None else codes), dev(w["dm"]), dev(xx), out.ptr, M, K, N)
    return out.get().reshape(N, M)


def check(w, rows=None, what=""):
    y = run(w)
    ref, a = oracle.q4_1_gemv(w["codes"], w["dm"], w["x"], w["M"], w["K"], rows=rows)
    assert_within(y if rows is None else y[:, rows], ref, a, what)


def test_worked_example(golden):
    g = golden("q4_1_worked_example.txt")
    M, K, codes, dm, x = _build_worked(g)
    y = run({"M": M, "K": K, "codes": codes, "dm": dm, "x": x})
    assert_within(y[0], np.array([float(v) for v in g["y"][0]]), np.array([float(v) for v in g["a"][0]]), "worked")


def test_dequant_bit_exact():
    M, K = 300, 1024
    w = syn.dense_q4_1(M, K, seed=3)
    w["dm"][0, :3] = [[0x0001, 0x7BFF], [0x8000, 0xBC00], [0x7BFF, 0xFBFF]]  # subnormal d, -0, the largest
    out = torch.full((M * K,), float("nan"), dtype=torch.float32, device="cuda")
    bqd.q4_1_dequant(dev(w["codes"]), dev(w["dm"]), out, M, K)
    ref = oracle.q4_1_dequant(w["codes"], w["dm"], M, K, dtype=np.float32)
    assert np.array_equal(out.cpu().numpy().reshape(M, K).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("M,K,N", [
    (1, 32, 1), (127, 64, 3), (129, 512, 5), (300, 4096, 1), (513, 1024, 8), (64, 2048, 16),
    (200, 8192, 9), (90, 12288, 16), (1000, 96, 2), (77, 16384, 1),
])
def test_edge_shapes(M, K, N):
    check(syn.dense_q4_1(M, K, N=N, seed=M + K + N), what=f"{M}x{K} N={N}")


def test_full_size_n1_and_sampled_verify():
    check(syn.dense_q4_1(12288, 4096, N=1, seed=0), what="12288x4096")
    w = syn.dense_q4_1(4096, 12288, N=8, seed=1)
    rows = np.unique(np.concatenate([[0, 1, 4095], np.random.default_rng(5).choice(4096, 512, replace=False)]))
    check(w, rows=rows, what="4096x12288 N=8")


def test_one_hot_columns_and_determinism():
    M, K = 700, 4096
    w = syn.dense_q4_1(M, K, N=1, seed=13)
    W = oracle.q4_1_dequant(w["codes"], w["dm"], M, K, dtype=np.float32)
    for k in (0, 15, 16, 31, 32, 2048, 4095):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80
        assert np.array_equal(run(w, x=x)[0], W[:, k]), f"one-hot k={k}"
    assert np.array_equal(run(w).view(np.uint32), run(w).view(np.uint32))


def test_rejections():
    w = syn.dense_q4_1(16, 1024, seed=1)
    out = Guarded(16)
    with pytest.raises(bqd.BqdError):  # K % 32 != 0
        bqd.q4_1_gemv(dev(w["codes"]), dev(w["dm"]), dev(w["x"]), out.ptr, 16, 1000, 1)
    with pytest.raises(bqd.BqdError):  # N = 17
        bqd.q4_1_gemv(dev(w["codes"]), dev(w["dm"]), dev(np.repeat(w["x"], 17, 0)), out.ptr, 16, 1024, 17)
    e = Guarded(6, fill=5.0)
    bqd.q4_1_gemv(None, None, None, e.ptr, 3, 0, 2)  # K == 0: zeros
    assert np.all(e.get() == 0)
