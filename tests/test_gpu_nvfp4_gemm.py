"""NVFP4 prefill GEMM (nvfp4_gemm: Y[T][M], many tokens, tcgen05 tensor
cores) against the fp64 oracle through the C ABI. Tolerance as for the
GEMVs: |y - y_ref| <= 1e-3 * sum|w x| + 1e-6; a one-hot token gives the
dequantised column bit for bit (one exact product)."""
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


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert bqd.bqd_device_error() == 0, "a wait ran out"


def run(w, x, M, K):
    T = x.shape[0]
    out = Guarded(T * M)
    bqd.nvfp4_gemm(dev(w["codes"]), dev(w["scales"]), w["ts"], dev(x), out.ptr, M, K, T)
    return out.get().reshape(T, M)


@pytest.mark.parametrize("M,K,T", [
    (1, 64, 1), (128, 64, 256), (256, 512, 300), (200, 1024, 17), (129, 192, 513), (384, 4096, 40),
    (70, 12288, 3),
])
def test_matches_oracle(M, K, T):
    w = syn.dense_nvfp4(M, K, N=T, seed=M + K + T)
    y = run(w, w["x"], M, K)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    assert_within(y, ref, a, f"{M}x{K} T={T}")


def test_layer_shape_sampled_rows():
    M, K, T = 12288, 4096, 512
    w = syn.dense_nvfp4(M, K, N=T, seed=7)
    y = run(w, w["x"], M, K)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], np.random.default_rng(3).choice(M, 60, replace=False)]))
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K, rows=rows)
    assert_within(y[:, rows], ref, a, "12288x4096 T=512")
    assert np.array_equal(y.view(np.uint32), run(w, w["x"], M, K).view(np.uint32))  # deterministic


def test_one_hot_tokens_give_the_dequantised_columns():
    M, K, T = 300, 1024, 260
    w = syn.dense_nvfp4(M, K, N=1, seed=11)
    ks = np.random.default_rng(4).integers(0, K, size=T)
    x = np.zeros((T, K), dtype=np.uint16)
    x[np.arange(T), ks] = 0x3F80
    y = run(w, x, M, K)
    W = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], M, K, dtype=np.float32)
    assert np.array_equal(y, W[:, ks].T)


def test_edge_cases_and_rejections():
    w = syn.dense_nvfp4(64, 128, N=4, seed=1)
    out = Guarded(8, fill=5.0)
    bqd.nvfp4_gemm(None, None, 1.0, None, out.ptr, 4, 0, 2)  # K == 0: zeros
    assert np.all(out.get() == 0)
    bqd.nvfp4_gemm(None, None, 1.0, None, None, 0, 128, 4)  # M == 0: nothing
    bqd.nvfp4_gemm(None, None, 1.0, None, None, 64, 128, 0)  # T == 0: nothing
    with pytest.raises(bqd.BqdError):  # K % 64 != 0
        bqd.nvfp4_gemm(dev(w["codes"]), dev(w["scales"]), 1.0, dev(w["x"]), Guarded(256).ptr, 64, 96, 4)
    with pytest.raises(bqd.BqdError):  # misaligned x
        bqd.nvfp4_gemm(dev(w["codes"]), dev(w["scales"]), 1.0, dev(w["x"]).data_ptr() + 2, Guarded(256).ptr, 64,
                       128, 4)
    torch.cuda.synchronize()
