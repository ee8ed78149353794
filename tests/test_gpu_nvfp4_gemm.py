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


# ---------------------------------------------------------------- grouped (per-expert) form
def _grouped_case(E, M, K, counts, seed):
    rng = np.random.default_rng(seed)
    ws = [syn.dense_nvfp4(M, K, N=1, seed=seed + e) for e in range(E)]
    codes = np.stack([w["codes"] for w in ws])
    scales = np.stack([w["scales"] for w in ws])
    ts = np.array([0.01 * (1 + e / 7) for e in range(E)], dtype=np.float32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    P = int(offsets[-1])
    x = syn.bf16_normal((P, K), rng)
    return codes, scales, ts, offsets, x, P


def run_grouped(codes, scales, ts, offsets, x, E, M, K, P):
    out = Guarded(P * M)
    bqd.nvfp4_gemm_grouped(dev(codes), dev(scales), dev(ts), dev(x), dev(offsets), out.ptr, E, M, K, P)
    return out.get().reshape(P, M)


# mean tokens per expert 14, 30, 66 and above 100: token tiles of 32, 64,
# 128 and 128, experts of one or several tiles each
@pytest.mark.parametrize("E,M,K,counts", [
    (8, 384, 1024, [0, 1, 15, 16, 17, 40, 3, 20]),
    (8, 384, 1024, [0, 1, 31, 32, 33, 100, 3, 40]),
    (8, 384, 1024, [0, 1, 63, 64, 65, 200, 3, 130]),
    (3, 256, 64, [17, 0, 300]),
    (1, 100, 512, [129]),
])
def test_grouped_matches_oracle_per_expert(E, M, K, counts):
    codes, scales, ts, offsets, x, P = _grouped_case(E, M, K, counts, seed=E * 10 + K)
    y = run_grouped(codes, scales, ts, offsets, x, E, M, K, P)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if a == b:
            continue
        ref, tol = oracle.nvfp4_gemv(codes[e], scales[e], ts[e], x[a:b], M, K)
        assert_within(y[a:b], ref, tol, f"expert {e}")


def test_grouped_moe_gate_up_shape_sampled():
    # the MoE layer's gate_up (2I = 1024 rows, H = 2048) over 32 experts and
    # 2048 routed pairs of uneven sizes, sampled rows of every expert
    E, M, K = 32, 1024, 2048
    counts = np.random.default_rng(5).multinomial(2048, np.ones(E) / E)
    codes, scales, ts, offsets, x, P = _grouped_case(E, M, K, counts, seed=3)
    y = run_grouped(codes, scales, ts, offsets, x, E, M, K, P)
    rows = np.array([0, 1, 255, 256, 511, 777, 1023])
    for e in range(0, E, 5):
        a, b = offsets[e], offsets[e + 1]
        ref, tol = oracle.nvfp4_gemv(codes[e], scales[e], ts[e], x[a:b], M, K, rows=rows)
        assert_within(y[a:b][:, rows], ref, tol, f"expert {e}")
    y2 = run_grouped(codes, scales, ts, offsets, x, E, M, K, P)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_grouped_rejections():
    codes, scales, ts, offsets, x, P = _grouped_case(2, 128, 128, [3, 4], seed=1)
    with pytest.raises(bqd.BqdError):  # K % 64 != 0
        run_grouped(codes, scales, ts, offsets, x, 2, 128, 96, P)
    with pytest.raises(bqd.BqdError):  # E = 0
        bqd.nvfp4_gemm_grouped(dev(codes), dev(scales), dev(ts), dev(x), dev(offsets), Guarded(P * 128).ptr, 0, 128,
                               128, P)
