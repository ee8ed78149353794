"""Pins of the oracle's decode-path epilogues (residual add, SiLU * up)
against library routines and closed forms, on the CPU."""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins


def _weights(fmt, M, K, seed):
    if fmt == "nvfp4":
        w = syn.dense_nvfp4(M, K, N=1, seed=seed)
        return w, (w["codes"], w["scales"], w["ts"]), pins.nvfp4_weight_lib(w["codes"], w["scales"], w["ts"])
    w = syn.dense_q8_0(M, K, N=1, seed=seed)
    return w, (w["q"], w["d"]), pins.q8_0_weight_lib(w["q"], w["d"])


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
def test_silu_mul_matches_library_expit(fmt):
    I, K = 48, 256
    w, wt, W = _weights(fmt, 2 * I, K, seed=3)
    h, g, u, ag, au = oracle.gemv_silu_mul(fmt, wt, w["x"], I, K)
    X = pins.bf16_lib(w["x"])
    g_np, u_np = X @ W[:I].T, X @ W[I:].T
    assert np.allclose(g, g_np, rtol=1e-12, atol=1e-12) and np.allclose(u, u_np, rtol=1e-12, atol=1e-12)
    assert np.allclose(h, g_np * expit(g_np) * u_np, rtol=1e-12, atol=1e-15)
    assert np.allclose(ag, np.abs(X) @ np.abs(W[:I]).T, rtol=1e-12)


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
def test_silu_mul_one_hot_and_special_cases(fmt):
    I, K = 16, 64
    w, wt, W = _weights(fmt, 2 * I, K, seed=5)
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, 37] = 0x3F80  # 1.0
    h, g, u, _, _ = oracle.gemv_silu_mul(fmt, wt, x, I, K)
    assert np.array_equal(g[0], W[:I, 37]) and np.array_equal(u[0], W[I:, 37])
    assert np.allclose(h[0], W[:I, 37] * expit(W[:I, 37]) * W[I:, 37], rtol=1e-15)
    # x = 0: g = u = 0, SiLU(0) = 0
    h0, *_ = oracle.gemv_silu_mul(fmt, wt, np.zeros((1, K), dtype=np.uint16), I, K)
    assert np.all(h0 == 0)
    # a planted transposition (gate and up swapped) is seen
    hs = oracle.silu(u) * g
    assert not np.allclose(hs, h)


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
def test_gemv_add_reduces_to_gemv_and_to_the_residual(fmt):
    M, K = 40, 128
    w, wt, W = _weights(fmt, M, K, seed=7)
    r = np.random.default_rng(1).standard_normal((1, M)).astype(np.float32)
    y, a = oracle.gemv_add(fmt, wt, w["x"], r, M, K)
    y0, a0 = (oracle.nvfp4_gemv(*wt, w["x"], M, K) if fmt == "nvfp4" else oracle.q8_0_gemv(*wt, w["x"], M, K))
    assert np.array_equal(a, a0)
    assert np.allclose(y - r.astype(np.float64), pins.bf16_lib(w["x"]) @ W.T, rtol=1e-12, atol=1e-12)
    # zero weights leave exactly the residual; a zero residual leaves the GEMV
    z = ((np.zeros_like(wt[0]), wt[1], wt[2]) if fmt == "nvfp4" else (np.zeros_like(wt[0]), wt[1]))
    yz, _ = oracle.gemv_add(fmt, z, w["x"], r, M, K)
    assert np.array_equal(yz, r.astype(np.float64))
    y00, _ = oracle.gemv_add(fmt, wt, w["x"], np.zeros_like(r), M, K)
    assert np.array_equal(y00, y0)
    rows = np.array([0, 7, 39])
    yr, _ = oracle.gemv_add(fmt, wt, w["x"], r, M, K, rows=rows)
    assert np.array_equal(yr, y[:, rows])
