"""Pins of the oracle's FP8 block-128 dequantisation and GEMV (E4M3 weights,
"Vemloir/LumenLLM" README, Quantization bullet; one fp32 scale per 128 x 128
tile of the weight, "avifenesh/memra" README, Loaders bullet): a hand-worked
example across both tile boundaries, every code against torch's E4M3 decode,
the tile grid against a numpy-built weight, exact-rational brute force,
library matmul and invariants."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins


def _build_worked(g):
    M, K = int(g["M"][0][0]), int(g["K"][0][0])
    codes = np.zeros((M, K), dtype=np.uint8)
    for m, k, v in g["code"]:
        codes[int(m), int(k)] = int(v, 16)
    scales = np.array([float(v) for v in g["scales"][0]], dtype=np.float32).reshape(2, 2)
    x = np.full((1, K), int(g["x_default"][0][0], 16), dtype=np.uint16)
    for k, v in g["x"]:
        x[0, int(k)] = int(v, 16)
    return M, K, codes, scales, x


def test_fp8_b128_worked_example(golden):
    g = golden("fp8_b128_worked_example.txt")
    M, K, codes, scales, x = _build_worked(g)
    y, a = oracle.fp8_b128_gemv(codes, scales, x, M, K)
    want_y, want_a = np.zeros(M), np.zeros(M)
    for m, yv, av in g["y"]:
        want_y[int(m)], want_a[int(m)] = float(yv), float(av)
    assert y[0].tolist() == want_y.tolist()
    assert a[0].tolist() == want_a.tolist()


def test_fp8_b128_every_code_is_torchs_e4m3():
    # all 256 codes in one row, tile scale 1: torch's float8_e4m3fn decode
    # (both NaN codes, 0x7f and 0xff, decode to NaN)
    codes = np.arange(256, dtype=np.uint8)[None, :]
    w = oracle.fp8_b128_dequant(codes, np.ones((1, 2), dtype=np.float32), 1, 256)
    lib = pins.e4m3_lib(codes)
    assert np.array_equal(np.isnan(w), np.isnan(lib)) and np.isnan(w[0, 0x7F]) and np.isnan(w[0, 0xFF])
    ok = ~np.isnan(lib)
    assert np.array_equal(w[ok], lib[ok])
    assert w[0, 0x7E] == 448.0 and w[0, 0x01] == 2.0 ** -9 and w[0, 0x80] == 0.0


@pytest.mark.parametrize("M,K", [(1, 128), (129, 130), (300, 257), (128, 384)])
def test_fp8_b128_dequant_matches_library_tile_grid(M, K):
    # ragged M and K: the last tile row / column is partial
    w = syn.fp8_b128_weight(M, K, *syn.streams(M * 7 + K, 2))
    W = pins.fp8_b128_weight_lib(w["codes"], w["scales"])
    assert np.array_equal(oracle.fp8_b128_dequant(w["codes"], w["scales"], M, K), W)
    W32 = oracle.fp8_b128_dequant(w["codes"], w["scales"], M, K, dtype=np.float32)
    assert np.array_equal(W32, W.astype(np.float32))


@pytest.mark.parametrize("K", [16, 130, 256])
def test_fp8_b128_gemv_exact_rational_bruteforce(K):
    rng = np.random.default_rng(400 + K)
    M, N = 130, 2
    w = syn.fp8_b128_weight(M, K, rng, rng)
    x = syn.bf16_normal((N, K), rng)
    rows = np.array([0, 1, 127, 128, 129], dtype=np.int64)
    y, a = oracle.fp8_b128_gemv(w["codes"], w["scales"], x, M, K, rows=rows)
    cv, xv = pins.e4m3_lib(w["codes"]), pins.bf16_lib(x)
    for n in range(N):
        for i, m in enumerate(rows):
            terms = [Fraction(cv[m, k]) * Fraction(float(w["scales"][m // 128, k // 128])) * Fraction(xv[n, k])
                     for k in range(K)]
            exact, abs_exact = sum(terms), sum(abs(t) for t in terms)
            assert abs(Fraction(y[n, i]) - exact) <= Fraction(2) ** -50 * abs_exact
            assert abs(Fraction(a[n, i]) - abs_exact) <= Fraction(2) ** -50 * abs_exact


def test_fp8_b128_gemv_matches_library_matmul():
    M, K = 260, 640
    w = syn.dense_fp8_b128(M, K, N=3, seed=8)
    W = pins.fp8_b128_weight_lib(w["codes"], w["scales"])
    X = pins.bf16_lib(w["x"])
    y, a = oracle.fp8_b128_gemv(w["codes"], w["scales"], w["x"], M, K)
    assert np.all(np.abs(y - X @ W.T) <= 1e-13 * a)
    assert np.allclose(a, np.abs(X) @ np.abs(W).T, rtol=1e-13, atol=0)


def test_fp8_b128_invariants():
    M, K = 200, 384
    w = syn.dense_fp8_b128(M, K, N=1, seed=3)
    c, s, x = w["codes"], w["scales"], w["x"]
    y, _ = oracle.fp8_b128_gemv(c, s, x, M, K)
    # the sign bit negates exactly
    yn, _ = oracle.fp8_b128_gemv(c ^ np.uint8(0x80), s, x, M, K)
    assert np.array_equal(yn, -y)
    # one tile's scale doubled: only that tile's rows and k move, by exactly its part
    s2 = s.copy()
    s2[1, 2] *= 2
    y2, _ = oracle.fp8_b128_gemv(c, s2, x, M, K)
    xt = x.copy()
    xt[0, :256] = 0  # k outside tile column 2
    part, _ = oracle.fp8_b128_gemv(c, s, xt, M, K)
    assert np.array_equal(y2[0, :128], y[0, :128])
    assert np.allclose(y2[0, 128:], y[0, 128:] + part[0, 128:], rtol=0, atol=1e-12 * np.abs(part).max())
    # a one-hot activation picks the dequantised column
    oh = np.zeros((1, K), dtype=np.uint16)
    oh[0, 300] = 0x3F80
    yc, _ = oracle.fp8_b128_gemv(c, s, oh, M, K)
    assert np.array_equal(yc[0], oracle.fp8_b128_dequant(c, s, M, K)[:, 300])
    # zero codes give zero
    yz, _ = oracle.fp8_b128_gemv(np.zeros_like(c), s, x, M, K)
    assert not yz.any()
