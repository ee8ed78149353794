"""Pins of the oracle's dequantisation and GEMV: hand-worked examples,
exact-rational brute force, library matmul, invariants."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins


def _hexbytes(vals):
    return [int(v, 16) for v in vals]


def test_nvfp4_worked_example(golden):
    g = golden("nvfp4_worked_example.txt")
    M, K, ts = int(g["M"][0][0]), int(g["K"][0][0]), float(g["ts"][0][0])
    codes = np.array([_hexbytes(g["codes_row0"][0]), _hexbytes(g["codes_row1"][0])], dtype=np.uint8)
    scales = np.array([_hexbytes(g["scales_row0"][0]), _hexbytes(g["scales_row1"][0])], dtype=np.uint8)
    x = np.array([_hexbytes(g["x_col0"][0]), _hexbytes(g["x_col1"][0])], dtype=np.uint16)
    y, a = oracle.nvfp4_gemv(codes, scales, ts, x, M, K)
    assert y[0].tolist() == [float(v) for v in g["y_col0"][0]]
    assert y[1].tolist() == [float(v) for v in g["y_col1"][0]]
    assert a[0].tolist() == [float(v) for v in g["a_col0"][0]]
    assert a[1].tolist() == [float(v) for v in g["a_col1"][0]]


def test_q8_0_worked_example(golden):
    g = golden("q8_0_worked_example.txt")
    M, K = int(g["M"][0][0]), int(g["K"][0][0])
    q = np.zeros((M, K), dtype=np.int8)
    for item in g["row0_q_nonzero"][0]:
        k, v = item.split(":")
        q[0, int(k)] = int(v)
    q[1, :] = int(g["row1_q_all"][0][0])
    d = np.array([_hexbytes(g["d_row0"][0]), _hexbytes(g["d_row1"][0])], dtype=np.uint16)
    x = np.full((1, K), int(g["x_default"][0][0], 16), dtype=np.uint16)
    for item in g["x_special"][0]:
        k, v = item.split(":")
        x[0, int(k)] = int(v, 16)
    y, a = oracle.q8_0_gemv(q, d, x, M, K)
    want_y = [float(v) for v in g["y"][0]]
    want_a = [float(v) for v in g["a"][0]]
    assert y[0, 0] == want_y[0] and a[0, 0] == want_a[0]
    assert abs(y[0, 1] - want_y[1]) <= 1e-15 * want_a[1]
    assert abs(a[0, 1] - want_a[1]) <= 1e-15 * want_a[1]


@pytest.mark.parametrize("K", [16, 32, 48])
def test_nvfp4_gemv_exact_rational_bruteforce(K):
    rng = np.random.default_rng(100 + K)
    M, N = 5, 2
    codes = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    scales = rng.choice(np.arange(0x01, 0x77, dtype=np.uint8), size=(M, K // 16))
    ts = 0.375
    x = syn.bf16_normal((N, K), rng)
    y, a = oracle.nvfp4_gemv(codes, scales, ts, x, M, K)
    tab = pins.e2m1_table()
    c = pins.nvfp4_codes_unpacked(codes)
    s = pins.e4m3_lib(scales)
    xv = pins.bf16_lib(x)
    for n in range(N):
        for m in range(M):
            exact = sum(Fraction(tab[c[m, k]]) * Fraction(s[m, k // 16]) * Fraction(ts) * Fraction(xv[n, k])
                        for k in range(K))
            abs_exact = sum(abs(Fraction(tab[c[m, k]]) * Fraction(s[m, k // 16]) * Fraction(ts) * Fraction(xv[n, k]))
                            for k in range(K))
            assert abs(Fraction(y[n, m]) - exact) <= Fraction(2) ** -50 * abs_exact
            assert abs(Fraction(a[n, m]) - abs_exact) <= Fraction(2) ** -50 * abs_exact


@pytest.mark.parametrize("K", [32, 64, 96])
def test_q8_0_gemv_exact_rational_bruteforce(K):
    rng = np.random.default_rng(200 + K)
    M, N = 4, 3
    w = syn.q8_0_weight(M, K, rng, rng)
    q, d = w["q"], w["d"]
    q[0, 0] = -128  # outside the generator's range, inside the format's
    x = syn.bf16_normal((N, K), rng)
    y, a = oracle.q8_0_gemv(q, d, x, M, K)
    dv = pins.fp16_lib(d)
    xv = pins.bf16_lib(x)
    for n in range(N):
        for m in range(M):
            terms = [Fraction(int(q[m, k])) * Fraction(dv[m, k // 32]) * Fraction(xv[n, k]) for k in range(K)]
            exact, abs_exact = sum(terms), sum(abs(t) for t in terms)
            assert abs(Fraction(y[n, m]) - exact) <= Fraction(2) ** -50 * abs_exact
            assert abs(Fraction(a[n, m]) - abs_exact) <= Fraction(2) ** -50 * abs_exact


def test_nvfp4_dequant_matches_library_decoders():
    w = syn.tiny_nvfp4(seed=3, M=64, K=256, ts=0.01)
    ref = pins.nvfp4_weight_lib(w["codes"], w["scales"], w["ts"])
    got = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], 64, 256)
    assert np.array_equal(got, ref)
    got32 = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], 64, 256, dtype=np.float32)
    assert np.array_equal(got32, ref.astype(np.float32))


def test_q8_0_dequant_matches_library_decoders():
    w = syn.dense_q8_0(48, 320, seed=4)
    ref = pins.q8_0_weight_lib(w["q"], w["d"])
    got = oracle.q8_0_dequant(w["q"], w["d"], 48, 320)
    assert np.array_equal(got, ref)
    got32 = oracle.q8_0_dequant(w["q"], w["d"], 48, 320, dtype=np.float32)
    assert np.array_equal(got32.astype(np.float64), ref)  # exact in fp32


def test_nvfp4_gemv_matches_library_matmul():
    w = syn.dense_nvfp4(96, 512, N=3, seed=5)
    W = pins.nvfp4_weight_lib(w["codes"], w["scales"], w["ts"])
    X = pins.bf16_lib(w["x"])
    ref = X @ W.T
    y, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], 96, 512)
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    assert np.allclose(a, np.abs(X)[:, None, :].__mul__(np.abs(W)[None]).sum(-1), rtol=1e-12)


def test_q8_0_gemv_matches_library_matmul():
    w = syn.dense_q8_0(80, 384, N=2, seed=6)
    W = pins.q8_0_weight_lib(w["q"], w["d"])
    X = pins.bf16_lib(w["x"])
    y, a = oracle.q8_0_gemv(w["q"], w["d"], w["x"], 80, 384)
    assert np.all(np.abs(y - X @ W.T) <= 1e-12 * a)


def test_gemv_rows_subset_matches_full():
    w = syn.dense_nvfp4(70, 256, N=2, seed=7)
    rows = np.array([69, 0, 33, 33, 5])
    y, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], 70, 256)
    ys, as_ = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], 70, 256, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(as_, a[:, rows])
    q = syn.dense_q8_0(70, 256, N=2, seed=7)
    y, a = oracle.q8_0_gemv(q["q"], q["d"], q["x"], 70, 256)
    ys, as_ = oracle.q8_0_gemv(q["q"], q["d"], q["x"], 70, 256, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(as_, a[:, rows])


# ---------------------------------------------------------------- invariants

def _one_hot_bf16(K, k):
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, k] = 0x3F80  # 1.0
    return x


def test_nvfp4_one_hot_selects_dequantised_column():
    w = syn.dense_nvfp4(40, 128, seed=8)
    W32 = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], 40, 128, dtype=np.float32)
    for k in (0, 1, 17, 127):
        y, _ = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], _one_hot_bf16(128, k), 40, 128)
        assert np.array_equal(y[0].astype(np.float32), W32[:, k])


def test_nvfp4_doubling_block_scale_doubles_block_contribution():
    w = syn.dense_nvfp4(16, 96, seed=9)
    M, K = 16, 96
    codes, scales = w["codes"], w["scales"].copy()
    e = (scales >> 3) & 15
    b = 3
    rows = np.where((e[:, b] >= 1) & (e[:, b] <= 13))[0]
    assert len(rows) > 0
    y0, a0 = oracle.nvfp4_gemv(codes, scales, w["ts"], w["x"], M, K)
    xb = np.zeros_like(w["x"])
    xb[:, 16 * b:16 * (b + 1)] = w["x"][:, 16 * b:16 * (b + 1)]
    contrib, _ = oracle.nvfp4_gemv(codes, scales, w["ts"], xb, M, K)
    s2 = scales.copy()
    s2[rows, b] = s2[rows, b] + (1 << 3)  # exponent field + 1
    y1, _ = oracle.nvfp4_gemv(codes, s2, w["ts"], w["x"], M, K)
    assert np.all(np.abs(y1[0, rows] - (y0[0, rows] + contrib[0, rows])) <= 1e-13 * a0[0, rows] * 2)
    others = np.setdiff1d(np.arange(M), rows)
    assert np.array_equal(y1[0, others], y0[0, others])


def test_nvfp4_sign_flip_negates_exactly():
    w = syn.dense_nvfp4(33, 160, N=2, seed=10)
    y0, _ = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], 33, 160)
    y1, _ = oracle.nvfp4_gemv(w["codes"] ^ 0x88, w["scales"], w["ts"], w["x"], 33, 160)
    assert np.array_equal(y1, -y0)


def test_nvfp4_zero_codes_and_tensor_scale():
    w = syn.dense_nvfp4(20, 64, seed=11)
    y, _ = oracle.nvfp4_gemv(np.zeros_like(w["codes"]), w["scales"], w["ts"], w["x"], 20, 64)
    assert np.all(y == 0)
    y1, _ = oracle.nvfp4_gemv(w["codes"], w["scales"], 1.0, w["x"], 20, 64)
    y2, _ = oracle.nvfp4_gemv(w["codes"], w["scales"], 2.0, w["x"], 20, 64)
    assert np.array_equal(y2, 2 * y1)


def test_nvfp4_block_permutation_invariance():
    w = syn.dense_nvfp4(24, 256, N=2, seed=12)
    M, K = 24, 256
    perm = np.random.default_rng(0).permutation(K // 16)
    c = w["codes"].reshape(M, K // 16, 8)[:, perm].reshape(M, K // 2)
    s = w["scales"][:, perm]
    x = w["x"].reshape(2, K // 16, 16)[:, perm].reshape(2, K)
    y0, a0 = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    y1, _ = oracle.nvfp4_gemv(c, s, w["ts"], x, M, K)
    assert np.all(np.abs(y1 - y0) <= 1e-13 * a0)


def test_q8_0_invariants():
    w = syn.dense_q8_0(30, 128, N=1, seed=13)
    M, K = 30, 128
    W = oracle.q8_0_dequant(w["q"], w["d"], M, K, dtype=np.float32)
    y, _ = oracle.q8_0_gemv(w["q"], w["d"], _one_hot_bf16(K, 77), M, K)
    assert np.array_equal(y[0].astype(np.float32), W[:, 77])
    yn, _ = oracle.q8_0_gemv(-w["q"], w["d"], w["x"], M, K)
    y0, _ = oracle.q8_0_gemv(w["q"], w["d"], w["x"], M, K)
    assert np.array_equal(yn, -y0)
    d2 = w["d"].copy()
    d2[:, 1] = d2[:, 1] ^ 0x8000  # negate block 1's scale
    xb = np.zeros_like(w["x"])
    xb[:, 32:64] = w["x"][:, 32:64]
    blk, _ = oracle.q8_0_gemv(w["q"], w["d"], xb, M, K)
    y2, a2 = oracle.q8_0_gemv(w["q"], d2, w["x"], M, K)
    assert np.all(np.abs(y2 - (y0 - 2 * blk)) <= 1e-13 * a2)
