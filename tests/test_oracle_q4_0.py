"""Pins of the oracle's Q4_0 dequantisation and GEMV (the format the
"avifenesh/memra" README's Decode kernels bullet names next to NVFP4 and
Q8_0; its block is GGUF's, split into a code plane and a scale plane): a
hand-worked example, the nibble order, exact-rational brute force, library
matmul and invariants."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins


def _build_worked(g):
    M, K = int(g["M"][0][0]), int(g["K"][0][0])
    codes = np.full((M, K // 2), int(g["row0_default"][0][0], 16), dtype=np.uint8)
    for item in g["row0_bytes"][0]:
        k, v = item.split(":")
        codes[0, int(k)] = int(v, 16)
    codes[1, :] = int(g["row1_default"][0][0], 16)
    d = np.array([[int(v, 16) for v in g["d_row0"][0]], [int(v, 16) for v in g["d_row1"][0]]], dtype=np.uint16)
    x = np.full((1, K), int(g["x_default"][0][0], 16), dtype=np.uint16)
    for item in g["x_special"][0]:
        k, v = item.split(":")
        x[0, int(k)] = int(v, 16)
    return M, K, codes, d, x


def test_q4_0_worked_example(golden):
    g = golden("q4_0_worked_example.txt")
    M, K, codes, d, x = _build_worked(g)
    y, a = oracle.q4_0_gemv(codes, d, x, M, K)
    assert y[0].tolist() == [float(v) for v in g["y"][0]]
    assert a[0].tolist() == [float(v) for v in g["a"][0]]


def test_q4_0_nibble_order_and_every_code():
    # byte j of a block holds element j (low nibble) and element j + 16 (high
    # nibble); every code q decodes to (q - 8) * d, for several d (subnormal,
    # negative, the largest finite)
    K = 64
    codes = np.zeros((1, K // 2), dtype=np.uint8)
    for j in range(16):
        codes[0, j] = j | ((15 - j) << 4)           # block 0
        codes[0, 16 + j] = ((j + 5) % 16) | (j << 4)  # block 1
    for dv in (0x3C00, 0x0001, 0xB800, 0x7BFF, 0x2E66):
        d = np.array([[dv, dv]], dtype=np.uint16)
        w = oracle.q4_0_dequant(codes, d, 1, K)
        s = float(np.array([dv], dtype=np.uint16).view(np.float16)[0])
        want = ([j - 8 for j in range(16)] + [(15 - j) - 8 for j in range(16)] +
                [(j + 5) % 16 - 8 for j in range(16)] + [j - 8 for j in range(16)])
        assert w[0].tolist() == [q * s for q in want]
        w32 = oracle.q4_0_dequant(codes, d, 1, K, dtype=np.float32)
        assert np.array_equal(w32.astype(np.float64), w)  # exact in fp32


@pytest.mark.parametrize("K", [32, 64, 96])
def test_q4_0_gemv_exact_rational_bruteforce(K):
    rng = np.random.default_rng(300 + K)
    M, N = 4, 3
    w = syn.q4_0_weight(M, K, rng, rng)
    x = syn.bf16_normal((N, K), rng)
    y, a = oracle.q4_0_gemv(w["codes"], w["d"], x, M, K)
    q = pins.q4_0_codes_unpacked(w["codes"])
    dv = pins.fp16_lib(w["d"])
    xv = pins.bf16_lib(x)
    for n in range(N):
        for m in range(M):
            terms = [Fraction(int(q[m, k]) - 8) * Fraction(dv[m, k // 32]) * Fraction(xv[n, k]) for k in range(K)]
            exact, abs_exact = sum(terms), sum(abs(t) for t in terms)
            assert abs(Fraction(y[n, m]) - exact) <= Fraction(2) ** -50 * abs_exact
            assert abs(Fraction(a[n, m]) - abs_exact) <= Fraction(2) ** -50 * abs_exact


def test_q4_0_dequant_and_gemv_match_library():
    w = syn.dense_q4_0(80, 384, N=2, seed=6)
    W = pins.q4_0_weight_lib(w["codes"], w["d"])
    assert np.array_equal(oracle.q4_0_dequant(w["codes"], w["d"], 80, 384), W)
    X = pins.bf16_lib(w["x"])
    y, a = oracle.q4_0_gemv(w["codes"], w["d"], w["x"], 80, 384)
    assert np.all(np.abs(y - X @ W.T) <= 1e-12 * a)
    rows = np.array([79, 0, 40, 40])
    ys, as_ = oracle.q4_0_gemv(w["codes"], w["d"], w["x"], 80, 384, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(as_, a[:, rows])


def test_q4_0_invariants():
    M, K = 24, 128
    w = syn.dense_q4_0(M, K, seed=9)
    codes, d, x = w["codes"], w["d"], w["x"]
    y, a = oracle.q4_0_gemv(codes, d, x, M, K)
    # one-hot x selects the dequantised column exactly
    W32 = oracle.q4_0_dequant(codes, d, M, K, dtype=np.float32)
    for k in (0, 15, 16, 31, 33, 127):
        e = np.zeros((1, K), dtype=np.uint16)
        e[0, k] = 0x3F80
        yk, _ = oracle.q4_0_gemv(codes, d, e, M, K)
        assert np.array_equal(yk[0].astype(np.float32), W32[:, k])
    # code 8 everywhere is zero
    z, _ = oracle.q4_0_gemv(np.full_like(codes, 0x88), d, x, M, K)
    assert np.all(z == 0)
    # q -> 16 - q (codes 1..15) negates every element, so y negates exactly
    lo, hi = codes & 0x0F, codes >> 4
    lo, hi = np.maximum(lo, 1), np.maximum(hi, 1)
    c1 = (lo | (hi << 4)).astype(np.uint8)
    c2 = ((16 - lo) | ((16 - hi) << 4)).astype(np.uint8)
    y1, _ = oracle.q4_0_gemv(c1, d, x, M, K)
    y2, _ = oracle.q4_0_gemv(c2, d, x, M, K)
    assert np.array_equal(y2, -y1)
    # doubling every d (fp16 exponent + 1, no overflow at these values) doubles y exactly
    y3, _ = oracle.q4_0_gemv(codes, (d + (1 << 10)).astype(np.uint16), x, M, K)
    assert np.array_equal(y3, 2 * y)
    # permuting whole 32-blocks of W and x together leaves y unchanged
    perm = np.array([3, 0, 2, 1])
    cp = codes.reshape(M, 4, 16)[:, perm].reshape(M, K // 2)
    dp = d[:, perm]
    xp = x.reshape(1, 4, 32)[:, perm].reshape(1, K)
    y4, _ = oracle.q4_0_gemv(cp, dp, xp, M, K)
    assert np.all(np.abs(y4 - y) <= 1e-13 * a)
