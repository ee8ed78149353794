"""Pins of the oracle's Q4_1 dequantisation and GEMV (a GGUF format the
"robertbfuentes7-cloud/bw24" README's GGUF bullet names beside Q4_0; its
block is GGUF's, split into a code plane and a (d, m) plane): a hand-worked
example, the nibble order and every code, exact-rational brute force,
library matmul and invariants."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins


def _build_worked(g):
    M, K = int(g["M"][0][0]), int(g["K"][0][0])
    codes = np.zeros((M, K // 2), dtype=np.uint8)
    for b, v in enumerate(g["row0_block_default"][0]):
        codes[0, 16 * b:16 * (b + 1)] = int(v, 16)
    for item in g["row0_bytes"][0]:
        k, v = item.split(":")
        codes[0, int(k)] = int(v, 16)
    codes[1, :] = int(g["row1_default"][0][0], 16)
    dm = np.array([[int(v, 16) for v in g["dm_row0"][0]], [int(v, 16) for v in g["dm_row1"][0]]],
                  dtype=np.uint16).reshape(M, K // 32, 2)
    x = np.full((1, K), int(g["x_default"][0][0], 16), dtype=np.uint16)
    for item in g["x_special"][0]:
        k, v = item.split(":")
        x[0, int(k)] = int(v, 16)
    return M, K, codes, dm, x


def test_q4_1_worked_example(golden):
    g = golden("q4_1_worked_example.txt")
    M, K, codes, dm, x = _build_worked(g)
    y, a = oracle.q4_1_gemv(codes, dm, x, M, K)
    assert y[0].tolist() == [float(v) for v in g["y"][0]]
    assert a[0].tolist() == [float(v) for v in g["a"][0]]


def test_q4_1_nibble_order_and_every_code():
    # byte j of a block holds element j (low nibble) and element j + 16 (high
    # nibble); every code q decodes to d * q + m, for several (d, m)
    # (subnormal, negative, the largest finite)
    K = 64
    codes = np.zeros((1, K // 2), dtype=np.uint8)
    for j in range(16):
        codes[0, j] = j | ((15 - j) << 4)
        codes[0, 16 + j] = ((j + 5) % 16) | (j << 4)
    want_q = ([j for j in range(16)] + [15 - j for j in range(16)] +
              [(j + 5) % 16 for j in range(16)] + [j for j in range(16)])
    for dv, mv in ((0x3C00, 0x0000), (0x0001, 0xBC00), (0xB800, 0x4500), (0x7BFF, 0xFBFF), (0x2E66, 0x0001)):
        dm = np.array([[[dv, mv], [dv, mv]]], dtype=np.uint16)
        w = oracle.q4_1_dequant(codes, dm, 1, K)
        d, m = (float(np.array([v], dtype=np.uint16).view(np.float16)[0]) for v in (dv, mv))
        assert w[0].tolist() == [q * d + m for q in want_q]
        w32 = oracle.q4_1_dequant(codes, dm, 1, K, dtype=np.float32)
        assert np.array_equal(w32, w.astype(np.float32))


@pytest.mark.parametrize("K", [32, 64, 96])
def test_q4_1_gemv_exact_rational_bruteforce(K):
    rng = np.random.default_rng(500 + K)
    M, N = 4, 3
    w = syn.q4_1_weight(M, K, rng, rng)
    x = syn.bf16_normal((N, K), rng)
    y, a = oracle.q4_1_gemv(w["codes"], w["dm"], x, M, K)
    q = pins.q4_0_codes_unpacked(w["codes"])
    f = pins.fp16_lib(w["dm"])
    xv = pins.bf16_lib(x)
    for n in range(N):
        for m in range(M):
            terms = [(Fraction(int(q[m, k])) * Fraction(f[m, k // 32, 0]) + Fraction(f[m, k // 32, 1]))
                     * Fraction(xv[n, k]) for k in range(K)]
            exact, abs_exact = sum(terms), sum(abs(t) for t in terms)
            assert abs(Fraction(y[n, m]) - exact) <= Fraction(2) ** -50 * abs_exact
            assert abs(Fraction(a[n, m]) - abs_exact) <= Fraction(2) ** -50 * abs_exact


def test_q4_1_dequant_and_gemv_match_library():
    w = syn.dense_q4_1(80, 384, N=2, seed=6)
    W = pins.q4_1_weight_lib(w["codes"], w["dm"])
    assert np.array_equal(oracle.q4_1_dequant(w["codes"], w["dm"], 80, 384), W)
    X = pins.bf16_lib(w["x"])
    y, a = oracle.q4_1_gemv(w["codes"], w["dm"], w["x"], 80, 384)
    assert np.all(np.abs(y - X @ W.T) <= 1e-13 * a)


def test_q4_1_invariants():
    M, K = 40, 256
    w = syn.dense_q4_1(M, K, N=1, seed=9)
    c, dm, x = w["codes"], w["dm"], w["x"]
    # d = 0: every weight is its block's m, y = sum over blocks of m * (sum of the block's x)
    dm0 = dm.copy()
    dm0[..., 0] = 0
    y0, _ = oracle.q4_1_gemv(c, dm0, x, M, K)
    xs = pins.bf16_lib(x)[0].reshape(K // 32, 32).sum(axis=1)
    assert np.allclose(y0[0], pins.fp16_lib(dm0[..., 1]) @ xs, rtol=1e-12, atol=1e-12)
    # m = 0: Q4_1 is Q4_0 with the codes shifted by 8 (q - 8 + 8), same d
    dmz = dm.copy()
    dmz[..., 1] = 0
    yz, _ = oracle.q4_1_gemv(c, dmz, x, M, K)
    yq, _ = oracle.q4_0_gemv(c, np.ascontiguousarray(dmz[..., 0]), x, M, K)
    d = pins.fp16_lib(dmz[..., 0])
    assert np.allclose(yz[0] - yq[0], 8 * (d @ xs), rtol=1e-12, atol=1e-12)
    # a one-hot activation picks the dequantised column
    oh = np.zeros((1, K), dtype=np.uint16)
    oh[0, 77] = 0x3F80
    yc, _ = oracle.q4_1_gemv(c, dm, oh, M, K)
    assert np.array_equal(yc[0], oracle.q4_1_dequant(c, dm, M, K)[:, 77])
