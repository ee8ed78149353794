"""Block-scaled MMA with split activations: how many NVFP4 planes of x meet
the tolerance? (CPU study, no GPU.)

A `kind::mxf4nvf4` tensor-core MMA multiplies NVFP4 by NVFP4, so the bf16
activations would have to be written as a sum of P NVFP4 "residual planes",
x ~ sum_p ts_p * s_pb * q_p (q_p E2M1, s_pb an E4M3 scale per 16 elements,
ts_p an fp32 scale per token and plane), each plane multiplied exactly by
the NVFP4 weights and the partial results added in fp32. The weights and
every plane are exact values, so the whole error of that path is the
representation error of x after P planes. This study measures it against
the oracle on the verify workload and pins the smallest P that meets the
method's tolerance |y - y_ref| <= 1e-3 * sum|w x| + 1e-6.

Splitting rule (the usual two-level NVFP4 quantisation, applied to the
residual): ts_p = amax(residual of the token) / (6 * 448); per block,
s = E4M3(amax(block) / (6 * ts_p)) (round to nearest even); q = the E2M1
value nearest to residual / (s * ts_p) (ties to the even code), |q| <= 6.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
MIDPOINTS = (E2M1_VALUES[1:] + E2M1_VALUES[:-1]) / 2


def round_e2m1(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 value, ties to the even code, saturating at +-6."""
    a = np.minimum(np.abs(v), 6.0)
    i = np.searchsorted(MIDPOINTS, a, side="left")  # index of the lower candidate at a tie
    tie = (i < len(MIDPOINTS)) & (a == MIDPOINTS[np.minimum(i, len(MIDPOINTS) - 1)])
    i = np.where(tie & (i % 2 == 1), i + 1, i)
    return np.sign(v) * E2M1_VALUES[i]


def round_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 (FN) value (torch's float8 cast, round to nearest even)."""
    return torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def split_planes(x: np.ndarray, P: int, pow2_ts: bool = False) -> list:
    """P residual NVFP4 planes of x [N][K] (K % 16 == 0), each an exact fp64
    array. pow2_ts: each plane's tensor scale is rounded up to a power of
    two (then every plane value and residual is exact in fp32 as well)."""
    N, K = x.shape
    r = x.copy()
    planes = []
    for _ in range(P):
        amax_tok = np.abs(r).max(axis=1, keepdims=True)
        ts = (amax_tok / (6.0 * 448.0)).astype(np.float32).astype(np.float64)
        if pow2_ts:
            with np.errstate(divide="ignore"):
                ts = np.where(ts > 0, 2.0 ** np.ceil(np.log2(np.where(ts > 0, ts, 1.0))), 0.0)
        rb = r.reshape(N, K // 16, 16)
        amax_b = np.abs(rb).max(axis=2, keepdims=True)
        with np.errstate(divide="ignore", invalid="ignore"):
            s = round_e4m3(np.where(ts[:, :, None] > 0, amax_b / (6.0 * ts[:, :, None]), 0.0))
            unit = s * ts[:, :, None]
            q = np.where(unit > 0, round_e2m1(rb / np.where(unit > 0, unit, 1.0)), 0.0)
        plane = (q * unit).reshape(N, K)
        planes.append(plane)
        r = r - plane
    return planes


def _workload():
    M, K, N = 4096, 4096, 8
    w = syn.dense_nvfp4(M, K, N=N, seed=0)
    rows = np.random.default_rng(7).choice(M, 512, replace=False)
    codes, scales = w["codes"][rows], w["scales"][rows]
    W = oracle.nvfp4_dequant(codes, scales, w["ts"], len(rows), K)
    y, a = oracle.nvfp4_gemv(codes, scales, w["ts"], w["x"], len(rows), K)
    x = pins.bf16_lib(w["x"]).astype(np.float64)
    return W, x, y, 1e-3 * a + 1e-6


def test_m2_planes_needed_for_the_tolerance():
    W, x, y, tol = _workload()
    ratios = []
    acc = np.zeros_like(x)
    for P, plane in enumerate(split_planes(x, 6), start=1):
        acc = acc + plane
        err = np.abs(acc @ W.T - y)
        ratios.append(float((err / tol).max()))
    # every extra plane shrinks the error several-fold
    for p in range(1, 5):
        assert ratios[p] < ratios[p - 1] / 2, ratios
    p_min = next(p for p, r in enumerate(ratios, start=1) if r <= 1.0)
    # finding: one plane (x quantised to NVFP4 once) is far outside the
    # tolerance; two planes are still outside on some outputs; three meet it
    assert ratios[0] > 10.0, ratios
    assert p_min == 3, ratios
    print("max err / tol for P = 1..6:", ["%.3g" % r for r in ratios])


def test_split_planes_sum_exactly_to_x_in_the_limit():
    # pins of the splitting itself: planes are exact NVFP4 values, the
    # residual shrinks by at least 4x per plane, and zeros stay zero
    x = pins.bf16_lib(syn.bf16_normal((3, 256), syn.streams(5, 1)[0])).astype(np.float64)
    x[1, :16] = 0.0
    planes = split_planes(x, 8)
    r_prev = np.abs(x).max()
    acc = np.zeros_like(x)
    for plane in planes:
        acc = acc + plane
        r = np.abs(x - acc).max()
        assert r <= r_prev / 4 + 1e-300
        r_prev = r
    assert np.all(planes[0][1, :16] == 0)
    assert np.abs(x - acc).max() <= 1e-4 * np.abs(x).max()
    assert set(np.unique(round_e2m1(np.array([0.25, 0.75, 2.5, 5.0, 7.0, -1.25])))) <= set(
        np.concatenate([E2M1_VALUES, -E2M1_VALUES]))
    assert list(round_e2m1(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_m2_power_of_two_plane_scales():
    # the device-side choice: power-of-two tensor scales per plane. Every
    # plane value and every residual is then exact in fp32, and three planes
    # still meet the tolerance
    W, x, y, tol = _workload()
    acc = np.zeros_like(x)
    ratios = []
    for plane in split_planes(x, 4, pow2_ts=True):
        acc = acc + plane
        ratios.append(float((np.abs(acc @ W.T - y) / tol).max()))
        assert np.array_equal(plane.astype(np.float32).astype(np.float64), plane)
        r = x - acc
        assert np.array_equal(r.astype(np.float32).astype(np.float64), r)
    assert ratios[2] <= 1.0, ratios
    print("pow2 ts, max err / tol for P = 1..4:", ["%.3g" % v for v in ratios])
