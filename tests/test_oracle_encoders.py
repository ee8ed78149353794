"""Pins of the oracle's bf16 -> NVFP4 / Q8_0 encoders (CPU): library casts
(torch float8_e4m3fn, numpy float16 and rint), the E2M1 grid's midpoints,
saturation, signs, and exact round trips of weights that are themselves
encodings."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins


def _bf16(v):
    return torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([2.0 ** rng.uniform(-12, 8.8, 20000), oracle.e4m3_positive_grid(),
                        (oracle.e4m3_positive_grid()[1:] + oracle.e4m3_positive_grid()[:-1]) / 2])
    v = v[v <= 448].astype(np.float32)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), lib)
    assert np.all(oracle.e4m3_encode(np.array([449.0, 1e6, np.float32(3e38)], dtype=np.float32)) == 0x7E)


def test_e2m1_encode_grid_midpoints_saturation_and_sign():
    g = oracle.e2m1_positive_grid()
    assert np.array_equal(oracle.e2m1_encode(g.astype(np.float32)), np.arange(8, dtype=np.uint8))
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    # ties to the even code: 0.25 -> 0, 0.75 -> 1.0 (code 2), 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5 -> 4.0
    assert np.array_equal(oracle.e2m1_encode(mids), np.array([0, 2, 2, 4, 4, 6, 6], dtype=np.uint8))
    assert np.array_equal(oracle.e2m1_encode(np.array([6.5, 100.0, 3e38], dtype=np.float32)), [7, 7, 7])
    neg = oracle.e2m1_encode(-g.astype(np.float32))
    assert np.array_equal(neg, np.arange(8, dtype=np.uint8) | 8)  # -0.0 is code 8
    assert oracle.e2m1_encode(np.array([-0.1], dtype=np.float32))[0] == 8
    # nearest value: encode then decode never moves a value by more than half a grid step (below 6)
    v = np.random.default_rng(1).uniform(-6, 6, 5000).astype(np.float32)
    dec = np.array([oracle.e2m1(int(c)) for c in oracle.e2m1_encode(v)])
    step = np.array([0.5, 0.5, 0.5, 0.5, 1, 1, 2, 2])[np.minimum(7, oracle.e2m1_encode(np.abs(v)) & 7)]
    assert np.all(np.abs(dec - v) <= step / 2 + 1e-9)


def test_nvfp4_encode_round_trips_its_own_weights():
    # blocks whose largest code is 6.0 (code 7) encode back to the same codes and scales
    # (a power-of-two tensor scale keeps every weight exact in bf16)
    M, K, ts = 64, 256, np.float32(2.0 ** -7)
    w = syn.dense_nvfp4(M, K, N=1, seed=5, ts=float(ts))
    codes = w["codes"].copy()
    codes[:, ::8] = (codes[:, ::8] & 0xF0) | 0x07  # element 16b of every block is +6
    W = oracle.nvfp4_dequant(codes, w["scales"], ts, M, K, dtype=np.float32)
    wb = _bf16(W)
    assert np.array_equal(pins.bf16_lib(wb), W.astype(np.float64))
    c2, s2 = oracle.nvfp4_encode(wb, ts, M, K)
    assert np.array_equal(s2, w["scales"]) and np.array_equal(c2, codes)


def test_nvfp4_encode_error_and_zero_blocks():
    M, K = 32, 512
    rng = np.random.default_rng(7)
    Wf = rng.standard_normal((M, K)).astype(np.float32)
    ts = np.float32(np.abs(Wf).max() / (6 * 448))  # the tensor's largest block maps to E4M3's largest scale
    Wf[3, 16:32] = 0.0
    wb = _bf16(Wf)
    c, s = oracle.nvfp4_encode(wb, ts, M, K)
    assert np.all(s[3, 1] == 0) and np.all(c[3, 8:16] == 0)
    D = oracle.nvfp4_dequant(c, s, ts, M, K)
    Wb = pins.bf16_lib(wb)
    # every element within half the block's E2M1 grid step at its scale (+ the scale's own rounding)
    blk = np.abs(Wb).reshape(M, K // 16, 16).max(-1)
    err = np.abs(D - Wb).reshape(M, K // 16, 16).max(-1)
    assert np.all(err <= blk * (1.0 / 6 + 1.0 / 16) + 1e-30)


def test_q8_0_encode_matches_library_rounding_and_round_trips():
    M, K = 16, 256
    rng = np.random.default_rng(3)
    Wf = (rng.standard_normal((M, K)) * 0.05).astype(np.float32)
    Wf[2, :32] = 0
    wb = _bf16(Wf)
    q, d = oracle.q8_0_encode(wb, M, K)
    Wb = pins.bf16_lib(wb).astype(np.float32)
    amax = np.abs(Wb).reshape(M, K // 32, 32).max(-1)
    d_lib = (amax / np.float32(127)).astype(np.float16)
    assert np.array_equal(d, d_lib.view(np.uint16))
    dq = np.repeat(d_lib.astype(np.float32), 32, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        q_lib = np.where(dq == 0, 0, np.clip(np.rint(Wb / dq), -127, 127)).astype(np.int8)
    assert np.array_equal(q, q_lib) and np.all(q[2, :32] == 0)
    # a Q8_0 weight whose blocks reach +-127, with power-of-two scales (so
    # every weight is exact in bf16), re-encodes to itself
    qq = syn.dense_q8_0(M, K, N=1, seed=2)
    qq["q"][:, ::32] = 127
    qq["d"] = (2.0 ** -rng.integers(6, 14, size=qq["d"].shape)).astype(np.float16).view(np.uint16)
    W2 = oracle.q8_0_dequant(qq["q"], qq["d"], M, K, dtype=np.float32)
    w2 = _bf16(W2)
    assert np.array_equal(pins.bf16_lib(w2), W2.astype(np.float64))
    # amax / 127 = d exactly, so the encoder finds the same scale and codes
    q2, d2 = oracle.q8_0_encode(w2, M, K)
    assert np.array_equal(d2, qq["d"]) and np.array_equal(q2, qq["q"])
