"""Dequantisation on the GPU is bit-exact against the oracle, over every
(E2M1 code, E4M3 scale) pair and every (int8, fp16 scale) class."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.gpu_util import Guarded, dev, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _nvfp4_all_pairs():
    # row m uses scale byte m for all of its blocks; each row holds all 16 codes
    M, K = 256, 32
    codes = np.tile(np.array([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE], dtype=np.uint8), (M, 2))
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], K // 16, axis=1)
    return codes, scales, M, K


@pytest.mark.parametrize("ts", [1.0, 0.01, -3.5])
def test_nvfp4_dequant_every_code_and_scale(ts):
    codes, scales, M, K = _nvfp4_all_pairs()
    out = Guarded(M * K)
    bqd.nvfp4_dequant(dev(codes), dev(scales), ts, out.ptr, M, K)
    got = out.get().reshape(M, K)
    ref = oracle.nvfp4_dequant(codes, scales, np.float32(ts), M, K, dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))  # bit-exact, signed zeros too


@pytest.mark.parametrize("M,K", [(1, 16), (129, 48), (256, 512), (64, 4096)])
def test_nvfp4_dequant_random(M, K):
    w = syn.dense_nvfp4(M, K, seed=M + K)
    out = Guarded(M * K)
    bqd.nvfp4_dequant(dev(w["codes"]), dev(w["scales"]), w["ts"], out.ptr, M, K)
    ref = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], M, K, dtype=np.float32)
    assert np.array_equal(out.get().reshape(M, K).view(np.uint32), ref.view(np.uint32))


def test_q8_0_dequant_every_int8_and_scale_class():
    M, K = 64, 256
    q = np.tile(np.arange(-128, 128, dtype=np.int16).astype(np.int8), (M, 1))
    rng = np.random.default_rng(0)
    d = rng.integers(0, 0x7C00, size=(M, K // 32)).astype(np.uint16)  # finite fp16 incl. subnormals
    d[0, :] = 0x0001
    d[1, :] = 0x8001
    d[2, :] = 0x7BFF
    d[3, :] = 0xFBFF
    d[4, :] = 0x0000
    d[5:32] |= 0x8000
    out = Guarded(M * K)
    bqd.q8_0_dequant(dev(q), dev(d), out.ptr, M, K)
    ref = oracle.q8_0_dequant(q, d, M, K, dtype=np.float32)
    assert np.array_equal(out.get().reshape(M, K).view(np.uint32), ref.view(np.uint32))


def test_q8_0_dequant_random_ragged():
    w = syn.dense_q8_0(333, 96, seed=3)
    out = Guarded(333 * 96)
    bqd.q8_0_dequant(dev(w["q"]), dev(w["d"]), out.ptr, 333, 96)
    ref = oracle.q8_0_dequant(w["q"], w["d"], 333, 96, dtype=np.float32)
    assert np.array_equal(out.get().reshape(333, 96).view(np.uint32), ref.view(np.uint32))
