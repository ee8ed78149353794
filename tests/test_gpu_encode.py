"""bf16 -> NVFP4 / Q8_0 encoders (nvfp4_encode, q8_0_encode) against the
oracle's encoders, bit for bit (every decision on fp32 values rounded to
nearest even on both sides), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.gpu_util import dev, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _bf16(v):
    return torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def gpu_nvfp4(wb, ts, M, K):
    codes = torch.full((M * K // 2,), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((M * K // 16,), 0xCD, dtype=torch.uint8, device="cuda")
    bqd.nvfp4_encode(dev(wb), ts, codes, scales, M, K)
    return codes.cpu().numpy().reshape(M, K // 2), scales.cpu().numpy().reshape(M, K // 16)


def gpu_q8(wb, M, K):
    q = torch.full((M * K,), 77, dtype=torch.int8, device="cuda")
    d = torch.full((M * K // 32,), 0x1234, dtype=torch.int16, device="cuda")
    bqd.q8_0_encode(dev(wb), q, d, M, K)
    return q.cpu().numpy().reshape(M, K), d.cpu().numpy().view(np.uint16).reshape(M, K // 32)


def _weights(M, K, seed, kind, top=40):
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((M, K)).astype(np.float32)
    if kind == "wide":  # blocks over many binades
        W *= (2.0 ** rng.integers(-40, top, size=(M, K // 16, 1))).repeat(16, 2).reshape(M, K).astype(np.float32)
    elif kind == "specials":  # zero blocks, signed zeros, tiny values, one huge block
        W[0, :64] = 0.0
        W[1, :16] = -0.0
        W[2, :16] = np.float32(1e-30)
        W[3, 5] = np.float32(3e38)
    return _bf16(W)


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (64, 256), (257, 1040), (4096, 4096), (1000, 12288)])
@pytest.mark.parametrize("kind", ["normal", "wide", "specials"])
def test_nvfp4_encode_matches_oracle(M, K, kind):
    if kind != "normal" and M < 4:
        pytest.skip("the special blocks need four rows")
    wb = _weights(M, K, M + K, kind)
    Wf = (wb.astype(np.uint32) << 16).view(np.float32)
    finite = np.abs(Wf[np.isfinite(Wf)])
    ts = np.float32(max(finite.max(), 1e-30) / (6 * 448))
    if not (2.0 ** -100 <= ts <= 2.0 ** 100):
        ts = np.float32(1.0)
    c, s = gpu_nvfp4(wb, float(ts), M, K)
    c_ref, s_ref = oracle.nvfp4_encode(wb, ts, M, K)
    assert np.array_equal(s, s_ref), f"scales {np.argwhere(s != s_ref)[:5].tolist()}"
    assert np.array_equal(c, c_ref), f"codes {np.argwhere(c != c_ref)[:5].tolist()}"


@pytest.mark.parametrize("ts", [2.0 ** -7, 0.01, 1.0, 37.5])
def test_nvfp4_encode_tensor_scales_and_round_trip(ts):
    M, K = 128, 2048
    wb = _weights(M, K, 11, "normal")
    c, s = gpu_nvfp4(wb, ts, M, K)
    c_ref, s_ref = oracle.nvfp4_encode(wb, np.float32(ts), M, K)
    assert np.array_equal(s, s_ref) and np.array_equal(c, c_ref)
    # weights that are an encoding (power-of-two ts, a code-7 element per block) come back unchanged
    w = syn.dense_nvfp4(M, K, N=1, seed=4, ts=2.0 ** -7)
    codes = w["codes"].copy()
    codes[:, ::8] = (codes[:, ::8] & 0xF0) | 0x07
    Wd = oracle.nvfp4_dequant(codes, w["scales"], np.float32(2.0 ** -7), M, K, dtype=np.float32)
    c2, s2 = gpu_nvfp4(_bf16(Wd), 2.0 ** -7, M, K)
    assert np.array_equal(s2, w["scales"]) and np.array_equal(c2, codes)


@pytest.mark.parametrize("M,K", [(1, 32), (5, 96), (64, 256), (1000, 4096), (4096, 12288)])
@pytest.mark.parametrize("kind", ["normal", "wide", "specials"])
def test_q8_0_encode_matches_oracle(M, K, kind):
    if kind != "normal" and M < 4:
        pytest.skip("the special blocks need four rows")
    # amax / 127 stays within fp16 (larger blocks are outside the contract);
    # the smallest blocks give subnormal and zero d
    wb = _weights(M, K, 3 * M + K, kind, top=8)
    if kind == "specials":  # amax above 65504 * 127 is outside the contract
        wb[3, 5] = _bf16(np.array([1e6], dtype=np.float32))[0]
    q, d = gpu_q8(wb, M, K)
    q_ref, d_ref = oracle.q8_0_encode(wb, M, K)
    assert np.array_equal(d, d_ref), f"d {np.argwhere(d != d_ref)[:5].tolist()}"
    assert np.array_equal(q, q_ref), f"q {np.argwhere(q != q_ref)[:5].tolist()}"


def test_encoded_weights_feed_the_gemv():
    # encode on the GPU, then the GEMV on those codes equals the oracle GEMV
    M, K = 2048, 4096
    wb = _weights(M, K, 21, "normal")
    ts = np.float32(np.abs((wb.astype(np.uint32) << 16).view(np.float32)).max() / (6 * 448))
    codes = torch.empty(M * K // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(M * K // 16, dtype=torch.uint8, device="cuda")
    bqd.nvfp4_encode(dev(wb), float(ts), codes, scales, M, K)
    x = syn.bf16_normal((1, K), np.random.default_rng(5))
    y = torch.empty(M, dtype=torch.float32, device="cuda")
    bqd.nvfp4_gemv(codes, scales, float(ts), dev(x), y, M, K, 1)
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    ref, a = oracle.nvfp4_gemv(c, s, ts, x, M, K)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref[0])
    assert np.all(err <= 1e-3 * a[0] + 1e-6)


def test_encoders_reject_bad_arguments():
    wb = dev(_weights(4, 64, 1, "normal"))
    codes = torch.empty(128, dtype=torch.uint8, device="cuda")
    scales = torch.empty(16, dtype=torch.uint8, device="cuda")
    for M, K, ts in ((4, 40, 1.0), (4, 64, 0.0), (4, 64, float("nan")), (4, 64, -1.0), (-1, 64, 1.0)):
        with pytest.raises(bqd.BqdError):
            bqd.nvfp4_encode(wb, ts, codes, scales, M, K)
    with pytest.raises(bqd.BqdError):  # misaligned codes
        bqd.nvfp4_encode(wb, 1.0, codes.data_ptr() + 1, scales, 4, 64)
    q = torch.empty(256, dtype=torch.int8, device="cuda")
    d = torch.empty(8, dtype=torch.int16, device="cuda")
    with pytest.raises(bqd.BqdError):  # K % 32 != 0
        bqd.q8_0_encode(wb, q, d, 4, 48)
    with pytest.raises(bqd.BqdError):  # odd d address
        bqd.q8_0_encode(wb, q, d.data_ptr() + 1, 4, 64)
    bqd.nvfp4_encode(wb, 1.0, codes, scales, 0, 64)  # M == 0: nothing to do
