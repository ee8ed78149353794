"""Tensor-core NVFP4 GEMV (BQD_PATH_MMA) against the fp64 oracle.

The tolerance is the method's, |y - y_ref| <= 1e-3 * sum|w x| + 1e-6 per
output; the exact invariants (one-hot columns, sign flips, power-of-two
tensor scales) are checked bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins
from tests.gpu_util import Guarded, assert_within, dev, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert bqd.bqd_device_error() == 0, "a pipeline wait ran out"


def run(w, path=bqd.BQD_PATH_MMA, N=None):
    M, K = w["M"], w["K"]
    N = N or w["x"].shape[0]
    out = Guarded(N * M)
    bqd.nvfp4_gemv_path(dev(w["codes"]), dev(w["scales"]), w["ts"], dev(w["x"]), out.ptr, M, K, N, path)
    return out.get().reshape(N, M)


def check(w, rows=None, what=""):
    y = run(w)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], w["M"], w["K"], rows=rows)
    assert_within(y if rows is None else y[:, rows], ref, a, what)
    return y


# Several 128-row tiles with a ragged last tile, one to many 256-k stages
# (so clusters of 1 to 8 CTAs), token counts from 1 to 16.
@pytest.mark.parametrize("M,K,N", [
    (1, 256, 1), (128, 256, 16), (129, 512, 2), (300, 768, 4), (257, 1024, 8), (640, 2304, 3),
    (1000, 4096, 16), (77, 8192, 5), (4096, 256, 2), (383, 3072, 7), (200, 16384, 9), (1, 12288, 16),
    (513, 1536, 11), (64, 2048, 13),
    # clusters of 2..6 CTAs over 2..4 tiles each (on a 152-SM part), one
    # accumulator per tile and a partial last cluster; and one CTA over 2
    # tiles with all of k (no cluster)
    (5979, 3072, 12), (9819, 2048, 3), (20000, 768, 4), (20000, 1024, 12), (20000, 512, 5), (30000, 256, 16),
])
def test_mma_matches_oracle(M, K, N):
    check(syn.dense_nvfp4(M, K, N=N, seed=3 * M + K + N), what=f"{M}x{K} N={N}")


@pytest.mark.parametrize("M,K", syn.VERIFY_SHAPES + [(4096, 12288)])
@pytest.mark.parametrize("N", [2, 4, 8, 16])
def test_mma_full_size_sampled_rows(M, K, N):
    w = syn.dense_nvfp4(M, K, N=N, seed=11)
    rng = np.random.default_rng(M + K + N)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, M - 2, M - 1], rng.choice(M, 384, replace=False)]))
    check(w, rows=rows, what=f"{M}x{K} N={N}")


def test_mma_lm_head_shape_sampled_rows():
    # 1187 row tiles: CTAs of four whole tiles each, two waves, a partial
    # last group
    M, K, N = 151936, 4096, 8
    w = syn.dense_nvfp4(M, K, N=N, seed=13)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 127, 128, 511, 512, M - 129, M - 128, M - 1], rng.choice(M, 256, replace=False)]))
    check(w, rows=rows, what=f"{M}x{K} N={N}")


def test_mma_deterministic_and_auto_selects_it():
    w = syn.dense_nvfp4(12288, 4096, N=8, seed=2)
    y1, y2 = run(w), run(w)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    y_auto = run(w, path=bqd.BQD_PATH_AUTO)
    assert np.array_equal(y1.view(np.uint32), y_auto.view(np.uint32))


def test_mma_one_hot_selects_dequantised_column_exactly():
    M, K = 300, 2048
    w = syn.dense_nvfp4(M, K, N=6, seed=5)
    ks = (0, 1, 255, 256, 1023, 2047)
    x = np.zeros((6, K), dtype=np.uint16)
    for n, k in enumerate(ks):
        x[n, k] = 0x3F80  # 1.0
    w["x"] = x
    y = run(w)
    W = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], M, K, dtype=np.float32)
    for n, k in enumerate(ks):
        assert np.array_equal(y[n], W[:, k]), f"column {k}"


def test_mma_sign_flip_zero_codes_and_tensor_scale_are_exact():
    w = syn.dense_nvfp4(500, 2048, N=3, seed=6)
    y = run(w)
    assert np.array_equal(run(dict(w, codes=w["codes"] ^ 0x88)), -y)
    assert np.all(run(dict(w, codes=np.zeros_like(w["codes"]))) == 0)
    assert np.array_equal(run(dict(w, ts=2.0)), 2 * run(dict(w, ts=1.0)))


def _bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", ["wide_range", "subnormal", "huge", "tiny", "zeros", "mixed_tokens"])
def test_mma_activation_range_cases(case):
    # f16 staging after a power-of-two prescale where the range allows it;
    # otherwise (or with subnormal input) bf16 operands.
    M, K, N = 300, 4096, 4
    w = syn.dense_nvfp4(M, K, N=N, seed=79)
    xf = torch.from_numpy(pins.bf16_lib(w["x"]).astype(np.float32))
    if case == "wide_range":
        xf[1, 5], xf[1, 100] = 2.0 ** 40, 2.0 ** -40
    elif case == "subnormal":
        xf[2, 7] = 2.0 ** -130
    elif case == "huge":
        xf = xf * 2.0 ** 100
    elif case == "tiny":
        xf = xf * 2.0 ** -120
    elif case == "zeros":
        xf = xf * 0
    elif case == "mixed_tokens":  # each token its own scale
        xf = xf * torch.tensor([2.0 ** -60, 1.0, 2.0 ** 50, 2.0 ** -100])[:, None]
    w["x"] = _bf16(xf.numpy())
    y = run(w)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    assert_within(y, ref, a, case)
    if case == "zeros":
        assert np.all(y == 0)


def test_mma_tokens_are_independent():
    # column n of an N = 8 call equals the N = 1 call on token n (tolerance:
    # the padded tokens and the staging mode may differ)
    M, K = 700, 3072
    w = syn.dense_nvfp4(M, K, N=8, seed=90)
    y = run(w)
    for n in (0, 3, 7):
        y1 = run(dict(w, x=w["x"][n:n + 1]))
        ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"][n:n + 1], M, K)
        assert_within(y[n:n + 1], ref, a, f"token {n} in N=8")
        assert_within(y1, ref, a, f"token {n} alone")


def test_mma_rejects_unsupported_arguments():
    for M, K, N in ((8, 4112, 2), (8, 128, 2)):  # K % 256 != 0
        w = syn.dense_nvfp4(M, K, N=N, seed=1)
        with pytest.raises(bqd.BqdError):
            run(w)
    q = syn.dense_q8_0(64, 1024, N=2, seed=1)
    y = torch.empty(2 * 64, dtype=torch.float32, device="cuda")
    with pytest.raises(bqd.BqdError):
        bqd.q8_0_gemv_path(dev(q["q"]), dev(q["d"]), dev(q["x"]), y, 64, 1024, 2, bqd.BQD_PATH_MMA)
    # an unsupported shape through AUTO still works (CUDA-core path)
    w = syn.dense_nvfp4(100, 4112, N=3, seed=2)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], 100, 4112)
    assert_within(run(w, path=bqd.BQD_PATH_AUTO), ref, a, "AUTO fallback")


def test_mma_back_to_back_calls_in_one_stream():
    # many launches in a row reuse TMEM and clusters: every result stays right
    ws = [syn.dense_nvfp4(M, K, N=N, seed=i % 4) for i, (M, K, N) in
          enumerate([(4096, 4096, 8), (300, 768, 2), (12288, 4096, 4), (129, 512, 16)] * 3)]
    outs = []
    for w in ws:
        out = torch.empty(w["x"].shape[0] * w["M"], dtype=torch.float32, device="cuda")
        bqd.nvfp4_gemv_path(dev(w["codes"]), dev(w["scales"]), w["ts"], dev(w["x"]), out, w["M"], w["K"],
                            w["x"].shape[0], bqd.BQD_PATH_MMA)
        outs.append(out)
    torch.cuda.synchronize()
    for w, out in zip(ws[:4], outs[:4]):
        rows = np.arange(0, w["M"], 7)
        ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], w["M"], w["K"], rows=rows)
        assert_within(out.cpu().numpy().reshape(-1, w["M"])[:, rows], ref, a, f"{w['M']}x{w['K']}")
    for i in range(4, len(ws)):
        assert torch.equal(outs[i], outs[i - 4])
