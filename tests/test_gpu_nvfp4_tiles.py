"""Warp-tile tensor-core NVFP4 GEMV (BQD_PATH_TILES) against the fp64 oracle.

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


def run(w, path=bqd.BQD_PATH_TILES, N=None):
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


# 8-row tiles with ragged last tiles; CTAs of one to many tiles whose
# (tile, chunk) units are split over 16 warps, so that tiles are shared by
# two or more warps (and some warps get no unit); token counts 2 to 16
# (slots 8..15 in use from N = 9); the largest activations (N K = 32768).
@pytest.mark.parametrize("M,K,N", [
    (1, 1024, 2), (3, 1024, 16), (8, 2048, 4), (9, 1024, 9), (40, 1024, 3), (100, 4096, 8), (257, 3072, 5),
    (1000, 2048, 16), (1217, 1024, 7), (2048, 8192, 2), (5000, 2048, 12), (300, 16384, 2), (77, 4096, 8),
    (4099, 1024, 4), (20000, 1024, 11), (64, 3072, 10),
])
def test_tiles_match_oracle(M, K, N):
    check(syn.dense_nvfp4(M, K, N=N, seed=5 * M + K + N), what=f"{M}x{K} N={N}")


@pytest.mark.parametrize("M,K", syn.VERIFY_SHAPES + [(4096, 12288)])
@pytest.mark.parametrize("N", [2, 4, 8])
def test_tiles_full_size_sampled_rows(M, K, N):
    if N * K > 32768:
        pytest.skip("activations larger than the path takes")
    w = syn.dense_nvfp4(M, K, N=N, seed=17)
    rng = np.random.default_rng(M + K + N)
    rows = np.unique(np.concatenate([[0, 1, 7, 8, M - 9, M - 8, M - 2, M - 1], rng.choice(M, 384, replace=False)]))
    check(w, rows=rows, what=f"{M}x{K} N={N}")


def test_tiles_lm_head_shape_sampled_rows():
    M, K, N = 151936, 4096, 8
    w = syn.dense_nvfp4(M, K, N=N, seed=19)
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, 7, 8, 999, 1000, M - 9, M - 8, M - 1], rng.choice(M, 256, replace=False)]))
    check(w, rows=rows, what=f"{M}x{K} N={N}")


def test_tiles_deterministic_and_agree_with_the_tcgen05_path():
    w = syn.dense_nvfp4(12288, 4096, N=8, seed=2)
    y1, y2 = run(w), run(w)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    rows = np.arange(0, 12288, 97)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], 12288, 4096, rows=rows)
    assert_within(y1[:, rows], ref, a, "tiles")
    assert_within(run(w, path=bqd.BQD_PATH_MMA)[:, rows], ref, a, "tcgen05")


def test_tiles_one_hot_selects_dequantised_column_exactly():
    M, K = 300, 2048
    w = syn.dense_nvfp4(M, K, N=10, seed=5)
    ks = (0, 1, 31, 32, 127, 128, 255, 1023, 1024, 2047)
    x = np.zeros((10, K), dtype=np.uint16)
    for n, k in enumerate(ks):
        x[n, k] = 0x3F80  # 1.0
    w["x"] = x
    y = run(w)
    W = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], M, K, dtype=np.float32)
    for n, k in enumerate(ks):
        assert np.array_equal(y[n], W[:, k]), f"column {k}"


def test_tiles_sign_flip_zero_codes_and_tensor_scale_are_exact():
    w = syn.dense_nvfp4(500, 2048, N=3, seed=6)
    y = run(w)
    assert np.array_equal(run(dict(w, codes=w["codes"] ^ 0x88)), -y)
    assert np.all(run(dict(w, codes=np.zeros_like(w["codes"]))) == 0)
    assert np.array_equal(run(dict(w, ts=2.0)), 2 * run(dict(w, ts=1.0)))


def _bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", ["wide_range", "subnormal", "huge", "tiny", "zeros", "mixed_tokens", "inf_nan"])
def test_tiles_activation_range_cases(case):
    # f16 staging after a power-of-two prescale per token where the ranges
    # allow it; otherwise (or with subnormal, inf or NaN input) bf16 operands
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
    elif case == "inf_nan":
        xf[3, 9] = float("inf")
    w["x"] = _bf16(xf.numpy())
    y = run(w)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    if case == "inf_nan":
        # token 3 meets an infinity: its outputs are not finite; the others are exact as usual
        assert not np.isfinite(y[3]).any()
        assert_within(y[:3], ref[:3], a[:3], case)
        return
    assert_within(y, ref, a, case)
    if case == "zeros":
        assert np.all(y == 0)


def test_tiles_tokens_are_independent():
    M, K = 700, 2048
    w = syn.dense_nvfp4(M, K, N=12, seed=90)
    y = run(w)
    for n in (0, 5, 8, 11):
        y2 = run(dict(w, x=np.ascontiguousarray(w["x"][[n, (n + 1) % 12]])))
        ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"][n:n + 1], M, K)
        assert_within(y[n:n + 1], ref, a, f"token {n} in N=12")
        assert_within(y2[:1], ref, a, f"token {n} in N=2")


def test_tiles_reject_unsupported_arguments():
    for M, K, N in ((8, 1536, 2), (8, 4096, 1), (8, 4096, 9), (8, 4096, 17)):
        w = syn.dense_nvfp4(M, K, N=min(N, 16), seed=1)
        with pytest.raises(bqd.BqdError):
            run(w, N=N) if N <= 16 else bqd.nvfp4_gemv_path(dev(w["codes"]), dev(w["scales"]), w["ts"],
                                                           dev(w["x"]), Guarded(N * M).ptr, M, K, N,
                                                           bqd.BQD_PATH_TILES)
    q = syn.dense_q8_0(64, 1024, N=2, seed=1)
    y = torch.empty(2 * 64, dtype=torch.float32, device="cuda")
    with pytest.raises(bqd.BqdError):
        bqd.q8_0_gemv_path(dev(q["q"]), dev(q["d"]), dev(q["x"]), y, 64, 1024, 2, bqd.BQD_PATH_TILES)
    # shapes the path does not take still work through AUTO
    for M, K, N in ((100, 1536, 3), (64, 16384, 16)):
        w = syn.dense_nvfp4(M, K, N=N, seed=2)
        ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
        assert_within(run(w, path=bqd.BQD_PATH_AUTO), ref, a, f"AUTO {M}x{K} N={N}")


def test_tiles_back_to_back_calls_in_one_stream():
    ws = [syn.dense_nvfp4(M, K, N=N, seed=i % 4) for i, (M, K, N) in
          enumerate([(4096, 4096, 8), (300, 1024, 2), (12288, 4096, 4), (129, 2048, 16)] * 3)]
    outs = []
    for w in ws:
        out = torch.empty(w["x"].shape[0] * w["M"], dtype=torch.float32, device="cuda")
        bqd.nvfp4_gemv_path(dev(w["codes"]), dev(w["scales"]), w["ts"], dev(w["x"]), out, w["M"], w["K"],
                            w["x"].shape[0], bqd.BQD_PATH_TILES)
        outs.append(out)
    torch.cuda.synchronize()
    for w, out in zip(ws[:4], outs[:4]):
        rows = np.arange(0, w["M"], 7)
        ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], w["M"], w["K"], rows=rows)
        assert_within(out.cpu().numpy().reshape(-1, w["M"])[:, rows], ref, a, f"{w['M']}x{w['K']}")
    for i in range(4, len(ws)):
        assert torch.equal(outs[i], outs[i - 4])
