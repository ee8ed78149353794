"""Decode-path epilogue fusions (nvfp4/q8_0_gemv_add, nvfp4/q8_0_gemv_silu_mul)
against the fp64 oracle, through the C ABI.

Tolerances are derived from the GEMV's, |y - y_ref| <= 1e-3 * sum|w x| + 1e-6:
  residual add: one more fp32 rounding of the sum, 2^-24 * (sum|w x| + |r|)
  beyond the GEMV bound;
  SiLU(g) * u: the GEMV bounds of g and u propagated through SiLU * u
  (tests/bounds.py silu_up_spread).
Exact cases (one-hot x, zero residual) are checked bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.bounds import silu_up_spread
from tests.gpu_util import Guarded, dev, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _weights(fmt, M, K, seed):
    if fmt == "nvfp4":
        w = syn.dense_nvfp4(M, K, N=1, seed=seed)
        return w, (w["codes"], w["scales"], w["ts"])
    w = syn.dense_q8_0(M, K, N=1, seed=seed)
    return w, (w["q"], w["d"])


def run_add(fmt, w, x, r, M, K, out=None):
    out = out if out is not None else Guarded(M)
    rp = r.data_ptr() if isinstance(r, torch.Tensor) else r
    if fmt == "nvfp4":
        bqd.nvfp4_gemv_add(dev(w["codes"]), dev(w["scales"]), w["ts"], dev(x), rp, out.ptr, M, K)
    else:
        bqd.q8_0_gemv_add(dev(w["q"]), dev(w["d"]), dev(x), rp, out.ptr, M, K)
    return out


def run_silu(fmt, w, x, I, K):
    out = Guarded(I)
    if fmt == "nvfp4":
        bqd.nvfp4_gemv_silu_mul(dev(w["codes"]), dev(w["scales"]), w["ts"], dev(x), out.ptr, I, K)
    else:
        bqd.q8_0_gemv_silu_mul(dev(w["q"]), dev(w["d"]), dev(x), out.ptr, I, K)
    return out.get()


def check_add(y, yref, a, r, what):
    tol = 1e-3 * a + 1e-6 + 2.0 ** -24 * (a + np.abs(r))
    err = np.abs(y.astype(np.float64) - yref)
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} outside, first {np.flatnonzero(bad)[:5]}"


def check_silu(h, href, g, u, ag, au, what):
    tol = silu_up_spread(g, u, href, ag, au)
    err = np.abs(h.astype(np.float64) - href)
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} outside, first {np.flatnonzero(bad)[:5]}"


# the layer shapes (down 4096 x 12288, attn out 4096 x 4096, a 6144-wide
# down) and ragged or small ones; every K the direct kernel takes
ADD_SHAPES = [(4096, 12288), (4096, 4096), (4096, 6144), (1, 1024), (7, 2048), (1000, 3072), (333, 8192),
              (77, 16384)]


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
@pytest.mark.parametrize("M,K", ADD_SHAPES)
def test_gemv_add_matches_oracle(fmt, M, K):
    w, wt = _weights(fmt, M, K, seed=M + K)
    r = np.random.default_rng(M).standard_normal((1, M)).astype(np.float32)
    y = run_add(fmt, w, w["x"], dev(r), M, K).get()
    yref, a = oracle.gemv_add(fmt, wt, w["x"], r, M, K)
    check_add(y, yref[0], a[0], r[0], f"{fmt} {M}x{K}")


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
def test_gemv_add_exact_cases_and_in_place(fmt):
    M, K = 1000, 4096
    w, wt = _weights(fmt, M, K, seed=4)
    r = np.random.default_rng(2).standard_normal((1, M)).astype(np.float32)
    # zero residual: the plain GEMV's result bit for bit
    y0 = run_add(fmt, w, w["x"], dev(np.zeros_like(r)), M, K).get()
    plain = Guarded(M)
    if fmt == "nvfp4":
        bqd.nvfp4_gemv(dev(w["codes"]), dev(w["scales"]), w["ts"], dev(w["x"]), plain.ptr, M, K, 1)
    else:
        bqd.q8_0_gemv(dev(w["q"]), dev(w["d"]), dev(w["x"]), plain.ptr, M, K, 1)
    assert np.array_equal(y0.view(np.uint32), plain.get().view(np.uint32))
    # one-hot x: fp32(dequantised column) + r, rounded once, bit for bit
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, 1234] = 0x3F80
    col = (oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], M, K, dtype=np.float32) if fmt == "nvfp4"
           else oracle.q8_0_dequant(w["q"], w["d"], M, K, dtype=np.float32))[:, 1234]
    y1 = run_add(fmt, w, x, dev(r), M, K).get()
    assert np.array_equal(y1, (col + r[0]).astype(np.float32))
    # in place: y is the residual
    buf = Guarded(M)
    buf.buf[64:64 + M] = torch.from_numpy(r[0]).cuda()
    run_add(fmt, w, w["x"], buf.ptr, M, K, out=buf)
    y2 = run_add(fmt, w, w["x"], dev(r), M, K).get()
    assert np.array_equal(buf.get().view(np.uint32), y2.view(np.uint32))


# gate_up shapes: the 12288 x 4096 gate/up (I = 6144), a 4096-wide MLP over
# K = 12288, and small or odd widths
SILU_SHAPES = [(6144, 4096), (2048, 12288), (1, 1024), (3, 2048), (500, 3072), (1000, 8192), (64, 16384)]


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
@pytest.mark.parametrize("I,K", SILU_SHAPES)
def test_gemv_silu_mul_matches_oracle(fmt, I, K):
    w, wt = _weights(fmt, 2 * I, K, seed=3 * I + K)
    h = run_silu(fmt, w, w["x"], I, K)
    href, g, u, ag, au = oracle.gemv_silu_mul(fmt, wt, w["x"], I, K)
    check_silu(h, href[0], g[0], u[0], ag[0], au[0], f"{fmt} I={I} K={K}")


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
def test_gemv_silu_mul_pairs_rows_and_is_deterministic(fmt):
    I, K = 777, 2048
    w, wt = _weights(fmt, 2 * I, K, seed=9)
    h1, h2 = run_silu(fmt, w, w["x"], I, K), run_silu(fmt, w, w["x"], I, K)
    assert np.array_equal(h1.view(np.uint32), h2.view(np.uint32))
    # gate and up rows swapped in memory: the oracle's swapped layer, not this one
    sw = dict(w)
    if fmt == "nvfp4":
        sw["codes"] = np.concatenate([w["codes"][I:], w["codes"][:I]])
        sw["scales"] = np.concatenate([w["scales"][I:], w["scales"][:I]])
        swt = (sw["codes"], sw["scales"], w["ts"])
    else:
        sw["q"] = np.concatenate([w["q"][I:], w["q"][:I]])
        sw["d"] = np.concatenate([w["d"][I:], w["d"][:I]])
        swt = (sw["q"], sw["d"])
    hs = run_silu(fmt, sw, w["x"], I, K)
    href, g, u, ag, au = oracle.gemv_silu_mul(fmt, swt, w["x"], I, K)
    check_silu(hs, href[0], g[0], u[0], ag[0], au[0], "swapped layout")
    assert not np.allclose(hs, h1)


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
def test_fusions_reject_unsupported_arguments(fmt):
    w, _ = _weights(fmt, 16, 1536, seed=1)
    r = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(bqd.BqdError):  # K not taken by the direct kernel
        run_add(fmt, w, w["x"], r, 16, 1536)
    with pytest.raises(bqd.BqdError):
        run_silu(fmt, w, w["x"], 8, 1536)
    w, _ = _weights(fmt, 16, 1024, seed=1)
    out = Guarded(16)
    with pytest.raises(bqd.BqdError):  # N = 2
        if fmt == "nvfp4":
            bqd.nvfp4_gemv_add(dev(w["codes"]), dev(w["scales"]), w["ts"], dev(np.repeat(w["x"], 2, 0)),
                               r.data_ptr(), out.ptr, 16, 1024, 2)
        else:
            bqd.q8_0_gemv_add(dev(w["q"]), dev(w["d"]), dev(np.repeat(w["x"], 2, 0)), r.data_ptr(), out.ptr, 16,
                              1024, 2)
    with pytest.raises(bqd.BqdError):  # no residual
        run_add(fmt, w, w["x"], 0, 16, 1024)
    with pytest.raises(bqd.BqdError):  # I = 0
        run_silu(fmt, w, w["x"], 0, 1024)


def test_mlp_block_in_a_captured_graph():
    # h = SiLU(gate . x) * (up . x), then y = down . h + x_res: a decode MLP
    # block as two fused launches, replayed from a CUDA graph, equals the
    # same launches run eagerly, bit for bit
    I, H = 6144, 4096
    gu = syn.dense_nvfp4(2 * I, H, N=1, seed=21)
    dn = syn.dense_nvfp4(H, I, N=1, seed=22)
    res = np.random.default_rng(3).standard_normal(H).astype(np.float32)
    d_gu = [dev(gu["codes"]), dev(gu["scales"])]
    d_dn = [dev(dn["codes"]), dev(dn["scales"])]
    x, r = dev(gu["x"]), dev(res)
    h = torch.empty(I, dtype=torch.float32, device="cuda")
    hbf = torch.empty(I, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(H, dtype=torch.float32, device="cuda")

    def block():
        bqd.nvfp4_gemv_silu_mul(d_gu[0], d_gu[1], gu["ts"], x, h, I, H)
        hbf.copy_(h)  # the down projection's activations are bf16, as the layer's input
        bqd.nvfp4_gemv_add(d_dn[0], d_dn[1], dn["ts"], hbf, r, y, H, I)

    block()
    torch.cuda.synchronize()
    y_eager = y.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        block()  # warm-up on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            bqd.nvfp4_gemv_silu_mul(d_gu[0], d_gu[1], gu["ts"], x, h, I, H, stream=s.cuda_stream)
            hbf.copy_(h)
            bqd.nvfp4_gemv_add(d_dn[0], d_dn[1], dn["ts"], hbf, r, y, H, I, stream=s.cuda_stream)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager)
    # and the block's result is the oracle's composition within the bounds
    href, gg, uu, ag, au = oracle.gemv_silu_mul("nvfp4", (gu["codes"], gu["scales"], gu["ts"]), gu["x"], I, H)
    check_silu(h.cpu().numpy(), href[0], gg[0], uu[0], ag[0], au[0], "graph h")
    hb = hbf.view(torch.int16).cpu().numpy().view(np.uint16)[None, :]
    yref, a = oracle.gemv_add("nvfp4", (dn["codes"], dn["scales"], dn["ts"]), hb, res[None, :], H, I)
    check_add(y.cpu().numpy(), yref[0], a[0], res, "graph y")
