"""NVFP4 GEMV on the GPU against the fp64 oracle: the method's tolerance
|y - y_ref| <= 1e-3 * sum|w x| + 1e-6 per output, plus exact invariants."""
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


def run(w, N=None, path=None):
    M, K = w["M"], w["K"]
    N = N or w["x"].shape[0]
    out = Guarded(N * M)
    args = (dev(w["codes"]), dev(w["scales"]), w["ts"], dev(w["x"]), out.ptr, M, K, N)
    if path is None:
        bqd.nvfp4_gemv(*args)
    else:
        bqd.nvfp4_gemv_path(*args, path)
    return out.get().reshape(N, M)


def check(w, rows=None, what=""):
    y = run(w)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], w["M"], w["K"], rows=rows)
    got = y if rows is None else y[:, rows]
    assert_within(got, ref, a, what)
    return y


def test_tiny_workload():
    check(syn.tiny_nvfp4(seed=0), what="256x512 N=1")


def test_worked_example(golden):
    g = golden("nvfp4_worked_example.txt")
    h = lambda v: [int(t, 16) for t in v]
    w = {"M": 2, "K": 32, "ts": float(g["ts"][0][0]),
         "codes": np.array([h(g["codes_row0"][0]), h(g["codes_row1"][0])], dtype=np.uint8),
         "scales": np.array([h(g["scales_row0"][0]), h(g["scales_row1"][0])], dtype=np.uint8),
         "x": np.array([h(g["x_col0"][0]), h(g["x_col1"][0])], dtype=np.uint16)}
    y = run(w)
    want = np.array([[float(v) for v in g["y_col0"][0]], [float(v) for v in g["y_col1"][0]]])
    a = np.array([[float(v) for v in g["a_col0"][0]], [float(v) for v in g["a_col1"][0]]])
    assert_within(y, want, a, "worked example")


@pytest.mark.parametrize("M,K,N", [
    (1, 16, 1), (1, 32, 1), (127, 48, 3), (129, 512, 5), (300, 4096, 1), (77, 4112, 2),
    (513, 1024, 8), (64, 2048, 16), (200, 8192, 9), (100, 12288, 16), (33, 16, 16), (1000, 96, 4),
])
def test_edge_shapes(M, K, N):
    check(syn.dense_nvfp4(M, K, N=N, seed=M * 7 + K + N), what=f"{M}x{K} N={N}")


@pytest.mark.parametrize("M,K", syn.NVFP4_SHAPES)
def test_full_size_n1(M, K):
    check(syn.dense_nvfp4(M, K, N=1, seed=0), what=f"{M}x{K} N=1")


@pytest.mark.parametrize("M,K", syn.VERIFY_SHAPES)
@pytest.mark.parametrize("N", [4, 8])
def test_full_size_verify_sampled_rows(M, K, N):
    w = syn.dense_nvfp4(M, K, N=N, seed=0)
    rng = np.random.default_rng(M + N)
    rows = np.unique(np.concatenate([[0, 1, M - 2, M - 1], rng.choice(M, 512, replace=False)]))
    check(w, rows=rows, what=f"{M}x{K} N={N}")


def test_deterministic_and_path_equivalence():
    w = syn.dense_nvfp4(12288, 4096, N=1, seed=1)
    y1, y2 = run(w), run(w)
    y3 = run(w, path=bqd.BQD_PATH_CUDA_CORE)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert np.array_equal(y1.view(np.uint32), y3.view(np.uint32))


def test_one_hot_selects_dequantised_column_exactly():
    w = syn.dense_nvfp4(300, 1024, N=4, seed=5)
    x = np.zeros((4, 1024), dtype=np.uint16)
    for n, k in enumerate((0, 1, 511, 1023)):
        x[n, k] = 0x3F80
    w["x"] = x
    y = run(w)
    W = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], 300, 1024, dtype=np.float32)
    for n, k in enumerate((0, 1, 511, 1023)):
        assert np.array_equal(y[n], W[:, k])


def test_sign_flip_zero_codes_and_tensor_scale_are_exact():
    w = syn.dense_nvfp4(500, 2048, N=2, seed=6)
    y = run(w)
    neg = dict(w, codes=w["codes"] ^ 0x88)
    assert np.array_equal(run(neg), -y)
    zero = dict(w, codes=np.zeros_like(w["codes"]))
    assert np.all(run(zero) == 0)
    y1 = run(dict(w, ts=1.0))
    y2 = run(dict(w, ts=2.0))
    assert np.array_equal(y2, 2 * y1)


def test_empty_shapes():
    out = Guarded(8, fill=5.0)
    bqd.nvfp4_gemv(None, None, 1.0, None, out.ptr, 4, 0, 2)  # K == 0: y = 0
    assert np.all(out.get() == 0)
    bqd.nvfp4_gemv(None, None, 1.0, None, None, 0, 64, 1)  # M == 0: nothing
    torch.cuda.synchronize()


# ---------------------------------------------------------------- compute paths
@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert bqd.bqd_device_error() == 0, "a pipeline wait ran out"


@pytest.mark.parametrize("M,K", syn.NVFP4_SHAPES + [(1, 256), (7, 512), (200, 2304), (3000, 16384)])
def test_stream_and_cuda_core_paths_match_oracle(M, K):
    w = syn.dense_nvfp4(M, K, N=1, seed=K + M)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    for path in (bqd.BQD_PATH_STREAM, bqd.BQD_PATH_CUDA_CORE):
        y = run(w, path=path)
        assert_within(y, ref, a, f"{M}x{K} path {path}")


# every K the direct path instantiates, row counts around the warp split
# (1 row; fewer rows than warps; odd splits; a multiple of 152 x 32 warps)
@pytest.mark.parametrize("M,K", syn.NVFP4_SHAPES + [(1, 1024), (31, 2048), (257, 3072), (4864, 4096),
                                                    (1000, 6144), (333, 8192), (77, 12288), (3001, 16384)])
def test_direct_path_matches_oracle(M, K):
    w = syn.dense_nvfp4(M, K, N=1, seed=K + 3 * M)
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    assert_within(run(w, path=bqd.BQD_PATH_DIRECT), ref, a, f"{M}x{K} direct")


def test_direct_path_rejects_unsupported_shapes():
    for M, K, N in ((8, 4112, 1), (8, 5120, 1), (8, 512, 1), (8, 1024, 2)):
        w = syn.dense_nvfp4(M, K, N=N, seed=1)
        with pytest.raises(bqd.BqdError):
            run(w, path=bqd.BQD_PATH_DIRECT)


def test_stream_path_rejects_unsupported_shapes():
    w = syn.dense_nvfp4(8, 4112, N=1, seed=1)
    with pytest.raises(bqd.BqdError):
        run(w, path=bqd.BQD_PATH_STREAM)
    w = syn.dense_nvfp4(8, 1024, N=2, seed=1)
    with pytest.raises(bqd.BqdError):
        run(w, path=bqd.BQD_PATH_STREAM)


def _bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", ["wide_range", "subnormal", "huge", "tiny", "zeros"])
def test_stream_activation_range_cases(case):
    M, K = 300, 4096
    w = syn.dense_nvfp4(M, K, N=1, seed=77)
    xf = torch.from_numpy(pins.bf16_lib(w["x"])[0].astype(np.float32))
    if case == "wide_range":      # 2^40 .. 2^-40: beyond f16's exact range -> exact fp32 path
        xf[5], xf[100] = 2.0 ** 40, 2.0 ** -40
    elif case == "subnormal":     # a bf16 subnormal -> exact fp32 path
        xf[7] = 2.0 ** -130
    elif case == "huge":          # everything large: f16 path with a large power-of-two prescale
        xf = xf * 2.0 ** 100
    elif case == "tiny":          # everything small: f16 path with a large power-of-two upscale
        xf = xf * 2.0 ** -120
    elif case == "zeros":
        xf = xf * 0
    w["x"] = _bf16(xf.numpy())[None]
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    for path in (bqd.BQD_PATH_STREAM, bqd.BQD_PATH_DIRECT):
        y = run(w, path=path)
        assert_within(y, ref, a, f"{case} path {path}", absol=0.0 if case != "zeros" else 0.0)
        if case == "zeros":
            assert np.all(y == 0)


def test_stream_nonfinite_activation_pattern():
    M, K = 64, 512
    w = syn.dense_nvfp4(M, K, N=1, seed=78)
    x = w["x"].copy()
    x[0, 3] = 0x7F80  # +inf
    w["x"] = x
    _nonfinite_check(w, run(w, path=bqd.BQD_PATH_STREAM), M, K)
    w2 = syn.dense_nvfp4(M, 1024, N=1, seed=79)
    x2 = w2["x"].copy()
    x2[0, 700] = 0xFF80  # -inf
    w2["x"] = x2
    _nonfinite_check(w2, run(w2, path=bqd.BQD_PATH_DIRECT), M, 1024)


def _nonfinite_check(w, y, M, K):
    ref, _ = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    assert np.array_equal(np.isnan(y[0]), np.isnan(ref[0]))
    assert np.array_equal(np.isinf(y[0]), np.isinf(ref[0]))
    fin = np.isfinite(ref[0])
    assert np.array_equal(np.sign(y[0][~fin & ~np.isnan(ref[0])]), np.sign(ref[0][~fin & ~np.isnan(ref[0])]))


# ---------------------------------------------------------------- dependent launch
@pytest.fixture
def pdl_on():
    prev = bqd.set_launch_flags(bqd.BQD_LAUNCH_PDL)
    yield
    bqd.set_launch_flags(prev)


def test_pdl_chain_is_bit_identical(pdl_on):
    ws = [syn.dense_nvfp4(M, K, N=1, seed=i) for i, (M, K) in enumerate(syn.NVFP4_SHAPES * 2)]
    dw = [(dev(w["codes"]), dev(w["scales"]), dev(w["x"])) for w in ws]
    outs = [torch.empty(w["M"], dtype=torch.float32, device="cuda") for w in ws]

    def chain():
        for w, (c, s, x), y in zip(ws, dw, outs):
            bqd.nvfp4_gemv(c, s, w["ts"], x, y, w["M"], w["K"], 1)
        torch.cuda.synchronize()
        return [y.cpu().numpy().copy() for y in outs]

    with_pdl = chain()
    bqd.set_launch_flags(0)
    without = chain()
    for a, b in zip(with_pdl, without):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_pdl_output_may_overwrite_previous_input(pdl_on):
    # call A reads x_a; call B, launched right after it, writes its output over
    # x_a's memory: B must not write before A has finished reading
    K = 8192
    wa = syn.dense_nvfp4(12288, K, N=1, seed=31)
    wb = syn.dense_nvfp4(K // 2, 4096, N=1, seed=32)
    ref_a, a_a = oracle.nvfp4_gemv(wa["codes"], wa["scales"], wa["ts"], wa["x"], 12288, K)
    for _ in range(3):
        shared = dev(wa["x"]).view(torch.uint8)  # K bf16 = 2K bytes, later K/2 fp32
        ya = torch.empty(12288, dtype=torch.float32, device="cuda")
        bqd.nvfp4_gemv(dev(wa["codes"]), dev(wa["scales"]), wa["ts"], shared, ya, 12288, K, 1)
        bqd.nvfp4_gemv(dev(wb["codes"]), dev(wb["scales"]), wb["ts"], dev(wb["x"]), shared, K // 2, 4096, 1)
        torch.cuda.synchronize()
        assert_within(ya.cpu().numpy()[None], ref_a, a_a, "A under PDL")


# ---------------------------------------------------------------- N = 1 stream kernel, exact invariants
@pytest.mark.parametrize("path", ["stream", "direct"])
def test_n1_exact_invariants(path):
    """Through the N = 1 paths (the decode hot path): a one-hot x
    gives the dequantised column bit for bit; a one-hot x of 3 gives the
    exact product rounded once; sign flip negates exactly; zero codes give
    zero; ts = 2 doubles exactly."""
    M, K = 1000, 4096
    P = bqd.BQD_PATH_STREAM if path == "stream" else bqd.BQD_PATH_DIRECT
    w = syn.dense_nvfp4(M, K, N=1, seed=12)
    W = oracle.nvfp4_dequant(w["codes"], w["scales"], w["ts"], M, K, dtype=np.float32)
    for k in (0, 1, 15, 16, 255, 256, 2047, 4095):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80  # 1.0
        assert np.array_equal(run(dict(w, x=x), path=P)[0], W[:, k]), f"one-hot k={k}"
        x[0, k] = 0x4040  # 3.0
        ref, _ = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], x, M, K)
        assert np.array_equal(run(dict(w, x=x), path=P)[0], ref[0].astype(np.float32)), f"one-hot 3 k={k}"
    y = run(w, path=P)
    assert np.array_equal(run(dict(w, codes=w["codes"] ^ 0x88), path=P), -y)
    assert np.all(run(dict(w, codes=np.zeros_like(w["codes"])), path=P) == 0)
    y1 = run(dict(w, ts=1.0), path=P)
    assert np.array_equal(run(dict(w, ts=2.0), path=P), 2 * y1)


def test_stream_bounded_wait_gives_up_and_reports():
    """Failure path without a GPU fault: the producer withholds each CTA's last
    ring stage (no copy of it is ever issued), so the consumers' bounded wait
    for it runs out after 2^20 cycles; the call completes, bit 0 of the
    device error word is set, a second read finds it cleared, and the next
    normal call is correct."""
    M, K = 2000, 4096
    w = syn.dense_nvfp4(M, K, N=1, seed=15)
    assert bqd.bqd_device_error() == 0
    bqd.debug_stream_fault(True, 1 << 20)
    try:
        run(w, path=bqd.BQD_PATH_STREAM)  # returns: the waits gave up instead of hanging
        torch.cuda.synchronize()
    finally:
        bqd.debug_stream_fault(False, 0)
    assert bqd.bqd_device_error() & 1
    assert bqd.bqd_device_error() == 0
    ref, a = oracle.nvfp4_gemv(w["codes"], w["scales"], w["ts"], w["x"], M, K)
    assert_within(run(w, path=bqd.BQD_PATH_STREAM), ref, a, "after the failure test")
