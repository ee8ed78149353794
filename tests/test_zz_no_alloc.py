"""The MoE entry point that allocates nothing (moe_grouped_gemv_noalloc).

It serves callers that cannot call cudaMalloc, such as plug-ins whose host
program owns all device memory, by keeping its scratch in an array inside
the library. This file runs last so that a failure here does not hide the
other GPU tests; it must pass on its own in a fresh process too.

The check: two calls in a row through the C ABI, the first on a larger layer
than the second (so the first leaves more partial sums, counters and h rows
in the shared array than the second writes). Each call's output must equal,
bit for bit, the workspace entry point (moe_grouped_gemv) on the same inputs
(the same kernels in the same order), and must lie within the propagated
MoE bound of the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.bounds import moe_check
from tests.gpu_util import dev, need_gpu

pytestmark = pytest.mark.gpu


def _inputs(L):
    T, E, topk = L["T"], L["E"], L["topk"]
    w = [dev(L[k]) for k in ("gu_codes", "gu_scales", "gu_ts", "dn_codes", "dn_scales", "dn_ts", "x")]
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ptok = torch.empty(T * topk, dtype=torch.int32, device="cuda")
    pw = torch.empty(T * topk, dtype=torch.float32, device="cuda")
    pslot = torch.empty(T * topk, dtype=torch.int32, device="cuda")
    bqd.moe_route_topk(dev(L["logits"]), T, E, topk, off, ptok, pw, pslot)
    return w, (off, ptok, pw, pslot)


def _noalloc(L, w, lst):
    T, E, H, I, topk = L["T"], L["E"], L["H"], L["I"], L["topk"]
    y = torch.full((T * H,), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = bqd.lib().moe_grouped_gemv_noalloc(*[t.data_ptr() for t in w], *[t.data_ptr() for t in lst],
                                            y.data_ptr(), E, H, I, T, topk, stream)
    assert st == 0, f"status {st}"
    return y.cpu().numpy().reshape(T, H)


def _workspace(L, w, lst):
    T, E, H, I, topk = L["T"], L["E"], L["H"], L["I"], L["topk"]
    wsb = bqd.moe_workspace_bytes(T, topk, H, I)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    y = torch.full((T * H,), float("nan"), dtype=torch.float32, device="cuda")
    bqd.moe_grouped_gemv(*w, *lst, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) == 0
    return y.cpu().numpy().reshape(T, H)


# I = 256 runs the bulk-copy expert streams, I = 128 the register-streaming kernels
@pytest.mark.parametrize("I", [256, 128])
def test_noalloc_two_calls_match_workspace_entry_point_and_oracle(I):
    need_gpu()
    big = syn.moe_layer(T=12, E=64, H=1024, I=I, topk=8, seed=41)
    small = syn.moe_layer(T=5, E=64, H=1024, I=I, topk=8, seed=42)
    args = [(L, *_inputs(L)) for L in (big, small)]
    got = [_noalloc(L, w, lst) for L, w, lst in args]  # two calls in a row on the shared array
    for (L, w, lst), y, what in zip(args, got, ("first call (T=12)", "second call (T=5)")):
        ref = _workspace(L, w, lst)
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32)), f"{what}: differs from moe_grouped_gemv"
        sel, wts = oracle.moe_route(L["logits"], L["topk"])
        yref, parts = oracle.moe_layer(L, sel=sel, weights=wts, want_parts=True)
        moe_check(y, L, sel, wts, parts, yref, what)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    need_gpu()
    t = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = t.data_ptr()
    # T * topk = 8192 pairs with H = 1024, I = 256 needs ~42 MB of scratch
    st = bqd.lib().moe_grouped_gemv_noalloc(*([p] * 12), 64, 1024, 256, 1024, 8, None)
    assert st == 6  # BQD_ERR_WORKSPACE, returned before any launch
    torch.cuda.synchronize()
