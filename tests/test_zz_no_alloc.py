"""The MoE entry point that allocates nothing (moe_grouped_gemv_noalloc).

It serves callers that cannot call cudaMalloc, such as plug-ins whose host
program owns all device memory, by keeping its scratch in an array inside
the library. This file runs last so that a failure here does not hide the
other GPU tests; it must pass on its own in a fresh process too. The check:
two calls in a row through the C ABI each match the workspace entry point
(moe_grouped_gemv) within the MoE tolerance of the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.gpu_util import assert_within, dev, need_gpu

pytestmark = pytest.mark.gpu


def _route(L):
    T, E, topk = L["T"], L["E"], L["topk"]
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    ptok = torch.empty(T * topk, dtype=torch.int32, device="cuda")
    pw = torch.empty(T * topk, dtype=torch.float32, device="cuda")
    pslot = torch.empty(T * topk, dtype=torch.int32, device="cuda")
    bqd.moe_route_topk(dev(L["logits"]), T, E, topk, off, ptok, pw, pslot)
    return off, ptok, pw, pslot


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    need_gpu()
    L = syn.moe_layer(T=6, E=64, H=1024, I=256, topk=8, seed=41)
    T, E, H, I, topk = L["T"], L["E"], L["H"], L["I"], L["topk"]
    w = [dev(L[k]) for k in ("gu_codes", "gu_scales", "gu_ts", "dn_codes", "dn_scales", "dn_ts", "x")]
    off, ptok, pw, pslot = _route(L)

    wsb = bqd.moe_workspace_bytes(T, topk, H, I)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    y_ref = torch.empty(T * H, dtype=torch.float32, device="cuda")
    bqd.moe_grouped_gemv(*w, off, ptok, pw, pslot, y_ref, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) == 0
    ref = y_ref.cpu().numpy().reshape(T, H)

    # the tolerance of the other MoE tests: 1e-3 * sum_s w_s * sum|W_dn h| + 1e-6
    sel, wts = oracle.moe_route(L["logits"], topk)
    _, parts = oracle.moe_layer(L, sel=sel, weights=wts, want_parts=True)
    scale = np.einsum("ts,tsh->th", wts, parts["ad"])

    L_ = bqd.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y = torch.full((T * H,), float("nan"), dtype=torch.float32, device="cuda")
        st = L_.moe_grouped_gemv_noalloc(*[t.data_ptr() for t in w], off.data_ptr(), ptok.data_ptr(),
                                         pw.data_ptr(), pslot.data_ptr(), y.data_ptr(), E, H, I, T, topk, stream)
        assert st == 0, f"call {call}: status {st}"
        got = y.cpu().numpy().reshape(T, H)
        assert_within(got, ref, scale, f"no-alloc call {call}", rel=1e-3, absol=1e-6)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    need_gpu()
    t = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = t.data_ptr()
    # T * topk = 8192 pairs with H = 1024, I = 256 needs ~42 MB of scratch
    st = bqd.lib().moe_grouped_gemv_noalloc(*([p] * 12), 64, 1024, 256, 1024, 8, None)
    assert st == 6  # BQD_ERR_WORKSPACE, returned before any launch
    torch.cuda.synchronize()
