"""MoE prefill layer (moe_prefill_layer: routing, gathered tokens, grouped
tensor-core GEMMs, SiLU * up with h split into two bf16 parts, fixed-order
combine) against the fp64 oracle within the propagated MoE bound
(tests/bounds.py), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.bounds import moe_check
from tests.gpu_util import dev, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert bqd.bqd_device_error() == 0, "a wait ran out"


def run(L):
    T, E, H, I, topk = L["T"], L["E"], L["H"], L["I"], L["topk"]
    wsb = bqd.moe_prefill_workspace_bytes(T, topk, H, I, E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    y = torch.full((T * H,), float("nan"), dtype=torch.float32, device="cuda")
    bqd.moe_prefill_layer(dev(L["logits"]), dev(L["gu_codes"]), dev(L["gu_scales"]), dev(L["gu_ts"]),
                          dev(L["dn_codes"]), dev(L["dn_scales"]), dev(L["dn_ts"]), dev(L["x"]), y, ws, wsb,
                          E, H, I, T, topk)
    return y.cpu().numpy().reshape(T, H)


@pytest.mark.parametrize("T,E,H,I,topk", [(64, 32, 1024, 256, 4), (7, 16, 512, 128, 2), (200, 64, 1024, 512, 8),
                                           (33, 8, 256, 64, 8)])
def test_prefill_layer_matches_oracle(T, E, H, I, topk):
    L = syn.moe_layer(T=T, E=E, H=H, I=I, topk=topk, seed=T + E)
    y = run(L)
    sel, w = oracle.moe_route(L["logits"], topk)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=w, want_parts=True)
    moe_check(y, L, sel, w, parts, yref, f"prefill T={T} E={E} H={H} I={I} top-{topk}")


def test_prefill_layer_full_shape_and_determinism():
    # the layer's shapes (E = 256, H = 2048, I = 512, top-8) over 128 tokens
    L = syn.moe_layer(T=128, seed=5)
    y = run(L)
    sel, w = oracle.moe_route(L["logits"], L["topk"])
    yref, parts = oracle.moe_layer(L, sel=sel, weights=w, want_parts=True)
    moe_check(y, L, sel, w, parts, yref, "prefill T=128 E=256")
    assert np.array_equal(y.view(np.uint32), run(L).view(np.uint32))


def test_prefill_layer_agrees_with_the_small_batch_path():
    # the same layer at T = 16 through moe_layer (small-batch kernels): both
    # within the bound of the oracle, and close to each other
    L = syn.moe_layer(T=16, E=64, H=1024, I=256, topk=8, seed=9)
    y = run(L)
    wsb = bqd.moe_layer_workspace_bytes(16, 8, 1024, 256, 64)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    ys = torch.empty(16 * 1024, dtype=torch.float32, device="cuda")
    bqd.moe_layer(dev(L["logits"]), dev(L["gu_codes"]), dev(L["gu_scales"]), dev(L["gu_ts"]), dev(L["dn_codes"]),
                  dev(L["dn_scales"]), dev(L["dn_ts"]), dev(L["x"]), ys, ws, wsb, 64, 1024, 256, 16, 8)
    sel, w = oracle.moe_route(L["logits"], 8)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=w, want_parts=True)
    moe_check(y, L, sel, w, parts, yref, "prefill")
    moe_check(ys.cpu().numpy().reshape(16, 1024), L, sel, w, parts, yref, "small path")


def test_prefill_layer_rejections():
    L = syn.moe_layer(T=4, E=8, H=256, I=64, topk=2, seed=1)
    wsb = bqd.moe_prefill_workspace_bytes(4, 2, 256, 64, 8)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    y = torch.empty(4 * 256, dtype=torch.float32, device="cuda")
    args = [dev(L[k]) for k in ("logits", "gu_codes", "gu_scales", "gu_ts", "dn_codes", "dn_scales", "dn_ts", "x")]
    with pytest.raises(bqd.BqdError):  # workspace too small
        bqd.moe_prefill_layer(*args, y, ws, wsb - 256, 8, 256, 64, 4, 2)
    with pytest.raises(bqd.BqdError):  # H % 64 != 0
        bqd.moe_prefill_layer(*args, y, ws, wsb, 8, 250, 64, 4, 2)
    with pytest.raises(bqd.BqdError):  # T * topk > 8192
        bqd.moe_prefill_layer(*args, y, ws, wsb, 8, 256, 64, 8193, 1)
