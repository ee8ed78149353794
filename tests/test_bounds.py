"""Pins of the propagated MoE bound (tests/bounds.py), on the CPU.

The bound must hold for an honest fp32 evaluation of the layer and must be
tight enough that plausible mistakes break it. The fp32 evaluation here uses
library decoders (tests/pins.py), numpy float32 matmuls and numpy's exp; the
mistakes are planted in that CPU evaluation, never on a GPU."""
import numpy as np
import pytest

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins
from tests.bounds import moe_y_tolerance


def _layer():
    return syn.moe_layer(T=3, E=16, H=256, I=128, topk=4, seed=11)


def _fp32_layer(L, sel, wts, mistake=None):
    """The layer in fp32 arithmetic, optionally with one planted mistake."""
    T, H, I, topk = L["T"], L["H"], L["I"], L["topk"]
    X = pins.bf16_lib(L["x"]).astype(np.float32)
    y = np.zeros((T, H), dtype=np.float32)
    for t in range(T):
        for s in range(topk):
            e = int(sel[t, s])
            if mistake == "wrong_expert" and s == 1:
                e = (e + 1) % L["E"]
            Wgu = pins.nvfp4_weight_lib(L["gu_codes"][e], L["gu_scales"][e], L["gu_ts"][e]).astype(np.float32)
            Wdn = pins.nvfp4_weight_lib(L["dn_codes"][e], L["dn_scales"][e], L["dn_ts"][e]).astype(np.float32)
            gu = Wgu @ X[t]
            g, u = gu[:I], gu[I:]
            if mistake == "gate_up_swapped":
                g, u = u, g
            h = g / (np.float32(1) + np.exp(-g)) * u
            if mistake == "no_silu":
                h = g * u
            d = Wdn @ h
            w = np.float32(wts[t, s])
            if mistake == "unnormalised":  # the full softmax's probability, not renormalised over the top k
                lg = L["logits"][t].astype(np.float64)
                w = np.float32(np.exp(lg[e] - lg.max()) / np.exp(lg - lg.max()).sum())
            if mistake == "slot_dropped" and s == topk - 1:
                continue
            y[t] = np.float32(y[t] + w * d)
    return y


def test_bound_holds_for_fp32_evaluation():
    L = _layer()
    sel, wts = oracle.moe_route(L["logits"], L["topk"])
    yref, parts = oracle.moe_layer(L, sel=sel, weights=wts, want_parts=True)
    tol = moe_y_tolerance(L, sel, wts, parts)
    y32 = _fp32_layer(L, sel, wts)
    assert np.all(np.abs(y32 - yref) <= tol)
    # the bound is a small fraction of the outputs' magnitude sum_s w_s * sum_j |W_dn h|
    # (it carries the GEMV tolerance 1e-3 * sum|w x| of both projections)
    scale = np.einsum("ts,tsh->th", wts, parts["ad"])
    assert np.max(tol / scale) < 0.05


@pytest.mark.parametrize("mistake", ["gate_up_swapped", "no_silu", "unnormalised", "slot_dropped", "wrong_expert"])
def test_bound_catches_planted_mistakes(mistake):
    L = _layer()
    sel, wts = oracle.moe_route(L["logits"], L["topk"])
    yref, parts = oracle.moe_layer(L, sel=sel, weights=wts, want_parts=True)
    tol = moe_y_tolerance(L, sel, wts, parts)
    y = _fp32_layer(L, sel, wts, mistake=mistake)
    assert np.any(np.abs(y - yref) > tol), f"{mistake} passed the bound"
