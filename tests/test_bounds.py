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


def _bf16(v):
    import torch
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _split_h(h):
    """h as the MoE prefill layer carries it to the down GEMM's bf16
    operands: hi = bf16(h), lo = bf16(h - hi), summed in fp32."""
    hi = _bf16(h)
    lo = _bf16(h.astype(np.float32) - hi)
    return (hi + lo).astype(np.float32)


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
            if mistake == "h_split":  # not a mistake: the prefill layer's h, bf16 hi plus bf16 lo
                h = _split_h(h)
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


def test_h_split_into_two_bf16_parts_is_exact_to_2_pow_minus_16():
    # the two parts recover fp32 h to 2^-16 of its size (each bf16 rounding
    # keeps 8 significant bits: |h - hi| <= 2^-9 |h|, |(h - hi) - lo| <=
    # 2^-9 |h - hi|), over 60 binades, signs and zeros. One bf16 alone can be
    # 2^-9 = 1.95e-3 off per element: when those errors align with the down
    # weights' signs, the down GEMV's error exceeds its 1e-3 * sum|w h|
    # allowance, which is why the prefill layer carries both parts
    rng = np.random.default_rng(7)
    h = (rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 30, 200000))).astype(np.float32)
    h[:4] = [0.0, -0.0, 1.0, -3.0]
    err = np.abs(_split_h(h).astype(np.float64) - h.astype(np.float64))
    assert np.all(err <= 2.0 ** -16 * np.abs(h.astype(np.float64)))
    # one bf16 alone is 2^-9 off at worst, and reaches well past 2^-12
    h64 = h.astype(np.float64)
    nz = h64 != 0
    err1 = np.abs(_bf16(h).astype(np.float64) - h64)
    assert np.max(err1[nz] / np.abs(h64[nz])) > 2.0 ** -10


def test_bound_holds_for_the_prefill_split_of_h():
    # the prefill layer's reading (h as bf16 hi + lo) stays inside the MoE
    # bound it is tested against, with room to spare
    L = _layer()
    sel, wts = oracle.moe_route(L["logits"], L["topk"])
    yref, parts = oracle.moe_layer(L, sel=sel, weights=wts, want_parts=True)
    tol = moe_y_tolerance(L, sel, wts, parts)
    assert np.all(np.abs(_fp32_layer(L, sel, wts, mistake="h_split") - yref) <= 1e-2 * tol)
