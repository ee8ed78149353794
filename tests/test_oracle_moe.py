"""Pins of the oracle's MoE router and routed FFN: the hand-worked routing
example, library softmax/expit, library matmul brute force and reductions to
the dense GEMV."""
import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests import pins


def test_route_worked_example(golden):
    g = golden("moe_route_example.txt")
    logits = np.array([[float(v) for v in g["logits"][0]]], dtype=np.float32)
    for k in (3, 2):
        sel, w = oracle.moe_route(logits, k)
        assert sel[0].tolist() == [int(v) for v in g[f"k{k}_experts"][0]]
        assert np.allclose(w[0], [float(v) for v in g[f"k{k}_weights"][0]], rtol=0, atol=1e-15)


def test_route_matches_library_softmax():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((16, 256), dtype=np.float32)
    sel, w = oracle.moe_route(logits, 8)
    for t in range(16):
        order = np.argsort(-logits[t].astype(np.float64), kind="stable")[:8]
        assert sel[t].tolist() == order.tolist()
        p = softmax(logits[t].astype(np.float64))
        assert np.allclose(w[t], p[order] / p[order].sum(), rtol=1e-14, atol=0)
        assert np.allclose(w[t], softmax(logits[t, order].astype(np.float64)), rtol=1e-14, atol=0)
        assert abs(w[t].sum() - 1) < 1e-15


def test_route_ties_and_full_selection():
    logits = np.zeros((1, 8), dtype=np.float32)
    sel, w = oracle.moe_route(logits, 8)
    assert sel[0].tolist() == list(range(8))
    assert np.all(w == 1 / 8)
    logits = np.array([[1, 5, 5, 5, 0]], dtype=np.float32)
    sel, _ = oracle.moe_route(logits, 2)
    assert sel[0].tolist() == [1, 2]


def _numpy_moe(layer, sel, wts):
    """Brute force with library decoders, numpy matmul and scipy expit."""
    T, H, I, topk = layer["T"], layer["H"], layer["I"], layer["topk"]
    X = pins.bf16_lib(layer["x"])
    y = np.zeros((T, H))
    hs = np.zeros((T, topk, I))
    for t in range(T):
        for s in range(topk):
            e = sel[t, s]
            Wgu = pins.nvfp4_weight_lib(layer["gu_codes"][e], layer["gu_scales"][e], layer["gu_ts"][e])
            Wdn = pins.nvfp4_weight_lib(layer["dn_codes"][e], layer["dn_scales"][e], layer["dn_ts"][e])
            gu = Wgu @ X[t]
            g, u = gu[:I], gu[I:]
            h = g * expit(g) * u
            hs[t, s] = h
            y[t] += wts[t, s] * (Wdn @ h)
    return y, hs


@pytest.mark.parametrize("T,topk", [(1, 2), (3, 4)])
def test_moe_layer_matches_library_bruteforce(T, topk):
    layer = syn.moe_layer(T=T, E=6, H=64, I=32, topk=topk, seed=21, ts=0.05)
    sel, w = oracle.moe_route(layer["logits"], topk)
    y, parts = oracle.moe_layer(layer, want_parts=True)
    yref, href = _numpy_moe(layer, sel, w)
    scale = np.einsum("ts,tsh->th", w, parts["ad"]) + 1e-300
    assert np.all(np.abs(y - yref) <= 1e-11 * scale)
    assert np.allclose(parts["h"], href, rtol=1e-11, atol=1e-14)


def test_moe_identical_experts_reduce_to_one_ffn():
    layer = syn.moe_layer(T=2, E=5, H=64, I=32, topk=3, seed=22, ts=0.05)
    for k in ("gu_codes", "gu_scales", "dn_codes", "dn_scales"):
        layer[k] = np.ascontiguousarray(np.broadcast_to(layer[k][0], layer[k].shape))
    y = oracle.moe_layer(layer)
    # one dense FFN with the oracle's (separately pinned) dense GEMV
    g_u, _ = oracle.nvfp4_gemv(layer["gu_codes"][0], layer["gu_scales"][0], float(layer["gu_ts"][0]),
                               layer["x"], 64, 64)
    g, u = g_u[:, :32], g_u[:, 32:]
    h = g * expit(g) * u
    d, a = oracle.nvfp4_gemv_f64x(layer["dn_codes"][0], layer["dn_scales"][0], float(layer["dn_ts"][0]), h, 64, 32)
    assert np.all(np.abs(y - d) <= 1e-12 * a + 1e-300)


def test_moe_top1_is_gemv_chain():
    layer = syn.moe_layer(T=2, E=4, H=32, I=16, topk=1, seed=23, ts=0.1)
    sel, w = oracle.moe_route(layer["logits"], 1)
    assert np.all(w == 1.0)
    y, parts = oracle.moe_layer(layer, want_parts=True)
    for t in range(2):
        e = sel[t, 0]
        gu, _ = oracle.nvfp4_gemv(layer["gu_codes"][e], layer["gu_scales"][e], float(layer["gu_ts"][e]),
                                  layer["x"][t:t + 1], 32, 32)
        assert np.array_equal(parts["g"][t, 0], gu[0, :16])
        assert np.array_equal(parts["u"][t, 0], gu[0, 16:])
        d, _ = oracle.nvfp4_gemv_f64x(layer["dn_codes"][e], layer["dn_scales"][e], float(layer["dn_ts"][e]),
                                      parts["h"][t, 0][None], 32, 16)
        assert np.array_equal(y[t], d[0])
