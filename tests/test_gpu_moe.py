"""MoE router, expert-major list and grouped layer on the GPU against the
oracle. Routing must match exactly; values within tolerances propagated
from the GEMV tolerance through SiLU(gate) * up and the down projection."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_decode_nvfp4_gb300 as bqd
from block_quantized_decode_nvfp4_gb300 import synthetic as syn
from tests.bounds import abs_planes, moe_check, silu_up_spread
from tests import pins
from tests.gpu_util import assert_within, dev, need_gpu

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def route(logits, topk):
    T, E = logits.shape
    P = T * topk
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    ptok = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    pw = torch.full((P,), float("nan"), dtype=torch.float32, device="cuda")
    pslot = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    bqd.moe_route_topk(dev(logits), T, E, topk, off, ptok, pw, pslot)
    return off, ptok, pw, pslot


def check_route(logits, topk):
    T, E = logits.shape
    off, ptok, pw, pslot = [t.cpu().numpy() for t in route(logits, topk)]
    sel, wref = oracle.moe_route(logits, topk)
    assert off[0] == 0 and off[E] == T * topk and np.all(np.diff(off) >= 0)
    got_e = np.full((T, topk), -1)
    got_w = np.zeros((T, topk))
    for e in range(E):
        toks = ptok[off[e]:off[e + 1]]
        assert np.all(np.diff(toks) > 0), "tokens ascending inside an expert"
        for p in range(off[e], off[e + 1]):
            assert got_e[ptok[p], pslot[p]] == -1
            got_e[ptok[p], pslot[p]] = e
            got_w[ptok[p], pslot[p]] = pw[p]
    assert np.array_equal(got_e, sel), "selected experts differ from the oracle"
    assert np.all(np.abs(got_w - wref) <= 1e-6 * wref + 1e-7)
    return off, ptok, pw, pslot


@pytest.mark.parametrize("T,E,topk", [(1, 256, 8), (16, 256, 8), (5, 64, 4), (1, 8, 8), (300, 128, 2),
                                      (1024, 1024, 8), (3, 33, 32)])
def test_route_random(T, E, topk):
    check_route(syn.router_logits(T, E, np.random.default_rng(T * E + topk)), topk)


def test_route_ties_and_worked_example(golden):
    g = golden("moe_route_example.txt")
    logits = np.array([[float(v) for v in g["logits"][0]]], dtype=np.float32)
    for k in (3, 2):
        off, ptok, pw, pslot = check_route(logits, k)
    z = np.zeros((4, 40), dtype=np.float32)
    z[1, 7] = 1.0
    check_route(z, 8)  # all ties: lowest indices, equal weights


def _layer_run(L, want_ws=False):
    T, E, H, I, topk = L["T"], L["E"], L["H"], L["I"], L["topk"]
    off, ptok, pw, pslot = route(L["logits"], topk)
    wsb = bqd.moe_workspace_bytes(T, topk, H, I)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    y = torch.full((T * H,), float("nan"), dtype=torch.float32, device="cuda")
    bqd.moe_grouped_gemv(dev(L["gu_codes"]), dev(L["gu_scales"]), dev(L["gu_ts"]), dev(L["dn_codes"]),
                         dev(L["dn_scales"]), dev(L["dn_ts"]), dev(L["x"]), off, ptok, pw, pslot, y, ws, wsb,
                         E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) == 0
    return y.cpu().numpy().reshape(T, H), ws, (off, ptok, pw, pslot)


def _ws_h(ws, T, topk, I):
    P = T * topk
    a256 = lambda n: (n + 255) // 256 * 256
    start = 256 + 2 * a256(4 * P)
    return ws[start:start + 4 * P * I].view(torch.float32).cpu().numpy().reshape(P, I)


@pytest.mark.parametrize("T", [1, 16])
def test_moe_layer_full_size(T):
    L = syn.moe_layer(T=T, seed=0)
    topk, H, I = L["topk"], L["H"], L["I"]
    y, ws, (off, ptok, pw, pslot) = _layer_run(L)
    sel, wref = oracle.moe_route(L["logits"], topk)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=wref, want_parts=True)
    off, ptok, pslot = off.cpu().numpy(), ptok.cpu().numpy(), pslot.cpu().numpy()
    h_gpu = _ws_h(ws, T, topk, I)

    tol_y = np.full((T, H), 1e-6)
    for p in range(T * topk):
        t, s = ptok[p], pslot[p]
        e = sel[t, s]
        h = parts["h"][t, s]
        dh = silu_up_spread(parts["g"][t, s], parts["u"][t, s], h, parts["ag"][t, s], parts["au"][t, s]) + 1e-30
        # stage 1: h = SiLU(gate) * up within the propagated GEMV tolerance
        assert np.all(np.abs(h_gpu[p] - h) <= dh), f"h of pair {p}"
        # stage 2: down projection of the GPU's own h within the GEMV tolerance
        dc, dsc = L["dn_codes"][e], L["dn_scales"][e]
        d_gpu_h, a_gpu_h = oracle.nvfp4_gemv_f64x(dc, dsc, float(L["dn_ts"][e]), h_gpu[p].astype(np.float64), H, I)
        ac, asc = abs_planes(dc, dsc)
        spread, _ = oracle.nvfp4_gemv_f64x(ac, asc, abs(float(L["dn_ts"][e])), dh, H, I)  # |W_dn| . dh
        tol_y[t] += wref[t, s] * (spread[0] + 1e-3 * a_gpu_h[0] + 1e-6 + 1e-6 * np.abs(d_gpu_h[0]))
    assert_within(y, yref, tol_y, f"MoE y T={T}", rel=1.0, absol=0.0)
    # end to end, from the oracle's stage values alone
    moe_check(y, L, sel, wref, parts, yref, f"MoE y T={T} (propagated bound)")


# I = 128 takes the register-streaming kernels, I = 256 the bulk-copy ones
@pytest.mark.parametrize("I", [128, 256])
def test_moe_deterministic_and_identical_experts(I):
    L = syn.moe_layer(T=4, E=32, H=512, I=I, topk=4, seed=3)
    y1, _, _ = _layer_run(L)
    y2, _, _ = _layer_run(L)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    # identical experts: routing cannot matter, y equals one dense FFN
    for k in ("gu_codes", "gu_scales", "dn_codes", "dn_scales"):
        L[k] = np.ascontiguousarray(np.broadcast_to(L[k][0], L[k].shape))
    y, _, _ = _layer_run(L)
    sel, w = oracle.moe_route(L["logits"], 4)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=w, want_parts=True)
    moe_check(y, L, sel, w, parts, yref, "identical experts")


@pytest.mark.parametrize("I", [64, 256])
def test_moe_small_shapes_and_many_tokens_per_expert(I):
    # few experts, many tokens: token groups of 8 and more per expert
    L = syn.moe_layer(T=40, E=4, H=256, I=I, topk=2, seed=4)
    y, _, _ = _layer_run(L)
    sel, w = oracle.moe_route(L["logits"], 2)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=w, want_parts=True)
    moe_check(y, L, sel, w, parts, yref, f"T=40 E=4 I={I}")


@pytest.mark.parametrize("H,I", [(128, 64), (256, 256)])
def test_moe_malformed_list_sets_status_without_faulting(H, I):
    L = syn.moe_layer(T=2, E=8, H=H, I=I, topk=2, seed=5)
    T, E, topk = 2, 8, 2
    off, ptok, pw, pslot = route(L["logits"], topk)
    wsb = bqd.moe_workspace_bytes(T, topk, H, I)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    y = torch.zeros(T * H, dtype=torch.float32, device="cuda")
    args = [dev(L[k]) for k in ("gu_codes", "gu_scales", "gu_ts", "dn_codes", "dn_scales", "dn_ts", "x")]
    bad_off = off.clone()
    bad_off[E] = T * topk + 3  # does not close the CSR
    bqd.moe_grouped_gemv(*args, bad_off, ptok, pw, pslot, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) & 1
    bad_tok = ptok.clone()
    bad_tok[0] = 99  # token id out of range
    bqd.moe_grouped_gemv(*args, off, bad_tok, pw, pslot, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) & 2
    dup = pslot.clone()
    dup[:] = 0  # every pair claims slot 0: slot 1 of each token is never produced
    bqd.moe_grouped_gemv(*args, off, ptok, pw, dup, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) & 4
    # a valid call afterwards clears the status
    bqd.moe_grouped_gemv(*args, off, ptok, pw, pslot, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) == 0


# ---------------------------------------------------------------- moe_layer and the small-batch path
def _layer_fused(L):
    T, E, H, I, topk = L["T"], L["E"], L["H"], L["I"], L["topk"]
    wsb = bqd.moe_layer_workspace_bytes(T, topk, H, I, E)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    y = torch.full((T * H,), float("nan"), dtype=torch.float32, device="cuda")
    bqd.moe_layer(dev(L["logits"]), dev(L["gu_codes"]), dev(L["gu_scales"]), dev(L["gu_ts"]), dev(L["dn_codes"]),
                  dev(L["dn_scales"]), dev(L["dn_ts"]), dev(L["x"]), y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) == 0
    return y.cpu().numpy().reshape(T, H), ws


# (T, E, H, I, topk): all but the last two take the batched kernels (T <= 16,
# T * topk <= 128, T * H <= 32768, H >= 2I, I in {256, 512, 1024}); the last
# two the route kernel and the expert streams
SMALL_AND_LARGE = [(1, 64, 1024, 256, 8), (2, 16, 1024, 512, 4), (3, 64, 2048, 256, 8), (4, 32, 2048, 1024, 8),
                   (4, 256, 2048, 512, 8), (5, 64, 1024, 256, 8), (16, 64, 1024, 256, 8), (11, 32, 2048, 512, 8),
                   (16, 256, 2048, 512, 8), (24, 64, 1024, 256, 4), (16, 64, 4096, 512, 8)]


@pytest.mark.parametrize("T,E,H,I,topk", SMALL_AND_LARGE)
def test_moe_layer_matches_route_then_grouped_and_oracle(T, E, H, I, topk):
    L = syn.moe_layer(T=T, E=E, H=H, I=I, topk=topk, seed=T * 131 + E + I)
    y_fused, ws = _layer_fused(L)
    y_two, ws2, _ = _layer_run(L)
    assert np.array_equal(y_fused.view(np.uint32), y_two.view(np.uint32)), "moe_layer differs from route + grouped"
    # h sits where moe_grouped_gemv documents it, in both workspaces
    assert np.array_equal(_ws_h(ws, T, topk, I), _ws_h(ws2, T, topk, I))
    sel, wts = oracle.moe_route(L["logits"], topk)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=wts, want_parts=True)
    moe_check(y_fused, L, sel, wts, parts, yref, f"moe_layer T={T} E={E} H={H} I={I} k={topk}")
    y3, _ = _layer_fused(L)
    assert np.array_equal(y_fused.view(np.uint32), y3.view(np.uint32)), "not deterministic"


def test_small_path_identical_experts_and_activation_range():
    L = syn.moe_layer(T=4, E=32, H=1024, I=256, topk=4, seed=17)
    for k in ("gu_codes", "gu_scales", "dn_codes", "dn_scales"):
        L[k] = np.ascontiguousarray(np.broadcast_to(L[k][0], L[k].shape))
    y, _, _ = _layer_run(L)
    sel, w = oracle.moe_route(L["logits"], 4)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=w, want_parts=True)
    moe_check(y, L, sel, w, parts, yref, "small path, identical experts")
    # one token with a range wider than f16 holds: the CTA takes the exact fp32 path
    xf = pins.bf16_lib(L["x"]).astype(np.float32)
    xf[2, 5], xf[2, 9] = 2.0 ** 40, 2.0 ** -40
    L["x"] = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y, _, _ = _layer_run(L)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=w, want_parts=True)
    moe_check(y, L, sel, w, parts, yref, "small path, wide-range token")


def test_small_path_malformed_list_sets_status_without_faulting():
    T, E, H, I, topk = 2, 8, 1024, 256, 2
    L = syn.moe_layer(T=T, E=E, H=H, I=I, topk=topk, seed=55)
    off, ptok, pw, pslot = route(L["logits"], topk)
    wsb = bqd.moe_workspace_bytes(T, topk, H, I)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    y = torch.zeros(T * H, dtype=torch.float32, device="cuda")
    args = [dev(L[k]) for k in ("gu_codes", "gu_scales", "gu_ts", "dn_codes", "dn_scales", "dn_ts", "x")]
    bad_off = off.clone()
    bad_off[E] = T * topk + 3
    bqd.moe_grouped_gemv(*args, bad_off, ptok, pw, pslot, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) & 1
    bad_tok = ptok.clone()
    bad_tok[0] = 99
    bqd.moe_grouped_gemv(*args, off, bad_tok, pw, pslot, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) & 2
    dup = pslot.clone()
    dup[:] = 0
    bqd.moe_grouped_gemv(*args, off, ptok, pw, dup, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) & 4
    bqd.moe_grouped_gemv(*args, off, ptok, pw, pslot, y, ws, wsb, E, H, I, T, topk)
    assert bqd.bqd_moe_read_status(ws) == 0
    sel, w = oracle.moe_route(L["logits"], topk)
    yref, parts = oracle.moe_layer(L, sel=sel, weights=w, want_parts=True)
    moe_check(y.cpu().numpy(), L, sel, w, parts, yref, "small path after malformed lists")
