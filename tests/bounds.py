"""Error bounds of the routed MoE layer, propagated from the GEMV tolerance.

The method states one tolerance, for a GEMV: |y - y_exact| <= 1e-3 * A + 1e-6
per output, A = sum_k |w_k x_k| ("robertbfuentes7-cloud/bw24" README, NVFP4
(W4) decode path, with the workload's accuracy rule). The MoE layer chains
two GEMVs through h = SiLU(g) * u and a weighted combine, so its bound is
that tolerance carried through each step:

  gate_up   |g~ - g| <= tg = 1e-3 * ag + 1e-6,  |u~ - u| <= tu = 1e-3 * au + 1e-6
  SiLU * up |h~ - h| <= dh = L * tg * (|u| + tu) + |SiLU(g)| * tu
                            + 2^-20 * (|h| + those two terms)
            with L = 1.1 >= sup |SiLU'| (1.0998 at g = 2.40) and 2^-20 for
            the fp32 evaluation of g / (1 + exp(-g)) * u (a few ulps).
  down      |d~ - W_dn h| <= |d~ - W_dn h~| + |W_dn| . dh
                          <= 1e-3 * (ad + |W_dn| . dh) + 1e-6 + |W_dn| . dh
  combine   y~ = sum_s w~_s d~_s in fp32, the slots in order, with
            |w~_s - w_s| <= 1e-6 * w_s + 1e-7 (the router's checked bound):
            |y~ - y| <= sum_s [ w_s * tol_d_s + (1e-6 w_s + 1e-7) (|d_s| + tol_d_s) ]
                        + k * 2^-24 * sum_s (w_s + ..) (|d_s| + tol_d_s) + 1e-6

Every quantity on the right comes from the oracle (g, u, h, ag, au, d, ad)
and from |W_dn| . dh, the oracle's GEMV over the magnitude planes (sign bits
cleared). Nothing is taken from the GPU, so the bound serves any path.
"""
import numpy as np

import oracle

SILU_LIP = 1.1  # sup over g of |d/dg (g * sigmoid(g))| = 1.0998...
EVAL_REL = 2.0 ** -20  # fp32 SiLU(g) * u evaluation (exp, divide, multiply)
GEMV_REL, GEMV_ABS = 1e-3, 1e-6  # the method's GEMV tolerance
ROUTE_REL, ROUTE_ABS = 1e-6, 1e-7  # routing weight tolerance checked on the router


def abs_planes(codes, scales):
    """Planes of |w|: E2M1 sign bits (bit 3 of each nibble) and E4M3 sign bits cleared."""
    return codes & 0x77, scales & 0x7F


def silu_up_spread(g, u, h, ag, au):
    """Bound dh on |h~ - h| for h = SiLU(g) * u from the gate_up GEMV bounds."""
    tg = GEMV_REL * ag + GEMV_ABS
    tu = GEMV_REL * au + GEMV_ABS
    silu = g / (1.0 + np.exp(-g))
    base = SILU_LIP * tg * (np.abs(u) + tu) + np.abs(silu) * tu
    return base + EVAL_REL * (np.abs(h) + base)


def moe_y_tolerance(layer, sel, wts, parts):
    """Per-output bound [T][H] on |y~ - y_oracle| of a routed MoE layer.

    layer: synthetic.moe_layer dict; sel, wts: the oracle's routing; parts:
    oracle.moe_layer(..., want_parts=True)'s stage values.
    """
    T, H, I, topk = layer["T"], layer["H"], layer["I"], layer["topk"]
    tol = np.full((T, H), GEMV_ABS)
    mag = np.zeros((T, H))  # sum_s (w_s + route error) * (|d_s| + tol_d_s), for the combine's rounding
    for t in range(T):
        for s in range(topk):
            e = int(sel[t, s])
            dh = silu_up_spread(parts["g"][t, s], parts["u"][t, s], parts["h"][t, s], parts["ag"][t, s],
                                parts["au"][t, s])
            ac, asc = abs_planes(layer["dn_codes"][e], layer["dn_scales"][e])
            spread, _ = oracle.nvfp4_gemv_f64x(ac, asc, abs(float(layer["dn_ts"][e])), dh, H, I)
            spread = spread[0]
            tol_d = GEMV_REL * (parts["ad"][t, s] + spread) + GEMV_ABS + spread
            dw = ROUTE_REL * wts[t, s] + ROUTE_ABS
            dabs = np.abs(parts["d"][t, s]) + tol_d
            tol[t] += wts[t, s] * tol_d + dw * dabs
            mag[t] += (wts[t, s] + dw) * dabs
    return tol + topk * 2.0 ** -24 * mag


def moe_check(y, layer, sel, wts, parts, yref, what=""):
    """Assert |y - yref| <= moe_y_tolerance elementwise."""
    tol = moe_y_tolerance(layer, sel, wts, parts)
    err = np.abs(np.asarray(y, dtype=np.float64).reshape(yref.shape) - yref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside the MoE bound; first {i.tolist()} "
                             f"err {err.ravel()[i].tolist()} tol {tol.ravel()[i].tolist()}")
