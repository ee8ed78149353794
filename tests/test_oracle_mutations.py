"""The pins pin something: each plausible mistake below is planted in a copy
of the oracle's C source, built into a temporary directory on the CPU, and
the committed pin tests named beside it must reject the mutant. Every
mutant keeps all memory accesses in bounds on the inputs its pins use."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle import build as obuild
from tests import test_oracle_decoders as t_dec
from tests import test_oracle_encoders as t_enc
from tests import test_oracle_fp8_b128 as t_fp8
from tests import test_oracle_gemv as t_gemv
from tests import test_oracle_moe as t_moe
from tests import test_oracle_q4_0 as t_q40
from tests import test_oracle_q4_1 as t_q41
from tests.conftest import read_golden

# (mistake, text in oracle.c, its replacement, pins that must catch it)
MUTANTS = [
    ("E2M1 subnormal read as m instead of 0.5 m",
     "mag = 0.5 * m;",
     "mag = 1.0 * m;",
     [lambda: t_dec.test_e2m1_all_codes_match_ocp_table(read_golden)]),
    ("fp16 exponent bias 14 instead of 15",
     "mag = ldexp(1.0 + f / 1024.0, e - 15);",
     "mag = ldexp(1.0 + f / 1024.0, e - 14);",
     [lambda: t_dec.test_fp16_all_codes_match_numpy(),
      lambda: t_q40.test_q4_0_worked_example(read_golden)]),
    ("NVFP4 block scale per 32 k instead of 16",
     "scales[m * (K / 16) + k / 16]",
     "scales[m * (K / 16) + k / 32]",
     [lambda: t_gemv.test_nvfp4_worked_example(read_golden),
      lambda: t_gemv.test_nvfp4_dequant_matches_library_decoders()]),
    ("GEMV magnitude sum without the absolute value",
     "abs_sum += fabs(p);",
     "abs_sum += p;",
     [lambda: t_q40.test_q4_0_worked_example(read_golden),
      lambda: t_fp8.test_fp8_b128_worked_example(read_golden)]),
    ("MoE gate and up halves swapped",
     "double pg = nvfp4_elem(gc, gs, H, i, k) * (double)gu_ts[e] * xv;\n"
     "                    double pu = nvfp4_elem(gc, gs, H, I + i, k) * (double)gu_ts[e] * xv;",
     "double pg = nvfp4_elem(gc, gs, H, I + i, k) * (double)gu_ts[e] * xv;\n"
     "                    double pu = nvfp4_elem(gc, gs, H, i, k) * (double)gu_ts[e] * xv;",
     [lambda: t_moe.test_moe_layer_matches_library_bruteforce(3, 4)]),
    ("NVFP4 nibble order swapped",
     "(k % 2 == 0) ? (uint8_t)(byte & 0x0F) : (uint8_t)(byte >> 4)",
     "(k % 2 == 0) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0x0F)",
     [lambda: t_gemv.test_nvfp4_worked_example(read_golden)]),
    ("E4M3 exponent bias 8 instead of 7",
     "mag = ldexp(1.0 + m / 8.0, e - 7);",
     "mag = ldexp(1.0 + m / 8.0, e - 8);",
     [lambda: t_fp8.test_fp8_b128_every_code_is_torchs_e4m3(),
      lambda: t_fp8.test_fp8_b128_worked_example(read_golden)]),
    ("FP8 tile scale indexed (k tile, m tile)",
     "scales[(m / 128) * kb + k / 128]",
     "scales[(k / 128) * kb + m / 128]",
     [lambda: t_fp8.test_fp8_b128_worked_example(read_golden)]),
    ("Q4_0 / Q4_1 block nibble order as NVFP4's",
     "return j < 16 ? (byte & 0x0F) : (byte >> 4);",
     "return (j % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
     [lambda: t_q40.test_q4_0_worked_example(read_golden),
      lambda: t_q41.test_q4_1_worked_example(read_golden)]),
    ("Q4_1 minimum subtracted",
     "(double)q4_0_code(codes, K, m, k) + oracle_fp16(f[1])",
     "(double)q4_0_code(codes, K, m, k) - oracle_fp16(f[1])",
     [lambda: t_q41.test_q4_1_worked_example(read_golden)]),
    ("Q4_0 code offset 7 instead of 8",
     "(double)(q4_0_code(codes, K, m, k) - 8)",
     "(double)(q4_0_code(codes, K, m, k) - 7)",
     [lambda: t_q40.test_q4_0_worked_example(read_golden)]),
    ("routing ties to the higher expert index",
     "if (best < 0 || l[e] > l[best])",
     "if (best < 0 || l[e] >= l[best])",
     [lambda: t_moe.test_route_ties_and_full_selection()]),
    ("routing weights not renormalised over the selected experts",
     "sel_weight[t * topk + s] /= psum;",
     "sel_weight[t * topk + s] /= 1.0;",
     [lambda: t_moe.test_route_worked_example(read_golden),
      lambda: t_moe.test_route_matches_library_softmax()]),
    ("SiLU with the wrong sign in the exponent",
     "h[i] = sg / (1.0 + exp(-sg)) * su;",
     "h[i] = sg / (1.0 + exp(sg)) * su;",
     [lambda: t_moe.test_moe_layer_matches_library_bruteforce(3, 4)]),
]


def _build_mutant(tmp_path, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) >= 1, f"mutation target not found: {old}"
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-o",
                    str(lib), str(path), "-lm"], check=True)
    return str(lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("mistake,old,new,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(tmp_path, monkeypatch, mistake, old, new, pins):
    lib = _build_mutant(tmp_path, old, new)
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(obuild, "build", lambda *a, **k: lib)
    caught = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught == len(pins), f"{mistake}: {len(pins) - caught} of {len(pins)} pins passed the mutant"


def test_real_oracle_passes_the_same_pins():
    # the unmutated oracle passes every pin used above
    for _, _, _, pins in MUTANTS:
        for pin in pins:
            pin()


def test_encoder_pins_reject_ties_away_from_zero(monkeypatch):
    # the encoders' grid rounding planted with ties to the larger value
    # (away from zero) instead of ties to even
    real = oracle._rn_grid

    def ties_away(v, grid):
        a = np.abs(np.asarray(v, dtype=np.float64))
        g = np.asarray(grid, dtype=np.float64)
        d = np.abs(a[..., None] - g)
        cand = d == d.min(axis=-1, keepdims=True)
        idx = len(g) - 1 - np.argmax(cand[..., ::-1], axis=-1)  # the highest index at the minimum distance
        return np.where(a >= g[-1], len(g) - 1, idx)

    monkeypatch.setattr(oracle, "_rn_grid", ties_away)
    for pin in (t_enc.test_e4m3_encode_matches_torch_cast_in_range,
                t_enc.test_e2m1_encode_grid_midpoints_saturation_and_sign):
        with pytest.raises(AssertionError):
            pin()
    monkeypatch.setattr(oracle, "_rn_grid", real)
    t_enc.test_e4m3_encode_matches_torch_cast_in_range()
    t_enc.test_e2m1_encode_grid_midpoints_saturation_and_sign()
