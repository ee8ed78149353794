"""Pins of the oracle's element decoders against published tables and library
conversions (never against a retyped copy of the oracle's own formulas)."""
import math

import numpy as np
import torch

import oracle


def test_e2m1_all_codes_match_ocp_table(golden):
    table = golden("e2m1_table.txt")
    rows = [r for k, v in table.items() for r in ([[k] + x for x in v])]
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, val = int(code_s), float(val_s)
        got = oracle.e2m1(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)


def test_e4m3_all_codes_match_torch_float8():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        got = oracle.e4m3(b)
        if math.isnan(ref[b]):
            assert math.isnan(got), b
        else:
            assert got == ref[b] and math.copysign(1, got) == math.copysign(1, ref[b]), (b, got, ref[b])


def test_e4m3_spot_values_from_ofp8_table(golden):
    spot = golden("e4m3_spot.txt")
    n = 0
    for k, vals in spot.items():
        for v in vals:
            b, want = int(k, 16), float(v[0])
            got = oracle.e4m3(b)
            if math.isnan(want):
                assert math.isnan(got)
            else:
                assert got == want and math.copysign(1, got) == math.copysign(1, want)
            n += 1
    assert n == 13
    # exactly two NaN codes and no infinities
    vals = [oracle.e4m3(b) for b in range(256)]
    assert sum(math.isnan(v) for v in vals) == 2
    assert not any(math.isinf(v) for v in vals)


def test_fp16_all_codes_match_numpy():
    ref = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    lib = oracle.lib()
    got = np.array([lib.oracle_fp16(h) for h in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_all_codes_match_torch():
    ref = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    lib = oracle.lib()
    got = np.array([lib.oracle_bf16(h) for h in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
