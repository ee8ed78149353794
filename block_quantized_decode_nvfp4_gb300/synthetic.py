"""Seeded synthetic inputs for the block-quantized decode matvec.

This module is shared by the tests, the benchmark and the oracle's callers. It
holds no arithmetic of the method itself: it draws random numbers with numpy's
PCG64 and turns them into the storage formats with library conversions only
(torch's float32 -> float8_e4m3fn and float32 -> bfloat16 casts, numpy's
float64 -> float16 cast; all three round to nearest, ties to even).

Workloads follow the five configurations the method is measured on (weights
of 9B-dense layer shapes, a Q8_0 LM head, speculative-verify widths and a
256-expert MoE layer):

* NVFP4 weight: E2M1 codes uniform over all 16 nibble values, two per byte with
  the low nibble holding the lower k; one E4M3 scale per 16 consecutive k of a
  row, drawn log2-uniform over [2^-6, 2^2] and rounded to E4M3; one FP32
  tensor scale.
* Q8_0 weight: int8 uniform in [-127, 127]; one fp16 scale per 32 consecutive
  k of a row, uniform in [1e-4, 1e-2] and rounded to fp16. Stored planar
  (a q plane and a d plane), not as interleaved 34-byte blocks.
* FP8 block-128 weight: E4M3 codes of N(0, 1) * 112 draws (a tile's
  largest |value| lands near the format's 448, as in checkpoints scaled per
  tile), rounded to E4M3; one fp32 scale per 128 x 128 tile, log2-uniform
  over [2^-14, 2^-8].
* Activations: bf16 ~ N(0, 1). Router logits: fp32 ~ N(0, 1).

Every tensor gets its own child stream of ``numpy.random.SeedSequence(seed)``
in a fixed, documented order, so the bytes depend only on (seed, shapes).
"""

from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "streams",
    "nvfp4_weight",
    "q8_0_weight",
    "q4_0_weight",
    "q4_1_weight",
    "fp8_b128_weight",
    "bf16_normal",
    "router_logits",
    "tiny_nvfp4",
    "dense_nvfp4",
    "dense_q8_0",
    "dense_q4_0",
    "dense_q4_1",
    "dense_fp8_b128",
    "moe_layer",
    "NVFP4_SHAPES",
    "Q8_0_SHAPES",
    "Q4_0_SHAPES",
    "FP8_B128_SHAPES",
    "VERIFY_SHAPES",
]

# (M, K) of the dense NVFP4 weights (gate/up, down, attention out).
NVFP4_SHAPES = [(12288, 4096), (4096, 12288), (4096, 4096)]
# (M, K) of the Q8_0 weights (gate/up, down, LM head).
Q8_0_SHAPES = [(12288, 4096), (4096, 12288), (151936, 4096)]
# (M, K) of the Q4_0 weights (gate/up, down).
Q4_0_SHAPES = [(12288, 4096), (4096, 12288)]
# (M, K) of the FP8 block-128 weights (gate/up, down).
FP8_B128_SHAPES = [(12288, 4096), (4096, 12288)]
# (M, K) of the speculative-verify weights; N in {4, 8}.
VERIFY_SHAPES = [(4096, 4096), (12288, 4096)]


def streams(seed: int, n: int) -> list[np.random.Generator]:
    """n independent PCG64 generators, child i of SeedSequence(seed)."""
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _to_e4m3_bytes(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _to_bf16_bits(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def nvfp4_weight(M: int, K: int, ts: float, rng_codes, rng_scales) -> dict:
    """NVFP4 planes: codes u8[M][K/2], scales u8[M][K/16], tensor scale ts."""
    if K % 16:
        raise ValueError("NVFP4 needs K % 16 == 0")
    codes = rng_codes.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    log2s = rng_scales.uniform(-6.0, 2.0, size=(M, K // 16))
    scales = _to_e4m3_bytes(np.exp2(log2s))
    return {"codes": codes, "scales": scales, "ts": float(np.float32(ts)), "M": M, "K": K}


def q8_0_weight(M: int, K: int, rng_q, rng_d) -> dict:
    """Q8_0 planes: q i8[M][K], d fp16 bits u16[M][K/32]."""
    if K % 32:
        raise ValueError("Q8_0 needs K % 32 == 0")
    q = rng_q.integers(-127, 128, size=(M, K), dtype=np.int8)
    d = rng_d.uniform(1e-4, 1e-2, size=(M, K // 32)).astype(np.float16).view(np.uint16)
    return {"q": q, "d": d, "M": M, "K": K}


def q4_0_weight(M: int, K: int, rng_c, rng_d) -> dict:
    """Q4_0 planes: codes u8[M][K/2] (16 bytes per 32-element block, uniform
    over all bytes), d fp16 bits u16[M][K/32]."""
    if K % 32:
        raise ValueError("Q4_0 needs K % 32 == 0")
    codes = rng_c.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    d = rng_d.uniform(1e-3, 1e-1, size=(M, K // 32)).astype(np.float16).view(np.uint16)
    return {"codes": codes, "d": d, "M": M, "K": K}


def q4_1_weight(M: int, K: int, rng_c, rng_d) -> dict:
    """Q4_1 planes: codes u8[M][K/2] (the Q4_0 block order, uniform over all
    bytes), dm fp16 bits u16[M][K/32][2]: d uniform in [1e-3, 1e-1], m
    uniform in [-1, 1] (a block's minimum, as encoders store it)."""
    if K % 32:
        raise ValueError("Q4_1 needs K % 32 == 0")
    codes = rng_c.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    d = rng_d.uniform(1e-3, 1e-1, size=(M, K // 32))
    m = rng_d.uniform(-1.0, 1.0, size=(M, K // 32))
    dm = np.stack([d, m], axis=-1).astype(np.float16).view(np.uint16)
    return {"codes": codes, "dm": np.ascontiguousarray(dm), "M": M, "K": K}


def fp8_b128_weight(M: int, K: int, rng_c, rng_s) -> dict:
    """FP8 block-128 planes: codes u8[M][K] (E4M3 bytes, row-major), scales
    f32[ceil(M/128)][ceil(K/128)]."""
    codes = _to_e4m3_bytes(np.clip(rng_c.standard_normal(size=(M, K), dtype=np.float32) * 112.0, -448.0, 448.0))
    log2s = rng_s.uniform(-14.0, -8.0, size=((M + 127) // 128, (K + 127) // 128))
    scales = np.exp2(log2s).astype(np.float32)
    return {"codes": codes, "scales": scales, "M": M, "K": K}


def bf16_normal(shape, rng) -> np.ndarray:
    """bf16 bits of N(0,1) draws (fp32 draw, then round-to-nearest-even)."""
    return _to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def router_logits(T: int, E: int, rng) -> np.ndarray:
    return rng.standard_normal(size=(T, E), dtype=np.float32)


# ---------------------------------------------------------------- workloads

def tiny_nvfp4(seed: int = 0, M: int = 256, K: int = 512, N: int = 1, ts: float = 1.0) -> dict:
    """Tiny NVFP4 GEMV (256 x 512, N = 1, ts = 1). Streams: codes, scales, x."""
    rc, rs, rx = streams(seed, 3)
    w = nvfp4_weight(M, K, ts, rc, rs)
    w["x"] = bf16_normal((N, K), rx)
    return w


def dense_nvfp4(M: int, K: int, N: int = 1, seed: int = 0, ts: float = 0.01) -> dict:
    """NVFP4 weight of a dense layer (ts = 0.01) with N bf16 columns.

    Streams of SeedSequence(seed): 0 codes, 1 scales, 2 x.
    """
    rc, rs, rx = streams(seed, 3)
    w = nvfp4_weight(M, K, ts, rc, rs)
    w["x"] = bf16_normal((N, K), rx)
    return w


def dense_q8_0(M: int, K: int, N: int = 1, seed: int = 0) -> dict:
    """Q8_0 weight with N bf16 columns. Streams: 0 q, 1 d, 2 x."""
    rq, rd, rx = streams(seed, 3)
    w = q8_0_weight(M, K, rq, rd)
    w["x"] = bf16_normal((N, K), rx)
    return w


def dense_q4_0(M: int, K: int, N: int = 1, seed: int = 0) -> dict:
    """Q4_0 weight with N bf16 columns. Streams: 0 codes, 1 d, 2 x."""
    rc, rd, rx = streams(seed, 3)
    w = q4_0_weight(M, K, rc, rd)
    w["x"] = bf16_normal((N, K), rx)
    return w


def dense_q4_1(M: int, K: int, N: int = 1, seed: int = 0) -> dict:
    """Q4_1 weight with N bf16 columns. Streams: 0 codes, 1 dm, 2 x."""
    rc, rd, rx = streams(seed, 3)
    w = q4_1_weight(M, K, rc, rd)
    w["x"] = bf16_normal((N, K), rx)
    return w


def dense_fp8_b128(M: int, K: int, N: int = 1, seed: int = 0) -> dict:
    """FP8 block-128 weight with N bf16 columns. Streams: 0 codes, 1 scales, 2 x."""
    rc, rs, rx = streams(seed, 3)
    w = fp8_b128_weight(M, K, rc, rs)
    w["x"] = bf16_normal((N, K), rx)
    return w


def moe_layer(T: int, E: int = 256, H: int = 2048, I: int = 512, topk: int = 8,
              seed: int = 0, ts: float = 0.01) -> dict:
    """MoE layer: per-expert NVFP4 gate_up [E][2I][H] and down [E][H][I].

    Rows 0..I-1 of gate_up are the gate projection, rows I..2I-1 the up
    projection. Streams of SeedSequence(seed): 0 gate_up codes, 1 gate_up
    scales, 2 down codes, 3 down scales, 4 x, 5 router logits.
    """
    r = streams(seed, 6)
    gu = nvfp4_weight(E * 2 * I, H, ts, r[0], r[1])
    dn = nvfp4_weight(E * H, I, ts, r[2], r[3])
    return {
        "E": E, "H": H, "I": I, "T": T, "topk": topk,
        "gu_codes": gu["codes"].reshape(E, 2 * I, H // 2),
        "gu_scales": gu["scales"].reshape(E, 2 * I, H // 16),
        "gu_ts": np.full(E, np.float32(ts), dtype=np.float32),
        "dn_codes": dn["codes"].reshape(E, H, I // 2),
        "dn_scales": dn["scales"].reshape(E, H, I // 16),
        "dn_ts": np.full(E, np.float32(ts), dtype=np.float32),
        "x": bf16_normal((T, H), r[4]),
        "logits": router_logits(T, E, r[5]),
    }
