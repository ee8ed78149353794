"""Independent decoders for pinning the oracle: published tables and library
conversions only (numpy float16, torch float8_e4m3fn and bfloat16)."""
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))


def e2m1_table() -> np.ndarray:
    vals = np.zeros(16)
    with open(os.path.join(_HERE, "golden", "e2m1_table.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                c, v = line.split()
                vals[int(c)] = float(v)
    return vals


def e4m3_lib(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_lib(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def fp16_lib(h: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(h, dtype=np.uint16).view(np.float16).astype(np.float64)


def nvfp4_codes_unpacked(codes: np.ndarray) -> np.ndarray:
    """[M][K/2] bytes -> [M][K] nibbles, low nibble first (the storage rule)."""
    lo = codes & 0x0F
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def nvfp4_weight_lib(codes, scales, ts) -> np.ndarray:
    """Real-valued NVFP4 weight (fp64) from library/table decoders."""
    c = nvfp4_codes_unpacked(codes)
    s = np.repeat(e4m3_lib(scales), 16, axis=1)
    return e2m1_table()[c] * s * float(np.float32(ts))


def q8_0_weight_lib(q, d) -> np.ndarray:
    return q.astype(np.float64) * np.repeat(fp16_lib(d), 32, axis=1)


def q4_0_codes_unpacked(codes: np.ndarray) -> np.ndarray:
    """[M][K/2] bytes -> [M][K] 4-bit codes in the GGUF Q4_0 block order: the
    16 low nibbles of a block's bytes are its elements 0..15, the 16 high
    nibbles its elements 16..31."""
    M = codes.shape[0]
    b = codes.reshape(M, -1, 16)
    return np.concatenate([b & 0x0F, b >> 4], axis=-1).reshape(M, -1)


def q4_0_weight_lib(codes, d) -> np.ndarray:
    return (q4_0_codes_unpacked(codes).astype(np.float64) - 8.0) * np.repeat(fp16_lib(d), 32, axis=1)


def fp8_b128_weight_lib(codes, scales) -> np.ndarray:
    """Real-valued FP8 block-128 weight: torch's E4M3 decode of every code
    times its tile's fp32 scale, the tile grid spread by numpy repeat."""
    M, K = codes.shape
    s = np.repeat(np.repeat(np.asarray(scales, dtype=np.float32).astype(np.float64), 128, axis=0), 128, axis=1)
    return e4m3_lib(codes) * s[:M, :K]


def q4_1_weight_lib(codes, dm) -> np.ndarray:
    """Real-valued Q4_1 weight: numpy's fp16 decode of (d, m), codes unpacked
    in the Q4_0 block order."""
    f = fp16_lib(dm)  # [M][K/32][2]
    return (q4_0_codes_unpacked(codes).astype(np.float64) * np.repeat(f[..., 0], 32, axis=1)
            + np.repeat(f[..., 1], 32, axis=1))
