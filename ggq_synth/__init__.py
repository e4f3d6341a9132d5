"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and writes them into the byte fields of the
GGUF block layouts.  It holds none of the method's arithmetic (no dequantize,
no quantizer, no dot): it only decides where each random field goes.  Both the
oracle and the CUDA path receive the same bytes from here.

Distributions follow the workload definitions of the keep-quant GEMV / MoE
path:
  * Q4_0: fp16 d ~ U[1e-3, 1e-2], nibbles uniform in 0..15.
  * Q8_0: fp16 d ~ U[1e-4, 1e-2], int8 quants uniform over all 256 values.
  * Q4_K / Q5_K: fp16 d, dmin ~ U[1e-4, 1e-2]; the 12 packed scale bytes, the
    nibbles and the high bits uniform bytes (so every 6-bit scale and min is
    uniform in 0..63).
  * Q6_K: fp16 d ~ U[1e-4, 1e-2]; low/high quant bits uniform bytes; int8
    sub-scales uniform in [-32, 31] (reading of "6-bit sub-scales uniform").
  * MXFP4: E8M0 exponent byte uniform in 117..123 (scale 2^-10 .. 2^-4),
    E2M1 nibbles uniform over the 16 codes.
  * Q2_K: fp16 d, dmin ~ U[1e-4, 1e-2]; scale/min bytes, 2-bit quants uniform
    bytes (every 4-bit scale and min uniform in 0..15).
  * Q3_K: fp16 d ~ U[1e-4, 1e-2]; high-bit mask, 2-bit quants and the 12
    packed scale bytes uniform bytes (every 6-bit scale uniform in 0..63).
  * Activations and router logits ~ N(0, 1) fp32; the prefill workload adds a
    Zipf(1.1) expert bias -1.1*ln(rank) over a seeded permutation of ranks.
"""
from __future__ import annotations

import numpy as np

BLOCK_ELEMS = {"Q4_0": 32, "Q8_0": 32, "MXFP4": 32, "Q8_1": 32, "Q4_K": 256, "Q5_K": 256, "Q6_K": 256, "Q8_K": 256,
               "Q2_K": 256, "Q3_K": 256}
BLOCK_BYTES = {"Q4_0": 18, "Q8_0": 34, "MXFP4": 17, "Q8_1": 36, "Q4_K": 144, "Q5_K": 176, "Q6_K": 210, "Q8_K": 292,
               "Q2_K": 84, "Q3_K": 110}
WEIGHT_FORMATS = ("Q4_0", "Q8_0", "Q4_K", "Q5_K", "Q6_K", "MXFP4", "Q2_K", "Q3_K")

BASE_SEED = 0x6767


def rng(config_index: int, stream: int) -> np.random.Generator:
    """Independent generator per (workload, input stream)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([BASE_SEED + config_index, stream])))


def row_bytes(fmt: str, K: int) -> int:
    if K % BLOCK_ELEMS[fmt]:
        raise ValueError(f"K={K} is not a multiple of the {fmt} block size")
    return K // BLOCK_ELEMS[fmt] * BLOCK_BYTES[fmt]


def _f16_bytes(vals: np.ndarray) -> np.ndarray:
    return vals.astype(np.float16).view(np.uint8).reshape(vals.shape + (2,))


def weights(fmt: str, rows: int, K: int, g: np.random.Generator, d_range=None) -> np.ndarray:
    """Random weight blocks, returned as uint8 [rows, row_bytes]."""
    nb = rows * (K // BLOCK_ELEMS[fmt])
    bb = BLOCK_BYTES[fmt]
    out = np.empty((nb, bb), dtype=np.uint8)
    lo, hi = d_range if d_range is not None else ((1e-3, 1e-2) if fmt == "Q4_0" else (1e-4, 1e-2))
    if fmt == "Q4_0":
        out[:, 0:2] = _f16_bytes(g.uniform(lo, hi, nb).astype(np.float32))
        out[:, 2:18] = g.integers(0, 256, (nb, 16), dtype=np.uint8)
    elif fmt == "Q8_0":
        out[:, 0:2] = _f16_bytes(g.uniform(lo, hi, nb).astype(np.float32))
        out[:, 2:34] = g.integers(0, 256, (nb, 32), dtype=np.uint8)
    elif fmt == "MXFP4":
        out[:, 0] = g.integers(117, 124, nb, dtype=np.uint8)
        out[:, 1:17] = g.integers(0, 256, (nb, 16), dtype=np.uint8)
    elif fmt in ("Q4_K", "Q5_K"):
        out[:, 0:2] = _f16_bytes(g.uniform(lo, hi, nb).astype(np.float32))
        out[:, 2:4] = _f16_bytes(g.uniform(lo, hi, nb).astype(np.float32))
        out[:, 4:bb] = g.integers(0, 256, (nb, bb - 4), dtype=np.uint8)
    elif fmt == "Q6_K":
        out[:, 0:192] = g.integers(0, 256, (nb, 192), dtype=np.uint8)
        out[:, 192:208] = g.integers(-32, 32, (nb, 16), dtype=np.int8).view(np.uint8)
        out[:, 208:210] = _f16_bytes(g.uniform(lo, hi, nb).astype(np.float32))
    elif fmt == "Q2_K":  # scales[16], qs[64], d, dmin
        out[:, 0:80] = g.integers(0, 256, (nb, 80), dtype=np.uint8)
        out[:, 80:82] = _f16_bytes(g.uniform(lo, hi, nb).astype(np.float32))
        out[:, 82:84] = _f16_bytes(g.uniform(lo, hi, nb).astype(np.float32))
    elif fmt == "Q3_K":  # hmask[32], qs[64], scales[12], d
        out[:, 0:108] = g.integers(0, 256, (nb, 108), dtype=np.uint8)
        out[:, 108:110] = _f16_bytes(g.uniform(lo, hi, nb).astype(np.float32))
    else:
        raise ValueError(fmt)
    return out.reshape(rows, (K // BLOCK_ELEMS[fmt]) * bb)


def activations(T: int, K: int, g: np.random.Generator) -> np.ndarray:
    return g.standard_normal((T, K), dtype=np.float32)


def router_logits(T: int, E: int, g: np.random.Generator, zipf_s: float | None = None) -> np.ndarray:
    logits = g.standard_normal((T, E), dtype=np.float32)
    if zipf_s is not None:
        rank = g.permutation(E) + 1  # rank of each expert, 1..E
        bias = (-zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)
        logits = (logits + bias[None, :]).astype(np.float32)
    return logits


def expert_bank(fmt: str, E: int, rows: int, K: int, g: np.random.Generator) -> np.ndarray:
    """[E][rows][row_bytes] bank of expert matrices."""
    return weights(fmt, E * rows, K, g).reshape(E, rows, row_bytes(fmt, K))


# Workload shapes.  Index = position in the workload list; the seed of every
# input of a workload is BASE_SEED + index.
GEMV_Q4_0 = dict(index=0, fmt="Q4_0", N=1024, K=4096, T=(1,))
GEMV_KQUANT = dict(index=1, fmts=("Q8_0", "Q4_K", "Q5_K", "Q6_K"), N=14336, K=4096, T=(1, 2, 4, 8))
MOE_DECODE = dict(index=2, E=128, H=2048, I=768, k=8, gate="Q4_K", up="Q4_K", down="Q6_K", T=(1, 2, 3, 4))
MOE_MXFP4 = dict(index=3, E=256, H=4096, I=2048, k=8, gate="MXFP4", up="MXFP4", down="MXFP4",
                 T=(1, 2, 3, 4, 5, 32, 128, 512))
MOE_PREFILL = dict(index=4, E=128, H=4096, I=1536, k=8, gate="Q8_0", up="Q8_0", down="Q4_K", T=(4096,), zipf=1.1)
