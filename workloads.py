"""Seeded synthetic inputs for the affine group-64 quantized matmul.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It draws random codes, scales, biases and activations with the
shapes and value distributions of the workloads below, and converts floats to
and from the 16-bit storage types.  It holds none of the method's arithmetic:
no packing, no unpacking, no dequantisation and no matmul.  Each side packs
the integer codes with its own packer.

Workloads (all group size 64; "N(0,s)" means a normal draw with standard
deviation s):

=========  =====  ======================================  ====================
name       bits   N x K, rows M                           x dtype
=========  =====  ======================================  ====================
small      4      1024 x 512, M=1                         fp16
decode     4      4096 x 4096, M=1                        bf16
split3     3      10240 x 5120, M in {1,9,16,32,64}       fp16
layer      4      seven projections of a 5120-hidden      bf16
                  decoder layer (q,k,v,o,gate,up,down), M=1
prefill    4      28672 x 8192, M in {128,512,256}        bf16
=========  =====  ======================================  ====================

Codes are uniform over [0, 2^bits).  Scales are |N(0,1)|*c + 1e-3 with
c = 0.01 (4-bit) or 0.02 (3-bit), rounded to fp16; biases are
-2^(bits-1)*scale + N(0,1e-3), rounded to fp16, so each weight is centred on
zero.  Activations are N(0,1), rounded to the x dtype.  The 3-bit
10240 x 5120 shape is the one the mlx-bun affine split-mma page measures
(kernels/quantization/affine-split-mma.ts header, M1 Max timings at 9/16/32/64
rows); the layer shapes stand in for a 5120-hidden decoder layer with 40 x 128
query heads, 8 KV heads and a 13824-wide MLP.  No dataset or trained weight is
involved.

Quantiser inputs (float weights for aq_quantize): N(0, 0.02) with a per-row
spread factor |N(0,1)| + 0.25 (rows of different magnitude, as in trained
projections), rounded to fp16 or bf16; shapes as the workloads above
(QUANTIZE_WORKLOADS).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np

GROUP = 64


@dataclasses.dataclass(frozen=True)
class Problem:
    """One y = x . W^T problem: integer codes plus fp16 scales/biases and x."""

    name: str
    bits: int
    M: int
    N: int
    K: int
    x_dtype: str  # "fp16" or "bf16"
    codes: np.ndarray  # uint8 [N, K], values < 2^bits
    scales: np.ndarray  # float16 [N, K/64]
    biases: np.ndarray  # float16 [N, K/64]
    x_bits: np.ndarray  # uint16 [M, K]: raw fp16 or bf16 bit patterns
    seed: int

    @property
    def G(self) -> int:
        return self.K // GROUP

    def x_f64(self) -> np.ndarray:
        return to_f64(self.x_bits, self.x_dtype)


# ----------------------------------------------------------------------------
# 16-bit float storage conversions (format handling, not method arithmetic)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); return bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_fp16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def to_f64(bits16: np.ndarray, dtype: str) -> np.ndarray:
    """Exact conversion of fp16 / bf16 bit patterns to float64."""
    if dtype == "fp16":
        return np.ascontiguousarray(bits16, dtype=np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f32(bits16).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def from_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to fp16 / bf16 bit patterns (via float32)."""
    if dtype == "fp16":
        return np.asarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(np.asarray(a, dtype=np.float64).astype(np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


# ----------------------------------------------------------------------------
# Generators
# ----------------------------------------------------------------------------

def make_problem(name: str, bits: int, N: int, K: int, M: int, x_dtype: str,
                 seed: int, scale_mul: float | None = None) -> Problem:
    """Draw one problem.  The draw order is codes, scales, bias noise, x, so
    problems that differ only in M share identical weights."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 64")
    if scale_mul is None:
        scale_mul = 0.01 if bits == 4 else 0.02
    rng = np.random.default_rng(seed)
    G = K // GROUP
    codes = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    scales = (np.abs(rng.standard_normal((N, G))) * scale_mul + 1e-3).astype(np.float16)
    noise = rng.standard_normal((N, G)) * 1e-3
    biases = (-(1 << (bits - 1)) * scales.astype(np.float64) + noise).astype(np.float16)
    xf = rng.standard_normal((M, K)).astype(np.float32)
    x_bits = f32_to_bf16_bits(xf) if x_dtype == "bf16" else f32_to_fp16_bits(xf)
    return Problem(name, bits, M, N, K, x_dtype, codes, scales, biases, x_bits, seed)


def make_x(M: int, K: int, x_dtype: str, seed: int) -> np.ndarray:
    """Activations alone (N(0,1) rounded to x_dtype), for sweeps over M."""
    rng = np.random.default_rng(seed)
    xf = rng.standard_normal((M, K)).astype(np.float32)
    return f32_to_bf16_bits(xf) if x_dtype == "bf16" else f32_to_fp16_bits(xf)


# Projection shapes (N, K) of one 5120-hidden decoder layer.
LAYER_PROJECTIONS: List[Tuple[str, int, int]] = [
    ("q", 5120, 5120),
    ("k", 1024, 5120),
    ("v", 1024, 5120),
    ("o", 5120, 5120),
    ("gate", 13824, 5120),
    ("up", 13824, 5120),
    ("down", 5120, 13824),
]

# name -> list of (bits, N, K, M, x_dtype, seed)
WORKLOADS: Dict[str, List[Tuple[int, int, int, int, str, int]]] = {
    "small": [(4, 1024, 512, 1, "fp16", 0)],
    "decode": [(4, 4096, 4096, 1, "bf16", 1)],
    "split3": [(3, 10240, 5120, m, "fp16", 2) for m in (1, 9, 16, 32, 64)],
    "layer": [(4, n, k, 1, "bf16", 30 + p) for p, (_, n, k) in enumerate(LAYER_PROJECTIONS)],
    "prefill": [(4, 28672, 8192, m, "bf16", 4) for m in (128, 512, 256)],
}


def workload(name: str, index: int = 0) -> Problem:
    bits, N, K, M, dt, seed = WORKLOADS[name][index]
    return make_problem(f"{name}[{index}]", bits, N, K, M, dt, seed)


def algorithmic_bytes(M: int, N: int, K: int, bits: int, out_bytes: int = 2) -> int:
    """Bytes one call must move at least: packed codes, fp16 scales and
    biases, x and y (2-byte elements)."""
    return N * K * bits // 8 + 4 * N * (K // GROUP) + 2 * M * K + out_bytes * M * N


def flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def make_weights(N: int, K: int, dtype: str, seed: int, std: float = 0.02):
    """Float weights for the quantiser: (16-bit patterns uint16 [N, K], the same
    values as float32 [N, K])."""
    rng = np.random.default_rng(seed)
    row = np.abs(rng.standard_normal((N, 1))) + 0.25
    wf = (rng.standard_normal((N, K)) * std * row).astype(np.float32)
    bits = f32_to_bf16_bits(wf) if dtype == "bf16" else f32_to_fp16_bits(wf)
    vals = bf16_bits_to_f32(bits) if dtype == "bf16" else bits.view(np.float16).astype(np.float32)
    return bits, vals


# name -> list of (bits, N, K, w dtype, seed) for the quantiser
QUANTIZE_WORKLOADS: Dict[str, List[Tuple[int, int, int, str, int]]] = {
    "quantize": [(4, 4096, 4096, "bf16", 51), (3, 10240, 5120, "fp16", 52),
                 (4, 13824, 5120, "bf16", 53), (4, 28672, 8192, "bf16", 54)],
}


def quantize_bytes(N: int, K: int, bits: int) -> int:
    """Bytes one quantiser call must move at least: the 16-bit weights in,
    packed codes and fp16 scales and biases out."""
    return 2 * N * K + N * K * bits // 8 + 4 * N * (K // GROUP)
