"""Helpers for the GPU parity tests: move a workloads.Problem to the device,
run it through the C ABI, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads


def dev_tensors(p: workloads.Problem, device="cuda"):
    """codes (uint8), scales/biases (fp16) and x (fp16 or bf16) on the GPU."""
    codes = torch.from_numpy(np.ascontiguousarray(p.codes)).to(device)
    s = torch.from_numpy(np.ascontiguousarray(p.scales)).to(device)
    b = torch.from_numpy(np.ascontiguousarray(p.biases)).to(device)
    xb = torch.from_numpy(np.ascontiguousarray(p.x_bits).view(np.int16)).to(device)
    x = xb.view(torch.bfloat16 if p.x_dtype == "bf16" else torch.float16)
    return codes, s, b, x


def y_to_f64(y: torch.Tensor, dtype: str) -> np.ndarray:
    bits = y.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return workloads.to_f64(bits, dtype)


def reference(p: workloads.Problem, threads: int = 8):
    words = oracle.pack(p.codes, p.bits)
    return oracle.matmul(p.x_f64(), words, p.scales, p.biases, p.bits, threads=threads)


def assert_within_tolerance(y: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, what: str = "",
                            tol: np.ndarray = None):
    """|y - y_ref| <= 2e-3 * sum_k |x*w| + 1e-5 (or the given tol), element
    by element."""
    err = np.abs(y - y_ref)
    if tol is None:
        tol = oracle.tolerance(bound)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"(m={i},n={j}): y={y[i, j]:.6g} ref={y_ref[i, j]:.6g} "
                           f"tol={tol[i, j]:.3g}" for i, j in idx)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"{detail}")


def bf16_tile_tolerance(bound: np.ndarray, y_ref: np.ndarray) -> np.ndarray:
    """Per-element bound for the tensor-core path with bf16 activations on
    the other code widths and group sizes (outside the 3/4-bit group-64
    format, whose tolerance is the stated 2e-3 * sum_k |x*w| + 1e-5).

    There the dequantised tile holds bf16 weights (a kind::f16 MMA takes
    both operands in one type, and x is bf16): each weight is rounded once,
    |w_bf16 - w| <= 2^-8 |w|, so the products are off by at most
    2^-8 * sum_k |x_k w_k|; fp32 accumulation adds at most K * 2^-24 of the
    same sum (K <= 2^15 here: 2^-9); y is rounded once to bf16, 2^-8 |y|.
    The bound is the larger of that and the stated tolerance."""
    derived = (2.0 ** -8 + 2.0 ** -9) * bound + 2.0 ** -8 * np.abs(y_ref) + 1e-5
    return np.maximum(derived, oracle.tolerance(bound))


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the output dtype at |v| (normal range)."""
    mant = 10 if dtype == "fp16" else 7
    e = np.floor(np.log2(np.maximum(np.abs(v), 1e-30)))
    return np.exp2(e - mant)
