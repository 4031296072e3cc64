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


def assert_within_tolerance(y: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, what: str = ""):
    """|y - y_ref| <= 2e-3 * sum_k |x*w| + 1e-5, element by element."""
    err = np.abs(y - y_ref)
    tol = oracle.tolerance(bound)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"(m={i},n={j}): y={y[i, j]:.6g} ref={y_ref[i, j]:.6g} "
                           f"tol={tol[i, j]:.3g}" for i, j in idx)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"{detail}")


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the output dtype at |v| (normal range)."""
    mant = 10 if dtype == "fp16" else 7
    e = np.floor(np.log2(np.maximum(np.abs(v), 1e-30)))
    return np.exp2(e - mant)
