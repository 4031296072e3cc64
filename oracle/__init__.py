"""Python access to the plain-C fp64 oracle (``oracle/aq_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The product package never
imports it.  It shares no code with the CUDA path; the only module both sides
use is ``workloads`` (seeded inputs, no method arithmetic).

Every function here is a thin ctypes call into the C file.  fp16 / bf16
inputs are widened to float64 before the call (exactly, so the oracle sees the
very values the GPU sees).  The definitions it follows are on the mlx-bun
pages, @mlx-bun/inference 1.0.0, kernels/quantization/: the LSB-first bit
stream of a 64-value group (affine-split-mma.ts, helper affine_unit), 2*B
words per group (affine3-mma.ts / affine4-mma.ts), and w = scale*q + bias.

Parity pins (tests/test_oracle_pins.py) tie every function to something
other than itself: hand-derived packed words, a bit-by-bit brute force, round
trips, closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "aq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libaq_oracle.so")
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32 = ctypes.c_int64, ctypes.c_int
            p = ctypes.c_void_p
            lib.oracle_words_per_row.argtypes = [i64, i32]
            lib.oracle_words_per_row.restype = i64
            lib.oracle_pack.argtypes = [p, i64, i64, i32, p]
            lib.oracle_unpack.argtypes = [p, i64, i64, i32, p]
            lib.oracle_dequant.argtypes = [p, p, p, i64, i64, i32, p]
            lib.oracle_matmul.argtypes = [p, p, p, p, i64, i64, i64, i32, p, p]
            lib.oracle_matmul_cols.argtypes = [p, p, p, p, i64, i64, i64, i32, p, i64, p, p]
            lib.oracle_matmul_threads.argtypes = [p, p, p, p, i64, i64, i64, i32, p, p, i32]
            lib.oracle_quantize.argtypes = [p, i64, i64, i32, p, p, p]
            lib.oracle_pack_g.argtypes = [p, i64, i64, i32, p]
            lib.oracle_unpack_g.argtypes = [p, i64, i64, i32, p]
            lib.oracle_dequant_g.argtypes = [p, p, p, i64, i64, i32, i32, p]
            lib.oracle_matmul_g.argtypes = [p, p, p, p, i64, i64, i64, i32, i32, p, p, i32]
            lib.oracle_quantize_g.argtypes = [p, i64, i64, i32, i32, p, p, p]
            lib.oracle_attention.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, i64, i32, i32,
                                             p, p, p]
            lib.oracle_gate_up_cols.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, i32, p, i64,
                                                p, p, p, p, p, p]
            lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16.restype = ctypes.c_uint16
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            for f in ("oracle_pack", "oracle_unpack", "oracle_dequant", "oracle_matmul",
                      "oracle_matmul_cols", "oracle_matmul_threads", "oracle_quantize",
                      "oracle_pack_g", "oracle_unpack_g", "oracle_dequant_g", "oracle_matmul_g",
                      "oracle_quantize_g", "oracle_attention", "oracle_gate_up_cols"):
                getattr(lib, f).restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


def words_per_row(K: int, bits: int) -> int:
    return K * bits // 32


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes uint8 [N, K] -> words uint32 [N, K*bits/32]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = codes.shape
    out = np.zeros((N, words_per_row(K, bits)), dtype=np.uint32)
    _check(_load().oracle_pack(_ptr(codes), N, K, bits, _ptr(out)), "pack")
    return out


def unpack(words: np.ndarray, K: int, bits: int) -> np.ndarray:
    """words uint32 [N, K*bits/32] -> codes uint8 [N, K]."""
    words = np.ascontiguousarray(words, dtype=np.uint32)
    N = words.shape[0]
    if words.shape[1] != words_per_row(K, bits):
        raise ValueError("words has the wrong row length for K and bits")
    out = np.zeros((N, K), dtype=np.uint8)
    _check(_load().oracle_unpack(_ptr(words), N, K, bits, _ptr(out)), "unpack")
    return out


def _f64(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def dequant(words: np.ndarray, scales: np.ndarray, biases: np.ndarray, K: int,
            bits: int) -> np.ndarray:
    """Dense W [N, K] in float64.  scales/biases: any float dtype (widened)."""
    words = np.ascontiguousarray(words, dtype=np.uint32)
    s, b = _f64(scales), _f64(biases)
    N = words.shape[0]
    out = np.zeros((N, K), dtype=np.float64)
    _check(_load().oracle_dequant(_ptr(words), _ptr(s), _ptr(b), N, K, bits, _ptr(out)),
           "dequant")
    return out


def matmul(x: np.ndarray, words: np.ndarray, scales: np.ndarray, biases: np.ndarray,
           bits: int, threads: int = 1):
    """y = x . dequant(W)^T in float64, and bound = sum_k |x*w|.

    x: float64 [M, K] (use workloads.to_f64 for fp16 / bf16 bit patterns).
    Returns (y [M, N], bound [M, N]).
    """
    x = _f64(x)
    words = np.ascontiguousarray(words, dtype=np.uint32)
    s, b = _f64(scales), _f64(biases)
    M, K = x.shape
    N = words.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    lib = _load()
    if threads > 1:
        rc = lib.oracle_matmul_threads(_ptr(x), _ptr(words), _ptr(s), _ptr(b), M, N, K, bits,
                                       _ptr(y), _ptr(bound), threads)
    else:
        rc = lib.oracle_matmul(_ptr(x), _ptr(words), _ptr(s), _ptr(b), M, N, K, bits,
                               _ptr(y), _ptr(bound))
    _check(rc, "matmul")
    return y, bound


def matmul_cols(x: np.ndarray, words: np.ndarray, scales: np.ndarray, biases: np.ndarray,
                bits: int, cols: Sequence[int]):
    """Only output columns `cols`: returns (y [M, len(cols)], bound [M, len(cols)])."""
    x = _f64(x)
    words = np.ascontiguousarray(words, dtype=np.uint32)
    s, b = _f64(scales), _f64(biases)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    M, K = x.shape
    N = words.shape[0]
    y = np.zeros((M, len(c)), dtype=np.float64)
    bound = np.zeros((M, len(c)), dtype=np.float64)
    _check(_load().oracle_matmul_cols(_ptr(x), _ptr(words), _ptr(s), _ptr(b), M, N, K, bits,
                                      _ptr(c), len(c), _ptr(y), _ptr(bound)), "matmul_cols")
    return y, bound


def gate_up(x: np.ndarray, gate, up, bits: int, cols: Optional[Sequence[int]] = None):
    """h = silu(g) * u with g = x . dequant(W_gate)^T, u = x . dequant(W_up)^T
    and silu(g) = g / (1 + exp(-g)), all in float64 (the gate/up epilogue of
    the mlx-bun 0.4.0 -> 1.0.0 page, src/model/trellis-shared-m.ts).

    gate, up: (words, scales, biases) each, laid out as for matmul().  cols:
    output columns to compute (all when None).  Returns a dict of [M, ncols]
    arrays: h, g, u, silu (= silu(g)), bound_g, bound_u (sum_k |x*w| of each
    product, for the tolerance)."""
    x = _f64(x)
    wg, sg, bg = gate
    wu, su, bu = up
    wg = np.ascontiguousarray(wg, dtype=np.uint32)
    wu = np.ascontiguousarray(wu, dtype=np.uint32)
    sg, bg, su, bu = _f64(sg), _f64(bg), _f64(su), _f64(bu)
    M, K = x.shape
    N = wg.shape[0]
    if wu.shape != wg.shape:
        raise ValueError("gate and up weights differ in shape")
    if cols is None:
        c, ncols, cp = None, N, None
    else:
        c = np.ascontiguousarray(cols, dtype=np.int64)
        ncols, cp = len(c), _ptr(c)
    out = {k: np.zeros((M, ncols), np.float64)
           for k in ("h", "g", "u", "silu", "bound_g", "bound_u")}
    _check(_load().oracle_gate_up_cols(
        _ptr(x), _ptr(wg), _ptr(sg), _ptr(bg), _ptr(wu), _ptr(su), _ptr(bu), M, N, K, bits,
        cp, ncols, *(_ptr(out[k]) for k in ("h", "g", "u", "silu", "bound_g", "bound_u"))),
        "gate_up")
    return out


def tolerance(bound: np.ndarray) -> np.ndarray:
    """Per-element acceptance bound |y - y_ref| <= 2e-3 * sum|x*w| + 1e-5."""
    return 2e-3 * bound + 1e-5


def f32_to_f16_bits(values) -> np.ndarray:
    """float32 values -> binary16 bit patterns (the oracle's own RNE conversion)."""
    v = np.asarray(values, dtype=np.float32).ravel()
    lib = _load()
    return np.array([lib.oracle_f32_to_f16(float(a)) for a in v], dtype=np.uint16)


def f16_bits_to_f32(bits) -> np.ndarray:
    """binary16 bit patterns -> float32 values (the oracle's own conversion)."""
    b = np.asarray(bits, dtype=np.uint16).ravel()
    lib = _load()
    return np.array([lib.oracle_f16_to_f32(int(h)) for h in b], dtype=np.float32)


def quantize(w: np.ndarray, bits: int):
    """Float weights [N, K] (float32 holding fp16 / bf16 values) -> (codes uint8
    [N, K], scale bits uint16 [N, K/64], bias bits uint16 [N, K/64]); pack the
    codes with pack().  The quantiser's rule is in aq_oracle.c."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    codes = np.zeros((N, K), dtype=np.uint8)
    G = K // 64
    sb = np.zeros((N, G), dtype=np.uint16)
    bb = np.zeros((N, G), dtype=np.uint16)
    _check(_load().oracle_quantize(_ptr(w), N, K, bits, _ptr(codes), _ptr(sb), _ptr(bb)),
           "quantize")
    return codes, sb, bb


# ---------------------------------------------------------------------------
# Other code widths (2, 3, 4, 5, 6, 8 bits) and group sizes (32, 64, 128)
# ---------------------------------------------------------------------------

def pack_g(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes uint8 [N, K] -> words uint32 [N, K*bits/32], any width of the set,
    K a multiple of 32."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = codes.shape
    out = np.zeros((N, K * bits // 32), dtype=np.uint32)
    _check(_load().oracle_pack_g(_ptr(codes), N, K, bits, _ptr(out)), "pack_g")
    return out


def unpack_g(words: np.ndarray, K: int, bits: int) -> np.ndarray:
    words = np.ascontiguousarray(words, dtype=np.uint32)
    N = words.shape[0]
    if words.shape[1] != K * bits // 32:
        raise ValueError("words has the wrong row length for K and bits")
    out = np.zeros((N, K), dtype=np.uint8)
    _check(_load().oracle_unpack_g(_ptr(words), N, K, bits, _ptr(out)), "unpack_g")
    return out


def dequant_g(words, scales, biases, K: int, bits: int, group: int) -> np.ndarray:
    words = np.ascontiguousarray(words, dtype=np.uint32)
    s, b = _f64(scales), _f64(biases)
    N = words.shape[0]
    out = np.zeros((N, K), dtype=np.float64)
    _check(_load().oracle_dequant_g(_ptr(words), _ptr(s), _ptr(b), N, K, bits, group, _ptr(out)),
           "dequant_g")
    return out


def matmul_g(x, words, scales, biases, bits: int, group: int, threads: int = 1):
    """y = x . dequant(W)^T and bound = sum_k |x*w| for any width and group size."""
    x = _f64(x)
    words = np.ascontiguousarray(words, dtype=np.uint32)
    s, b = _f64(scales), _f64(biases)
    M, K = x.shape
    N = words.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    bound = np.zeros((M, N), dtype=np.float64)
    _check(_load().oracle_matmul_g(_ptr(x), _ptr(words), _ptr(s), _ptr(b), M, N, K, bits, group,
                                   _ptr(y), _ptr(bound), threads), "matmul_g")
    return y, bound


def quantize_g(w: np.ndarray, bits: int, group: int):
    """quantize() for any width and group size."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    codes = np.zeros((N, K), dtype=np.uint8)
    G = K // group
    sb = np.zeros((N, G), dtype=np.uint16)
    bb = np.zeros((N, G), dtype=np.uint16)
    _check(_load().oracle_quantize_g(_ptr(w), N, K, bits, group, _ptr(codes), _ptr(sb), _ptr(bb)),
           "quantize_g")
    return codes, sb, bb


# ---------------------------------------------------------------------------
# Decode attention over a quantised KV cache
# ---------------------------------------------------------------------------

def attention(q, kwords, kscales, kbiases, vwords, vscales, vbiases, KV: int, N: int,
              bits: int, group: int):
    """o = softmax(q . Kd^T) . Vd per query head (grouped-query: head h reads
    KV head h / (H/KV)).  q float64 [H, D]; K/V words uint32 [KV*N, D*bits/32],
    scales/biases [KV*N, D/group].  Returns (o [H, D], smag [H, N], vmag [H, D])
    with smag = sum_d |q*k| and vmag = sum_n p*|v| (for the tolerance)."""
    q = _f64(q)
    H, D = q.shape
    kw = np.ascontiguousarray(kwords, dtype=np.uint32)
    vw = np.ascontiguousarray(vwords, dtype=np.uint32)
    ks, kb, vs, vb = _f64(kscales), _f64(kbiases), _f64(vscales), _f64(vbiases)
    o = np.zeros((H, D), np.float64)
    smag = np.zeros((H, N), np.float64)
    vmag = np.zeros((H, D), np.float64)
    _check(_load().oracle_attention(_ptr(q), _ptr(kw), _ptr(ks), _ptr(kb), _ptr(vw), _ptr(vs),
                                    _ptr(vb), H, KV, N, D, bits, group, _ptr(o), _ptr(smag),
                                    _ptr(vmag)), "attention")
    return o, smag, vmag
