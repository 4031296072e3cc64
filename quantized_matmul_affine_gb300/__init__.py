"""Python binding of libaq (include/aq.h): affine group-64 3/4-bit matmul on GB300.

Argument marshalling only.  Every function has the name of the C entry point
it calls; tensors are torch tensors (device memory for ``*_dev`` arguments),
``stream`` defaults to torch's current CUDA stream.  All the work runs in the
library's CUDA kernels; there is no Python or CPU compute path, and importing
this package fails if libaq.so cannot be loaded.

    y = aq_matmul(x, Wq, scales, biases, bits)        # fp16 x -> fp16 y
    y = aq_matmul_bf16(x, Wq, scales, biases, bits)   # bf16 x -> bf16 y
    Wq = aq_pack(codes, bits)                         # uint8 codes -> uint32 words
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional

import torch

from . import build as _build

__all__ = [
    "AqError", "AQ_F16", "AQ_BF16", "AQ_VARIANT_AUTO", "AQ_VARIANT_GENERIC", "AQ_VARIANT_QMV",
    "AQ_VARIANT_TC", "AQ_VARIANT_GEMV", "AQ_VARIANT_TCW", "AQ_NUM_VARIANTS", "aq_pack", "aq_quantize",
    "aq_quantize_bf16", "aq_matmul", "aq_matmul_bf16", "aq_matmul_multi", "aq_matmul_gate_up",
    "aq_matmul_ex", "aq_quantize_ex", "aq_attention_decode", "aq_attention_describe",
    "aq_attention_workspace_bytes", "aq_attention_decode_ws", "aq_attention_describe_ws",
    "aq_attention_decode_static",
    "aq_matmul_variant", "aq_matmul_host", "aq_select", "aq_describe", "aq_stats", "aq_stats_reset",
    "aq_device_error",
    "aq_free", "aq_status_string", "aq_variant_name", "aq_version", "lib_path", "load",
]

AQ_OK = 0
AQ_F16, AQ_BF16 = 0, 1
AQ_VARIANT_AUTO, AQ_VARIANT_GENERIC, AQ_VARIANT_QMV, AQ_VARIANT_TC = -1, 0, 1, 2
AQ_VARIANT_GEMV = 3
AQ_VARIANT_TCW = 4
AQ_NUM_VARIANTS = 5

_lib: Optional[ctypes.CDLL] = None


class AqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {aq_status_string(status)} (status {status})")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libaq.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise ImportError(f"libaq.so not built at {path}")
    lib = ctypes.CDLL(path)
    p, i64, i32, u32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    sz = ctypes.c_size_t
    sig = {
        "aq_pack": ([p, i64, i64, i32, p, p], i32),
        "aq_quantize": ([p, i64, i64, i32, p, p, p, p], i32),
        "aq_matmul_multi": ([i32, p, i32, p, p, p, p, i64, i64, i32, p, p], i32),
        "aq_matmul_ex": ([i32, p, p, p, p, i64, i64, i64, i32, i32, p, p], i32),
        "aq_attention_decode": ([i32, p, p, p, p, p, p, p, i64, i64, i64, i64, i32, i32, p, p],
                                i32),
        "aq_quantize_ex": ([i32, p, i64, i64, i32, i32, p, p, p, p], i32),
        "aq_matmul_gate_up": ([i32, p, p, p, p, p, p, p, i64, i64, i64, i32, p, p], i32),
        "aq_quantize_bf16": ([p, i64, i64, i32, p, p, p, p], i32),
        "aq_matmul": ([p, p, p, p, i64, i64, i64, i32, p, p], i32),
        "aq_matmul_bf16": ([p, p, p, p, i64, i64, i64, i32, p, p], i32),
        "aq_matmul_variant": ([i32, i32, p, p, p, p, i64, i64, i64, i32, p, p], i32),
        "aq_matmul_host": ([i32, p, p, p, p, i64, i64, i64, i32, p, p, p, p], i32),
        "aq_select": ([i64, i64, i64, i32, i32], i32),
        "aq_describe": ([i64, i64, i64, i32, i32, p, i32], i32),
        "aq_attention_describe": ([i64, i64, i64, i64, i32, i32, p, i32], i32),
        "aq_attention_workspace_bytes": ([i64, i64, i64, i64, i32, i32], sz),
        "aq_attention_decode_ws": ([i32, p, p, p, p, p, p, p, i64, i64, i64, i64, i32, i32, p, p,
                                    sz, p], i32),
        "aq_attention_describe_ws": ([i64, i64, i64, i64, i32, i32, sz, p, i32], i32),
        "aq_attention_decode_static": ([i32, p, p, p, p, p, p, p, i64, i64, i64, i64, i32, i32, p,
                                        p], i32),
        "aq_stats": ([p, i32], i32),
        "aq_stats_reset": ([], None),
        "aq_device_error": ([u32p, i32], i32),
        "aq_free": ([], None),
        "aq_status_string": ([i32], ctypes.c_char_p),
        "aq_variant_name": ([i32], ctypes.c_char_p),
        "aq_version": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, what: str) -> None:
    if status != AQ_OK:
        raise AqError(status, what)


def _dev(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _sized(t: torch.Tensor, name: str, nbytes: int, dtype=None) -> None:
    """The library reads or writes exactly nbytes through t's pointer: a
    buffer of another size (or dtype) is refused here, before any launch."""
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if _nbytes(t) != nbytes:
        raise ValueError(f"{name} holds {_nbytes(t)} bytes; this call uses {nbytes}")


_ACT = (torch.float16, torch.bfloat16)


def _check_weights(Wq, scales, biases, N: int, K: int, bits: int, group: int,
                   tag: str = "") -> None:
    """Sizes of one packed weight matrix; checked only when the arguments are
    otherwise valid (the library reports invalid ones with its own status)."""
    if bits not in (2, 3, 4, 5, 6, 8) or group not in (32, 64, 128) or K <= 0 or N <= 0:
        return
    if K % group or (K * bits) % 32:
        return
    _sized(Wq, f"Wq{tag}", N * K * bits // 8)
    _sized(scales, f"scales{tag}", 2 * N * (K // group), torch.float16)
    _sized(biases, f"biases{tag}", 2 * N * (K // group), torch.float16)


def _check_out(out, name: str, numel: int, dtype) -> None:
    if out.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {out.dtype}")
    _sized(out, name, numel * out.element_size())


def aq_status_string(status: int) -> str:
    return load().aq_status_string(status).decode()


def aq_variant_name(variant: int) -> str:
    return load().aq_variant_name(variant).decode()


def aq_version() -> str:
    return load().aq_version().decode()


def aq_pack(codes: torch.Tensor, bits: int, words: Optional[torch.Tensor] = None,
            stream=None) -> torch.Tensor:
    """codes uint8 [N, K] (device) -> words uint32-as-int32 [N, K*bits/32]."""
    N, K = codes.shape
    if codes.dtype != torch.uint8:
        raise ValueError("codes must be uint8")
    if words is None:
        words = torch.empty((N, K * bits // 32), dtype=torch.int32, device=codes.device)
    elif bits in (2, 3, 4, 5, 6, 8) and K % 32 == 0:
        _sized(words, "words", N * K * bits // 8)
    _check(load().aq_pack(_dev(codes, "codes"), N, K, bits, _dev(words, "words"),
                          _stream(stream)), "aq_pack")
    return words


def _quantize(dtype, w: torch.Tensor, bits: int, stream) -> tuple:
    want = torch.float16 if dtype == AQ_F16 else torch.bfloat16
    if w.dtype != want:
        raise ValueError(f"w must be {want}")
    N, K = w.shape
    Wq = torch.empty((N, K * bits // 32), dtype=torch.int32, device=w.device)
    scales = torch.empty((N, K // 64), dtype=torch.float16, device=w.device)
    biases = torch.empty((N, K // 64), dtype=torch.float16, device=w.device)
    f = load().aq_quantize if dtype == AQ_F16 else load().aq_quantize_bf16
    _check(f(_dev(w, "w"), N, K, bits, _dev(Wq, "Wq"), _dev(scales, "scales"),
             _dev(biases, "biases"), _stream(stream)), "aq_quantize")
    return Wq, scales, biases


def aq_quantize(w: torch.Tensor, bits: int, stream=None) -> tuple:
    """fp16 weights [N, K] (device) -> (Wq uint32-as-int32 [N, K*bits/32],
    scales fp16 [N, K/64], biases fp16 [N, K/64])."""
    return _quantize(AQ_F16, w, bits, stream)


def aq_quantize_bf16(w: torch.Tensor, bits: int, stream=None) -> tuple:
    """aq_quantize for bf16 weights."""
    return _quantize(AQ_BF16, w, bits, stream)


def _mm(variant: int, dtype: int, x, Wq, scales, biases, bits, out, stream) -> torch.Tensor:
    want = torch.float16 if dtype == AQ_F16 else torch.bfloat16
    if x.dtype != want:
        raise ValueError(f"x must be {want}")
    if scales.dtype != torch.float16 or biases.dtype != torch.float16:
        raise ValueError("scales and biases must be float16")
    K = x.shape[-1]
    M = x.numel() // K if K else 0
    N = scales.shape[0]
    if bits in (3, 4):
        _check_weights(Wq, scales, biases, N, K, bits, 64)
    if out is None:
        out = torch.empty((*x.shape[:-1], N), dtype=x.dtype, device=x.device)
    _check_out(out, "out", M * N, x.dtype)
    _check(load().aq_matmul_variant(variant, dtype, _dev(x, "x"), _dev(Wq, "Wq"),
                                    _dev(scales, "scales"), _dev(biases, "biases"), M, N, K,
                                    bits, _dev(out, "out"), _stream(stream)), "aq_matmul")
    return out


def aq_matmul(x, Wq, scales, biases, bits, out=None, stream=None) -> torch.Tensor:
    """y = x . dequant(W)^T for fp16 x [..., K]; returns fp16 [..., N]."""
    return _mm(AQ_VARIANT_AUTO, AQ_F16, x, Wq, scales, biases, bits, out, stream)


def aq_matmul_bf16(x, Wq, scales, biases, bits, out=None, stream=None) -> torch.Tensor:
    """y = x . dequant(W)^T for bf16 x [..., K]; returns bf16 [..., N]."""
    return _mm(AQ_VARIANT_AUTO, AQ_BF16, x, Wq, scales, biases, bits, out, stream)


def aq_matmul_ex(x, Wq, scales, biases, bits, group_size, out=None, stream=None):
    """Any code width of 2/3/4/5/6/8 bits and group size of 32/64/128; the
    dtype follows x (fp16 or bf16)."""
    if x.dtype not in _ACT:
        raise ValueError("x must be float16 or bfloat16")
    dtype = AQ_BF16 if x.dtype == torch.bfloat16 else AQ_F16
    K = x.shape[-1]
    M = x.numel() // K if K else 0
    N = scales.shape[0]
    _check_weights(Wq, scales, biases, N, K, bits, group_size)
    if out is None:
        out = torch.empty((*x.shape[:-1], N), dtype=x.dtype, device=x.device)
    _check_out(out, "out", M * N, x.dtype)
    _check(load().aq_matmul_ex(dtype, _dev(x, "x"), _dev(Wq, "Wq"), _dev(scales, "scales"),
                               _dev(biases, "biases"), M, N, K, bits, group_size,
                               _dev(out, "out"), _stream(stream)), "aq_matmul_ex")
    return out


def _attention_args(q, k, v, bits, group_size, out):
    if q.dtype not in _ACT:
        raise ValueError("q must be float16 or bfloat16")
    if q.dim() != 2 or len(k) != 3 or len(v) != 3 or any(t.dim() != 3 for t in (*k, *v)):
        raise ValueError("q must be [H, D]; k and v (words, scales, biases), each [KV, N, ...]")
    dtype = AQ_BF16 if q.dtype == torch.bfloat16 else AQ_F16
    H, D = q.shape
    KV, N = k[0].shape[0], k[0].shape[1]
    if bits in (4, 8) and group_size in (32, 64, 128) and D > 0 and D % group_size == 0:
        for side, (w, sc, bi) in (("k", k), ("v", v)):
            _sized(w, f"{side}_words", KV * N * D * bits // 8)
            _sized(sc, f"{side}_scales", 2 * KV * N * (D // group_size), torch.float16)
            _sized(bi, f"{side}_biases", 2 * KV * N * (D // group_size), torch.float16)
    if out is None:
        out = torch.empty((H, D), dtype=q.dtype, device=q.device)
    _check_out(out, "out", H * D, q.dtype)
    ptrs = (_dev(q, "q"), _dev(k[0], "k_words"), _dev(k[1], "k_scales"), _dev(k[2], "k_biases"),
            _dev(v[0], "v_words"), _dev(v[1], "v_scales"), _dev(v[2], "v_biases"))
    return dtype, ptrs, (H, KV, N, D), out


def aq_attention_decode(q, k, v, bits, group_size, out=None, stream=None) -> torch.Tensor:
    """Decode attention over a quantised KV cache.  q [H, D] (fp16 or bf16);
    k and v are (words [KV, N, D*bits/32] int32, scales [KV, N, D/group] fp16,
    biases [KV, N, D/group] fp16).  Returns o [H, D] in q's dtype."""
    dtype, ptrs, (H, KV, N, D), out = _attention_args(q, k, v, bits, group_size, out)
    _check(load().aq_attention_decode(dtype, *ptrs, H, KV, N, D, bits, group_size,
                                      _dev(out, "out"), _stream(stream)), "aq_attention_decode")
    return out


def aq_attention_decode_static(q, k, v, bits, group_size, out=None, stream=None) -> torch.Tensor:
    """aq_attention_decode_ws with the library's own fixed scratch instead of
    a workspace (nothing allocated per call); calls on one device must not
    overlap in time."""
    dtype, ptrs, (H, KV, N, D), out = _attention_args(q, k, v, bits, group_size, out)
    _check(load().aq_attention_decode_static(dtype, *ptrs, H, KV, N, D, bits, group_size,
                                             _dev(out, "out"), _stream(stream)),
           "aq_attention_decode_static")
    return out


def aq_attention_workspace_bytes(H: int, KV: int, N: int, D: int, bits: int,
                                 group_size: int) -> int:
    """Workspace bytes for aq_attention_decode_ws's several-cluster plan (0:
    one cluster per KV head is best, or the sizes are refused)."""
    return int(load().aq_attention_workspace_bytes(H, KV, N, D, bits, group_size))


def aq_attention_decode_ws(q, k, v, bits, group_size, workspace=None, out=None,
                           stream=None) -> torch.Tensor:
    """aq_attention_decode with a workspace (a uint8 device tensor whose
    first KV 32-bit words are zero before the first call; every call leaves
    them zero).  workspace=None allocates a zeroed one of the size the plan
    needs for this call."""
    dtype, ptrs, (H, KV, N, D), out = _attention_args(q, k, v, bits, group_size, out)
    if workspace is None:
        n = aq_attention_workspace_bytes(H, KV, N, D, bits, group_size)
        workspace = torch.zeros(max(n, 1), dtype=torch.uint8, device=q.device)
    if workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor")
    _check(load().aq_attention_decode_ws(dtype, *ptrs, H, KV, N, D, bits, group_size,
                                         _dev(out, "out"), _dev(workspace, "workspace"),
                                         workspace.numel(), _stream(stream)),
           "aq_attention_decode_ws")
    return out


def aq_quantize_ex(w: torch.Tensor, bits: int, group_size: int, stream=None) -> tuple:
    """aq_quantize for any code width and group size; w fp16 or bf16 [N, K]."""
    dtype = AQ_BF16 if w.dtype == torch.bfloat16 else AQ_F16
    N, K = w.shape
    Wq = torch.empty((N, K * bits // 32), dtype=torch.int32, device=w.device)
    scales = torch.empty((N, K // group_size), dtype=torch.float16, device=w.device)
    biases = torch.empty((N, K // group_size), dtype=torch.float16, device=w.device)
    _check(load().aq_quantize_ex(dtype, _dev(w, "w"), N, K, bits, group_size, _dev(Wq, "Wq"),
                                 _dev(scales, "scales"), _dev(biases, "biases"), _stream(stream)),
           "aq_quantize_ex")
    return Wq, scales, biases


def aq_matmul_multi(x, weights, bits, outs=None, stream=None) -> list:
    """Several projections of the same x in one call: weights is a list of
    (Wq, scales, biases) triples (1..4); returns [y_j] in x's dtype."""
    dtype = AQ_BF16 if x.dtype == torch.bfloat16 else AQ_F16
    P = len(weights)
    K = x.shape[-1]
    M = x.numel() // K if K else 0
    Ns = [w[1].shape[0] for w in weights]
    if bits in (3, 4):
        for j, (w, n) in enumerate(zip(weights, Ns)):
            _check_weights(w[0], w[1], w[2], n, K, bits, 64, f"[{j}]")
    if outs is None:
        outs = [torch.empty((*x.shape[:-1], n), dtype=x.dtype, device=x.device) for n in Ns]
    if len(outs) != P:
        raise ValueError("one output per projection")
    for j, (o, n) in enumerate(zip(outs, Ns)):
        _check_out(o, f"outs[{j}]", M * n, x.dtype)
    ptr_arr = ctypes.c_void_p * max(P, 1)
    Wp = ptr_arr(*[_dev(w[0], "Wq") for w in weights])
    Sp = ptr_arr(*[_dev(w[1], "scales") for w in weights])
    Bp = ptr_arr(*[_dev(w[2], "biases") for w in weights])
    Op = ptr_arr(*[_dev(o, "out") for o in outs])
    Na = (ctypes.c_int64 * max(P, 1))(*Ns)
    _check(load().aq_matmul_multi(dtype, _dev(x, "x"), P, ctypes.cast(Wp, ctypes.c_void_p),
                                  ctypes.cast(Sp, ctypes.c_void_p), ctypes.cast(Bp, ctypes.c_void_p),
                                  ctypes.cast(Na, ctypes.c_void_p), M, K, bits,
                                  ctypes.cast(Op, ctypes.c_void_p), _stream(stream)),
           "aq_matmul_multi")
    return outs


def aq_matmul_gate_up(x, gate, up, bits, out=None, stream=None) -> torch.Tensor:
    """h = silu(x . W_gate^T) * (x . W_up^T); gate and up are (Wq, scales,
    biases) triples with the same N."""
    dtype = AQ_BF16 if x.dtype == torch.bfloat16 else AQ_F16
    K = x.shape[-1]
    M = x.numel() // K if K else 0
    N = gate[1].shape[0]
    if bits in (3, 4):
        _check_weights(gate[0], gate[1], gate[2], N, K, bits, 64, " (gate)")
        _check_weights(up[0], up[1], up[2], N, K, bits, 64, " (up)")
    if out is None:
        out = torch.empty((*x.shape[:-1], N), dtype=x.dtype, device=x.device)
    _check_out(out, "out", M * N, x.dtype)
    _check(load().aq_matmul_gate_up(dtype, _dev(x, "x"), _dev(gate[0], "Wq"),
                                    _dev(gate[1], "scales"), _dev(gate[2], "biases"),
                                    _dev(up[0], "Wq"), _dev(up[1], "scales"),
                                    _dev(up[2], "biases"), M, N, K, bits, _dev(out, "out"),
                                    _stream(stream)), "aq_matmul_gate_up")
    return out


def aq_matmul_variant(variant, x, Wq, scales, biases, bits, out=None, stream=None):
    """Explicit kernel variant; the dtype follows x (fp16 or bf16)."""
    dtype = AQ_BF16 if x.dtype == torch.bfloat16 else AQ_F16
    return _mm(variant, dtype, x, Wq, scales, biases, bits, out, stream)


def aq_matmul_host(x_host: torch.Tensor, Wq, scales, biases, bits, out_host: torch.Tensor,
                   x_dev: torch.Tensor, out_dev: torch.Tensor, stream=None) -> torch.Tensor:
    """Host x in, host y out (device staging buffers supplied); synchronises."""
    dtype = AQ_BF16 if x_host.dtype == torch.bfloat16 else AQ_F16
    if x_host.is_cuda or out_host.is_cuda:
        raise ValueError("x_host and out_host must be host tensors")
    K = x_host.shape[-1]
    M = x_host.numel() // K
    N = scales.shape[0]
    if bits in (3, 4):
        _check_weights(Wq, scales, biases, N, K, bits, 64)
    _check_out(out_host, "out_host", M * N, x_host.dtype)
    _check_out(x_dev, "x_dev", M * K, x_host.dtype)
    _check_out(out_dev, "out_dev", M * N, x_host.dtype)
    _check(load().aq_matmul_host(dtype, x_host.data_ptr(), _dev(Wq, "Wq"),
                                 _dev(scales, "scales"), _dev(biases, "biases"), M, N, K, bits,
                                 out_host.data_ptr(), _dev(x_dev, "x_dev"),
                                 _dev(out_dev, "out_dev"), _stream(stream)), "aq_matmul_host")
    return out_host


def aq_select(M: int, N: int, K: int, bits: int, dtype: int = AQ_F16) -> int:
    return load().aq_select(M, N, K, bits, dtype)


def aq_describe(M: int, N: int, K: int, bits: int, dtype: int = AQ_F16) -> str:
    buf = ctypes.create_string_buffer(256)
    load().aq_describe(M, N, K, bits, dtype, ctypes.addressof(buf), 256)
    return buf.value.decode()


def aq_attention_describe(H: int, KV: int, N: int, D: int, bits: int, group_size: int) -> str:
    """The launch geometry of aq_attention_decode for these sizes (needs the
    device for its count of co-resident clusters)."""
    buf = ctypes.create_string_buffer(256)
    load().aq_attention_describe(H, KV, N, D, bits, group_size, ctypes.addressof(buf), 256)
    return buf.value.decode()


def aq_attention_describe_ws(H: int, KV: int, N: int, D: int, bits: int, group_size: int,
                             workspace_bytes: int) -> str:
    """The launch geometry of aq_attention_decode_ws with a workspace of
    workspace_bytes."""
    buf = ctypes.create_string_buffer(256)
    load().aq_attention_describe_ws(H, KV, N, D, bits, group_size, workspace_bytes,
                                    ctypes.addressof(buf), 256)
    return buf.value.decode()


def aq_stats(reset: bool = False) -> List[int]:
    """Calls per variant (aq_stats); reset=True also calls aq_stats_reset."""
    buf = (ctypes.c_uint64 * AQ_NUM_VARIANTS)()
    _check(load().aq_stats(ctypes.cast(buf, ctypes.c_void_p), AQ_NUM_VARIANTS), "aq_stats")
    if reset:
        aq_stats_reset()
    return list(buf)


def aq_stats_reset() -> None:
    load().aq_stats_reset()


def aq_device_error(clear: bool = False) -> int:
    code = ctypes.c_uint32(0)
    _check(load().aq_device_error(ctypes.addressof(code), int(clear)), "aq_device_error")
    return code.value


def aq_free() -> None:
    load().aq_free()


load()
