"""Host-side checks of the C ABI (no GPU needed).

* libaq.so loads and exports every function that include/aq.h declares;
* argument validation rejects bad calls before touching the GPU;
* the dispatch rule (aq_select) picks the expected kernel per shape.
"""
import ctypes
import os
import re

import pytest

import quantized_matmul_affine_gb300 as aq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "aq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(aq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("aq_pack", "aq_matmul", "aq_matmul_bf16", "aq_free", "aq_status_string",
                     "aq_stats"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(aq.lib_path())
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_test_hook_only_in_the_test_library():
    # the wait-expiry hook (tests/test_gpu_waits.py) exists only in the
    # separately built test library, never in libaq.so
    from quantized_matmul_affine_gb300 import build
    prod = ctypes.CDLL(aq.lib_path())
    assert not hasattr(prod, "aq_test_withhold")
    if build.up_to_date(build.TEST_LIB):
        assert hasattr(ctypes.CDLL(build.TEST_LIB), "aq_test_withhold")


def test_binding_has_the_same_names():
    for n in header_functions():
        assert hasattr(aq, n), n


def test_status_strings_and_version():
    assert aq.aq_status_string(0) == "ok"
    assert "invalid" in aq.aq_status_string(1)
    assert aq.aq_status_string(99) == "unknown status"
    assert aq.aq_variant_name(aq.AQ_VARIANT_QMV) == "qmv"
    assert aq.aq_variant_name(aq.AQ_VARIANT_GEMV) == "gemv"
    assert "sm_103a" in aq.aq_version()


def _raw():
    return aq.load()


A = 0x100000  # a 256-byte-aligned placeholder address; validation never dereferences


@pytest.mark.parametrize("M,N,K,bits,status", [
    (0, 16, 512, 4, 1),      # no rows (affineSplitMma throws on M < 1)
    (1, 0, 512, 4, 1),
    (1, 16, 0, 4, 1),
    (1, 16, 100, 4, 1),      # K not a multiple of 64
    (1, 16, 512, 5, 1),      # bits not 3 or 4
    (1, 16, 512, 2, 1),
    (-1, 16, 512, 4, 1),
])
def test_matmul_rejects_bad_shapes(M, N, K, bits, status):
    assert _raw().aq_matmul(A, A, A, A, M, N, K, bits, A, None) == status


def test_matmul_rejects_null_and_misaligned():
    lib = _raw()
    assert lib.aq_matmul(None, A, A, A, 1, 16, 512, 4, A, None) == 1
    assert lib.aq_matmul(A, A, A, A, 1, 16, 512, 4, None, None) == 1
    assert lib.aq_matmul(A + 1, A, A, A, 1, 16, 512, 4, A, None) == 3   # x not 2-aligned
    assert lib.aq_matmul(A, A + 2, A, A, 1, 16, 512, 4, A, None) == 3   # Wq not 4-aligned
    assert lib.aq_matmul_bf16(A, A, A + 1, A, 1, 16, 512, 4, A, None) == 3
    assert lib.aq_matmul_variant(7, 0, A, A, A, A, 1, 16, 512, 4, A, None) == 1
    assert lib.aq_matmul_variant(0, 5, A, A, A, A, 1, 16, 512, 4, A, None) == 1  # bad dtype


def test_pack_validation():
    lib = _raw()
    assert lib.aq_pack(A, 0, 512, 4, A, None) == 0       # empty: nothing to do
    assert lib.aq_pack(A, 4, 0, 4, A, None) == 0
    assert lib.aq_pack(A, 4, 100, 4, A, None) == 1
    assert lib.aq_pack(A, 4, 64, 7, A, None) == 1        # width outside 2, 3, 4, 5, 6, 8
    assert lib.aq_pack(A, 4, 48, 4, A, None) == 1        # K % 32 != 0
    assert lib.aq_pack(None, 4, 64, 4, A, None) == 1
    assert lib.aq_pack(A, 4, 64, 4, A + 2, None) == 3


def test_stats_interface():
    lib = _raw()
    assert lib.aq_stats(None, -1) == 1
    assert lib.aq_stats(None, 0) == 0
    assert len(aq.aq_stats()) == aq.AQ_NUM_VARIANTS
    aq.aq_stats_reset()
    assert aq.aq_stats() == [0] * aq.AQ_NUM_VARIANTS


def _declaration(name):
    text = open(os.path.join(ROOT, "include", "aq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    m = re.search(r"([A-Za-z_][A-Za-z0-9_ \*]*?)\b" + name + r"\s*\(([^)]*)\)\s*;", text)
    assert m, name
    ret = " ".join(m.group(1).split())
    params = [" ".join(p.split()) for p in m.group(2).split(",")]
    return ret, params


# The boundary's signatures as the scope table of the build fixes them
# (parameter names aside): return type and parameter types in order.
@pytest.mark.parametrize("name,ret,types", [
    ("aq_pack", "aq_status", ["const uint8_t *", "int64_t", "int64_t", "int", "uint32_t *",
                              "void *"]),
    ("aq_matmul", "aq_status", ["const void *", "const uint32_t *", "const void *",
                                "const void *", "int64_t", "int64_t", "int64_t", "int", "void *",
                                "void *"]),
    ("aq_matmul_bf16", "aq_status", ["const void *", "const uint32_t *", "const void *",
                                     "const void *", "int64_t", "int64_t", "int64_t", "int",
                                     "void *", "void *"]),
    ("aq_free", "void", ["void"]),
    ("aq_status_string", "const char *", ["aq_status"]),
    ("aq_stats", "aq_status", ["uint64_t *", "int"]),
    ("aq_stats_reset", "void", ["void"]),
])
def test_boundary_signatures(name, ret, types):
    r, params = _declaration(name)
    assert r.replace(" *", " *") == ret or r == ret.replace(" *", "*"), (name, r)
    got = []
    for p in params:
        if p == "void":
            got.append("void")
            continue
        # drop the parameter name: the last identifier
        t = re.sub(r"\s*\b[A-Za-z_][A-Za-z0-9_]*$", "", p)
        got.append(" ".join(t.replace("*", " * ").split()).replace(" *", " *"))
    norm = [" ".join(t.replace("*", " * ").split()) for t in types]
    assert got == norm, (name, got)


# The dispatch rule, on the shapes of the workloads (alignment assumed).
@pytest.mark.parametrize("M,N,K,bits,variant", [
    (1, 1024, 512, 4, aq.AQ_VARIANT_GEMV),
    (1, 4096, 4096, 4, aq.AQ_VARIANT_GEMV),
    (1, 10240, 5120, 3, aq.AQ_VARIANT_GEMV),
    (8, 10240, 5120, 3, aq.AQ_VARIANT_GEMV),
    (9, 10240, 5120, 3, aq.AQ_VARIANT_GEMV),
    (16, 10240, 5120, 3, aq.AQ_VARIANT_GEMV),
    (17, 10240, 5120, 3, aq.AQ_VARIANT_GEMV),
    (32, 10240, 5120, 3, aq.AQ_VARIANT_GEMV),
    (33, 10240, 5120, 3, aq.AQ_VARIANT_TC),     # 80 tiles: the clustered K split
    (64, 5120, 13824, 4, aq.AQ_VARIANT_TC),
    (128, 13824, 5120, 4, aq.AQ_VARIANT_TC),    # 108 tc tiles
    (129, 4096, 4096, 4, aq.AQ_VARIANT_TC),
    (1, 5120, 13824, 4, aq.AQ_VARIANT_GEMV),
    (1, 13824, 5120, 4, aq.AQ_VARIANT_GEMV),
    (1, 19456, 4096, 4, aq.AQ_VARIANT_GEMV),   # one pass of 128 rows per SM at M = 1
    (1, 19457, 4096, 4, aq.AQ_VARIANT_QMV),
    (1, 28672, 8192, 4, aq.AQ_VARIANT_QMV),
    (1, 128256, 4096, 4, aq.AQ_VARIANT_QMV),
    (8, 13824, 5120, 4, aq.AQ_VARIANT_GEMV),
    (2, 28672, 8192, 4, aq.AQ_VARIANT_GEMV),   # two passes of 95 rows per CTA
    (64, 10240, 5120, 3, aq.AQ_VARIANT_TC),
    (128, 28672, 8192, 4, aq.AQ_VARIANT_TC),
    (512, 28672, 8192, 4, aq.AQ_VARIANT_TC),
    (1, 100, 576, 4, aq.AQ_VARIANT_GENERIC),   # K % 512 != 0 -> generic
    (3, 7, 64, 3, aq.AQ_VARIANT_GENERIC),
])
def test_select(M, N, K, bits, variant):
    assert aq.aq_select(M, N, K, bits) == variant


def test_quantize_rejects_bad_arguments_before_any_launch():
    # validation happens on the host, before anything touches the device
    lib = ctypes.CDLL(aq.lib_path())
    for f in (lib.aq_quantize, lib.aq_quantize_bf16):
        f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        f.restype = ctypes.c_int
        assert f(16, 2, 100, 4, 16, 16, 16, None) == 1   # K % 64 != 0
        assert f(16, 2, 128, 5, 16, 16, 16, None) == 1   # bits
        assert f(16, -1, 128, 4, 16, 16, 16, None) == 1  # N < 0
        assert f(None, 2, 128, 4, 16, 16, 16, None) == 1  # NULL weights
        assert f(8, 2, 128, 4, 16, 16, 16, None) == 3    # weights not 16-byte aligned
        assert f(16, 2, 128, 4, 18, 16, 16, None) == 3   # words not 4-byte aligned
        assert f(16, 2, 128, 4, 16, 17, 16, None) == 3   # scales not 2-byte aligned
        assert f(16, 0, 128, 4, None, None, None, None) == 0  # empty: nothing queued


def test_select_invalid():
    assert aq.aq_select(0, 16, 512, 4) == -1
    assert aq.aq_select(1, 16, 512, 7) == -1


@pytest.mark.parametrize("M,N,K,bits,want", [
    (1, 4096, 4096, 4, "rows/cta=27 passes=1 tiles=2 colblocks=1 groups/stage=32 stages=2 ring=2 x=whole grid=152"),
    (2, 28672, 8192, 4, "rows/cta=190 passes=2"),
    (8, 600, 13824, 4, "x=staged"),
    (16, 10240, 5120, 3, "rows/cta=68 passes=1 tiles=5 colblocks=2"),
    (32, 10240, 5120, 3, "rows/cta=68 passes=1 tiles=5 colblocks=4 groups/stage=8 stages=10"),
    (32, 28672, 8192, 4, "rows/cta=190 passes=2 tiles=6 colblocks=4"),
])
def test_gemv_plan(M, N, K, bits, want):
    # The resident kernel's plan on a 152-SM GB300 (the SM count the library
    # assumes when no device is present): rows per CTA = ceil(N / SMs), whole
    # K per CTA, at most 128 rows per pass (96 with two or four column
    # blocks), ring as deep as 112 KB allows (two CTAs per SM) or, with two or
    # four column blocks (one CTA per SM), 227 KB.
    import torch
    if torch.cuda.is_available():
        pytest.skip("plan depends on the device's SM count")
    d = aq.aq_describe(M, N, K, bits)
    assert d.startswith("gemv ") and want in d, d
    smem = int(d.split("smem=")[1])
    assert smem <= (112 if M <= 8 else 227) * 1024


def test_attention_describe_host_checks():
    # argument checks need no device; without one the geometry is refused
    import torch
    assert aq.aq_attention_describe(3, 2, 100, 64, 4, 64) == "invalid arguments"
    assert aq.aq_attention_describe(4, 2, 100, 96, 4, 32) == "unsupported"
    assert aq.aq_attention_describe(4, 2, 100, 64, 3, 64) == "unsupported"
    d = aq.aq_attention_describe(16, 8, 8192, 256, 4, 64)
    if not torch.cuda.is_available():
        assert d == "no device"
    else:
        assert d.startswith("attn cluster=")
