"""GPU parity for the tensor-core kernel's clustered K split.

With fewer weight tiles than SMs and x tiles of at most 128 rows, the
large-M kernel can share T consecutive tiles among the C > T CTAs of a
cluster: the cluster's K stages, tile after tile, are dealt out in even runs
of whole 4-group super-stages, each CTA accumulates one or two partial
tiles, and the partials are added in rank (K) order through distributed
shared memory.  These tests force several (C, T) plans through the test
build of the library (aq_test_cluster_split), so that runs straddling tile
boundaries, last clusters with fewer tiles, ragged N and ragged M are all
covered whatever the planner would pick on this GPU, and compare each
result with the oracle element by element.  They also check that the sums
are deterministic and that the product library's own plan is correct at the
pages' 3-bit 10240x5120 shape (sampled columns).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._gpu import (assert_within_tolerance, bf16_tile_tolerance, dev_tensors, reference,
                        y_to_f64)

pytestmark = pytest.mark.gpu

aq = pytest.importorskip("quantized_matmul_affine_gb300")
from quantized_matmul_affine_gb300 import build as aq_build  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not aq_build.up_to_date(aq_build.TEST_LIB):
        aq_build.build()
    L = ctypes.CDLL(aq_build.TEST_LIB)
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.aq_matmul_variant.argtypes = [i32, i32, p, p, p, p, i64, i64, i64, i32, p, p]
    L.aq_matmul_variant.restype = i32
    L.aq_matmul_ex.argtypes = [i32, p, p, p, p, i64, i64, i64, i32, i32, p, p]
    L.aq_matmul_ex.restype = i32
    L.aq_device_error.argtypes = [p, i32]
    L.aq_device_error.restype = i32
    L.aq_test_cluster_split.argtypes = [i32, i32]
    L.aq_test_cluster_split.restype = None
    L.aq_test_describe_tc.argtypes = [i64, i64, i64, i32, i32, ctypes.c_char_p, i32]
    L.aq_test_describe_tc.restype = i32
    code = ctypes.c_uint32(0)
    assert L.aq_device_error(ctypes.addressof(code), 1) == 0
    yield L
    L.aq_test_cluster_split(0, 0)


def _device_error(L):
    code = ctypes.c_uint32(0)
    assert L.aq_device_error(ctypes.addressof(code), 0) == 0
    return code.value


def _describe(L, M, N, K, bits, dtype):
    buf = ctypes.create_string_buffer(512)
    L.aq_test_describe_tc(M, N, K, bits, dtype, buf, 512)
    return buf.value.decode()


def _tc(L, p, x, Wq, s, b):
    y = torch.empty((p.M, p.N), dtype=x.dtype, device="cuda")
    st = L.aq_matmul_variant(aq.AQ_VARIANT_TC, aq.AQ_BF16 if p.x_dtype == "bf16" else aq.AQ_F16,
                             x.data_ptr(), Wq.data_ptr(), s.data_ptr(), b.data_ptr(), p.M, p.N,
                             p.K, p.bits, y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return y


# (M, N, K, bits, x dtype, C, T).  Tiles are 128 weight rows; G = K / 64
# stages a tile.  Comments: tiles, clusters (tiles in the last), runs.
FORCED = [
    (64, 1000, 2048, 4, "bf16", 3, 2),   # 8 tiles, 4 clusters; runs 20/20/24 of G=32
    (100, 1000, 2048, 3, "fp16", 5, 3),  # 128-row x tile, M ragged; 3 clusters (2)
    (33, 300, 1024, 4, "fp16", 8, 5),    # 3 tiles, one cluster of 8 short runs
    (64, 2000, 512, 3, "bf16", 7, 4),    # G=8: runs of one or two super-stages
    (128, 640, 4096, 4, "bf16", 4, 3),   # 5 tiles: clusters of 3 and 2 tiles
    (50, 129, 1024, 4, "bf16", 2, 1),    # N ragged: the second tile holds one row
    (5, 700, 1024, 3, "bf16", 4, 3),     # few x rows: 6 tiles, 2 clusters of 3
    (128, 384, 1536, 3, "fp16", 6, 1),   # G=24: six runs of one super-stage a tile
]


@pytest.mark.parametrize("M,N,K,bits,dtype,C,T", FORCED)
def test_forced_cluster_split_parity(lib, M, N, K, bits, dtype, C, T):
    p = workloads.make_problem("cs", bits, N, K, M, dtype, seed=M * 7 + N + K + C)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, bits)
    torch.cuda.synchronize()
    dt = aq.AQ_BF16 if dtype == "bf16" else aq.AQ_F16
    lib.aq_test_cluster_split(C, T)
    try:
        desc = _describe(lib, M, N, K, bits, dt)
        assert f"cluster_split={C}x{T}" in desc, desc
        y1 = _tc(lib, p, x, Wq, s, b)
        y2 = _tc(lib, p, x, Wq, s, b)
    finally:
        lib.aq_test_cluster_split(0, 0)
    assert _device_error(lib) == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), "sums not deterministic"
    y_ref, bound = reference(p)
    assert_within_tolerance(y_to_f64(y1, dtype), y_ref, bound, f"{desc}")


def test_forced_off_matches_the_oracle_too(lib):
    # the same problem with the split disabled (whole tiles / halves): both
    # plans within tolerance of the oracle
    M, N, K, bits = 64, 1000, 2048, 4
    p = workloads.make_problem("cs", bits, N, K, M, "bf16", seed=11)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, bits)
    torch.cuda.synchronize()
    lib.aq_test_cluster_split(-1, 0)
    try:
        assert "cluster_split=0x0" in _describe(lib, M, N, K, bits, aq.AQ_BF16)
        y_off = _tc(lib, p, x, Wq, s, b)
    finally:
        lib.aq_test_cluster_split(0, 0)
    lib.aq_test_cluster_split(3, 2)
    try:
        y_on = _tc(lib, p, x, Wq, s, b)
    finally:
        lib.aq_test_cluster_split(0, 0)
    y_ref, bound = reference(p)
    assert_within_tolerance(y_to_f64(y_off, "bf16"), y_ref, bound, "split off")
    assert_within_tolerance(y_to_f64(y_on, "bf16"), y_ref, bound, "split 3x2")


@pytest.mark.parametrize("bits,group,dtype,C,T", [(8, 32, "bf16", 4, 1), (5, 128, "fp16", 3, 2),
                                                  (2, 64, "bf16", 8, 5)])
def test_forced_cluster_split_general_widths(lib, bits, group, dtype, C, T):
    # the general-width dequantisation (A tiles in shared memory) on the same split
    M, N, K = 70, 900, 1024
    rng = np.random.default_rng(bits + group)
    G = K // group
    codes = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    s = (np.abs(rng.standard_normal((N, G))) * (0.16 / (1 << bits)) + 1e-3).astype(np.float16)
    b = (-(1 << (bits - 1)) * s.astype(np.float64) + rng.standard_normal((N, G)) * 1e-3).astype(
        np.float16)
    x_bits = workloads.make_x(M, K, dtype, seed=bits * 3 + group)
    xt = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda().view(
        torch.bfloat16 if dtype == "bf16" else torch.float16)
    Wq = aq.aq_pack(torch.from_numpy(codes).cuda(), bits)
    st, bt = torch.from_numpy(s).cuda(), torch.from_numpy(b).cuda()
    y = torch.empty((M, N), dtype=xt.dtype, device="cuda")
    torch.cuda.synchronize()
    lib.aq_test_cluster_split(C, T)
    try:
        rc = lib.aq_matmul_ex(aq.AQ_BF16 if dtype == "bf16" else aq.AQ_F16, xt.data_ptr(),
                              Wq.data_ptr(), st.data_ptr(), bt.data_ptr(), M, N, K, bits, group,
                              y.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
    finally:
        lib.aq_test_cluster_split(0, 0)
    assert rc == 0
    assert _device_error(lib) == 0
    y_ref, bound = oracle.matmul_g(workloads.to_f64(x_bits, dtype), oracle.pack_g(codes, bits),
                                   s, b, bits, group, threads=8)
    tol = bf16_tile_tolerance(bound, y_ref) if dtype == "bf16" else None
    assert_within_tolerance(y_to_f64(y, dtype), y_ref, bound, f"bits={bits} group={group}", tol)


@pytest.mark.parametrize("M", [33, 64, 128])
def test_planner_choice_at_the_pages_shape(M):
    # the product library's own plan on the pages' 3-bit 10240x5120 shape,
    # forced onto the tensor-core kernel; sampled columns against the oracle
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    N, K, bits = 10240, 5120, 3
    # 80 weight tiles on more SMs: the dispatch takes tc, whose planner
    # shares the tiles' K ranges over clusters
    plan = aq.aq_describe(M, N, K, bits, aq.AQ_F16)
    assert plan.startswith("tc ") and "cluster_split=0x0" not in plan, plan
    p = workloads.make_problem("cs", bits, N, K, M, "fp16", seed=M + 5)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, bits)
    y = aq.aq_matmul_variant(aq.AQ_VARIANT_TC, x, Wq, s, b, bits)
    y2 = aq.aq_matmul_variant(aq.AQ_VARIANT_TC, x, Wq, s, b, bits)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    cols = np.unique(np.concatenate([np.arange(0, 130), np.arange(N - 130, N),
                                     np.random.default_rng(M).integers(0, N, 200)]))
    y_ref, bound = oracle.matmul_cols(p.x_f64(), oracle.pack(p.codes, bits), p.scales, p.biases,
                                      bits, cols)
    assert_within_tolerance(y_to_f64(y, "fp16")[:, cols], y_ref, bound, f"M={M}")
    assert aq.aq_device_error() == 0
