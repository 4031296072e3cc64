"""Bounded waits that run out, on the GPU, without a fault or a hang.

Every pipeline wait in the kernels gives up after a time limit, records a
code in the library's device error word and lets the CTA wind down: the
copies and MMAs it issued complete, its tensor memory is released, and the
kernel returns.  These tests make such a wait run out on purpose and check
that the error is reported and that the next call is correct again.

They use the test-only build of the library (_build/test/libaq_test.so,
compiled from the same sources with AQ_TEST_HOOKS and a 1 ms wait limit): in
it, aq_test_withhold(1) makes the resident small-M kernel's producer skip the
copies of its first stage, and aq_test_withhold(2) does the same for the x
tiles of the large-M tensor-core kernel.  Nothing then completes that
stage's barrier (no copy is in flight for it), so the consumers' bounded
waits run out.  The product library libaq.so has no such hook.
"""
import ctypes

import pytest
import torch

import workloads
from tests._gpu import assert_within_tolerance, dev_tensors, reference, y_to_f64

pytestmark = pytest.mark.gpu

aq = pytest.importorskip("quantized_matmul_affine_gb300")
from quantized_matmul_affine_gb300 import build as aq_build  # noqa: E402

ERR_FAMILY_GEMV = 0x03  # low byte of the resident kernel's wait codes
ERR_FAMILY_TC = 0x02    # low byte of the tensor-core kernels' wait codes


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
    L.aq_select.argtypes = [i64, i64, i64, i32, i32]
    L.aq_select.restype = i32
    L.aq_device_error.argtypes = [p, i32]
    L.aq_device_error.restype = i32
    L.aq_test_withhold.argtypes = [i32]
    L.aq_test_withhold.restype = None
    L.aq_test_cluster_split.argtypes = [i32, i32]
    L.aq_test_cluster_split.restype = None
    code = ctypes.c_uint32(0)
    assert L.aq_device_error(ctypes.addressof(code), 1) == 0
    yield L
    L.aq_test_withhold(0)


def _device_error(L, clear):
    code = ctypes.c_uint32(0)
    assert L.aq_device_error(ctypes.addressof(code), int(clear)) == 0
    return code.value


def _call(L, variant, p, x, Wq, s, b):
    y = torch.empty((p.M, p.N), dtype=x.dtype, device="cuda")
    st = L.aq_matmul_variant(variant, aq.AQ_BF16 if p.x_dtype == "bf16" else aq.AQ_F16,
                             x.data_ptr(), Wq.data_ptr(), s.data_ptr(), b.data_ptr(), p.M, p.N,
                             p.K, p.bits, y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("withhold,variant,shape,family", [
    (1, aq.AQ_VARIANT_GEMV, (1, 1024, 4096), ERR_FAMILY_GEMV),   # two weight stages
    (2, aq.AQ_VARIANT_TC, (128, 1024, 1024), ERR_FAMILY_TC),     # 8 tiles, 16 stages each
])
def test_wait_runs_out_then_next_call_is_correct(lib, withhold, variant, shape, family):
    M, N, K = shape
    p = workloads.make_problem("w", 4, N, K, M, "bf16", seed=M + N + K)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, 4)
    torch.cuda.synchronize()
    try:
        lib.aq_test_withhold(withhold)
        _call(lib, variant, p, x, Wq, s, b)  # returns: the waits are bounded
    finally:
        lib.aq_test_withhold(0)
    code = _device_error(lib, clear=True)
    assert code != 0, "the withheld stage did not make a wait give up"
    assert code & 0xFF == family, hex(code)
    assert _device_error(lib, clear=False) == 0
    # the kernel wound down cleanly: the next call on the same SMs (tensor
    # memory allocated again) is correct and reports nothing
    y = y_to_f64(_call(lib, variant, p, x, Wq, s, b), "bf16")
    y_ref, bound = reference(p)
    assert_within_tolerance(y, y_ref, bound, f"after a withheld stage ({hex(code)})")
    assert _device_error(lib, clear=False) == 0


@pytest.mark.parametrize("ctas,tiles", [(4, 3), (8, 1)])
def test_wait_runs_out_under_the_clustered_split(lib, ctas, tiles):
    # the same with the tensor-core kernel's K range shared over the CTAs of
    # a cluster: every CTA still meets both cluster barriers after its wait
    # gives up, stores nothing, and the next call (same plan) is correct
    M, N, K = 64, 1000, 2048  # 8 tiles of 32 stages
    p = workloads.make_problem("w", 4, N, K, M, "bf16", seed=M + N + ctas)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, 4)
    torch.cuda.synchronize()
    lib.aq_test_cluster_split(ctas, tiles)
    try:
        try:
            lib.aq_test_withhold(2)
            _call(lib, aq.AQ_VARIANT_TC, p, x, Wq, s, b)
        finally:
            lib.aq_test_withhold(0)
        code = _device_error(lib, clear=True)
        assert code != 0, "the withheld stage did not make a wait give up"
        assert code & 0xFF == ERR_FAMILY_TC, hex(code)
        y = y_to_f64(_call(lib, aq.AQ_VARIANT_TC, p, x, Wq, s, b), "bf16")
    finally:
        lib.aq_test_cluster_split(0, 0)
    y_ref, bound = reference(p)
    assert_within_tolerance(y, y_ref, bound, f"after a withheld stage ({hex(code)})")
    assert _device_error(lib, clear=False) == 0
