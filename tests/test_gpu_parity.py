"""GPU parity: every kernel variant against the fp64 oracle, through the C ABI.

Tolerance (per element): |y - y_ref| <= 2e-3 * sum_k |x_k * w_nk| + 1e-5, on
inputs drawn like the workloads (centred weights).  Packing is bit-exact.
Closed forms whose value is exact in fp32 are checked to within one unit of
the output dtype's rounding.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _golden
from tests._gpu import assert_within_tolerance, dev_tensors, reference, ulp, y_to_f64

pytestmark = pytest.mark.gpu

aq = pytest.importorskip("quantized_matmul_affine_gb300")

GENERIC, QMV, TC, GEMV, TCW = (aq.AQ_VARIANT_GENERIC, aq.AQ_VARIANT_QMV, aq.AQ_VARIANT_TC,
                               aq.AQ_VARIANT_GEMV, aq.AQ_VARIANT_TCW)
ALL = [GENERIC, QMV, TC, GEMV, TCW]
ALL_IDS = ["generic", "qmv", "tc", "gemv", "tcw"]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    aq.aq_device_error(clear=True)
    yield
    assert aq.aq_device_error() == 0


def run(p: workloads.Problem, variant=aq.AQ_VARIANT_AUTO, Wq=None):
    codes, s, b, x = dev_tensors(p)
    if Wq is None:
        Wq = aq.aq_pack(codes, p.bits)
    y = aq.aq_matmul_variant(variant, x, Wq, s, b, p.bits)
    torch.cuda.synchronize()
    return y_to_f64(y, p.x_dtype)


# --------------------------------------------------------------------------
# Pack
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", list(_golden.pack_vectors()), ids=lambda c: c[0])
def test_pack_golden(case):
    name, bits, K, codes, words = case
    got = aq.aq_pack(torch.from_numpy(codes[None, :]).cuda(), bits)
    np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32)[0], words)


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("N,K", [(1, 64), (7, 192), (33, 1024), (300, 5120)])
def test_pack_bit_exact(bits, N, K):
    rng = np.random.default_rng(N * K + bits)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)  # high bits must be ignored
    got = aq.aq_pack(torch.from_numpy(codes).cuda(), bits).cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got, oracle.pack(codes, bits))


# --------------------------------------------------------------------------
# Matmul parity on small shapes spanning several tiles and ragged tails
# --------------------------------------------------------------------------

SHAPES = [
    # (M, N, K): one or several tiles of each kernel, with ragged N and M
    (1, 1024, 512),
    (1, 100, 512),
    (1, 37, 2048),
    (2, 256, 1024),
    (3, 61, 1536),
    (8, 128, 512),
    (9, 250, 1024),
    (16, 64, 3072),
    (17, 33, 512),
    (32, 96, 1024),
    (33, 40, 512),
    (64, 80, 1024),
    (100, 48, 512),
    (130, 300, 1024),
    (257, 200, 1536),
    # resident small-M kernel: several CTAs per partial tile, two passes per
    # CTA, a ring that wraps many times, x through its 4-slot ring
    (5, 1000, 1024),
    (2, 20000, 512),
    (1, 3000, 13824),
    (8, 600, 13824),
    # two 8-column blocks: staged x, rows past M, several passes, ring wraps
    (12, 700, 1536),
    (16, 2100, 2048),
    (11, 9000, 1024),
    # four 8-column blocks (one CTA per SM): rows past M, two passes
    (24, 700, 1536),
    (32, 2100, 2048),
    (29, 15000, 512),
    # swapped-role tensor-core kernel: K split over clusters of 2..8, a partial
    # last weight tile, several tiles
    (40, 300, 4096),
    (64, 700, 2048),
    (128, 1000, 1024),
    (77, 3000, 1536),
    # 512-row x tiles of the tc kernel (M > 512): two N = 256 MMAs per
    # k-step, a second x tile, rows past M
    (600, 300, 1024),
]

GEMV_MAX_M = 32


@pytest.mark.parametrize("variant", ALL + [aq.AQ_VARIANT_AUTO], ids=ALL_IDS + ["auto"])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_matmul_parity(shape, bits, dtype, variant):
    M, N, K = shape
    if variant == GEMV and M > GEMV_MAX_M:
        pytest.skip("the resident kernel serves M <= 32")
    if variant == TCW and M > 128:
        pytest.skip("the swapped-role tensor-core kernel serves M <= 128")
    p = workloads.make_problem("t", bits, N, K, M, dtype, seed=M * 7 + N + K + bits)
    y = run(p, variant)
    y_ref, bound = reference(p)
    assert_within_tolerance(y, y_ref, bound, f"{shape} bits={bits} {dtype} v={variant}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("shape", [(1, 17, 64), (5, 9, 576), (2, 300, 704)],
                         ids=lambda s: "x".join(map(str, s)))
def test_generic_ragged_k(shape, bits, dtype):
    # K % 512 != 0: only the generic kernel serves these, and auto must pick it.
    M, N, K = shape
    p = workloads.make_problem("t", bits, N, K, M, dtype, seed=K + N)
    y_ref, bound = reference(p)
    assert_within_tolerance(run(p), y_ref, bound, "auto")
    assert_within_tolerance(run(p, GENERIC), y_ref, bound, "generic")
    with pytest.raises(aq.AqError):
        run(p, QMV)


# --------------------------------------------------------------------------
# Closed forms (exact in fp32 up to the output rounding)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("variant", [GENERIC, QMV, TC], ids=["generic", "qmv", "tc"])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
def test_unit_rows_read_back_every_weight(bits, dtype, variant):
    # x = e_k (rows of the identity): y[k][n] = scale*q + bias, the single
    # dequantised weight, through the full decode path of the kernel.
    K, N = 512, 48
    p = workloads.make_problem("t", bits, N, K, K, dtype, seed=3)
    eye = np.eye(K, dtype=np.float32)
    xb = workloads.f32_to_bf16_bits(eye) if dtype == "bf16" else workloads.f32_to_fp16_bits(eye)
    p = workloads.Problem(p.name, bits, K, N, K, dtype, p.codes, p.scales, p.biases, xb, p.seed)
    y = run(p, variant)
    s = p.scales.astype(np.float64)
    b = p.biases.astype(np.float64)
    w = (s[:, np.arange(K) // 64] * p.codes + b[:, np.arange(K) // 64]).T  # [K, N]
    assert np.all(np.abs(y - w) <= ulp(w, dtype)), np.abs(y - w).max()


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
def test_gemv_unit_rows_read_back_every_weight(bits, dtype):
    # The resident kernel takes at most 8 rows: 64 calls of 8 rows of the
    # identity read back all 512 weights of every row.
    K, N = 512, 300
    p = workloads.make_problem("t", bits, N, K, 8, dtype, seed=4)
    codes, s, b, _ = dev_tensors(p)
    Wq = aq.aq_pack(codes, bits)
    sf = p.scales.astype(np.float64)
    bf = p.biases.astype(np.float64)
    w = (sf[:, np.arange(K) // 64] * p.codes + bf[:, np.arange(K) // 64]).T  # [K, N]
    conv = workloads.f32_to_bf16_bits if dtype == "bf16" else workloads.f32_to_fp16_bits
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    for k0 in range(0, K, 8):
        e = np.zeros((8, K), np.float32)
        e[np.arange(8), k0 + np.arange(8)] = 1.0
        x = torch.from_numpy(conv(e).view(np.int16)).view(tdt).cuda()
        y = y_to_f64(aq.aq_matmul_variant(GEMV, x, Wq, s, b, bits), dtype)
        ref = w[k0:k0 + 8]
        assert np.all(np.abs(y - ref) <= ulp(ref, dtype)), (k0, np.abs(y - ref).max())


@pytest.mark.parametrize("variant", ALL, ids=ALL_IDS)
@pytest.mark.parametrize("bits", [3, 4])
def test_zero_codes_and_zero_scales(bits, variant):
    p = workloads.make_problem("t", bits, 64, 1024, 4, "fp16", seed=11)
    xs = p.x_f64().reshape(p.M, p.G, 64).sum(axis=2)
    expected = xs @ p.biases.astype(np.float64).T
    pz = workloads.Problem(p.name, bits, p.M, p.N, p.K, "fp16", np.zeros_like(p.codes),
                           p.scales, p.biases, p.x_bits, p.seed)
    _, bound = reference(pz)
    assert_within_tolerance(run(pz, variant), expected, bound, "zero codes")
    ps = workloads.Problem(p.name, bits, p.M, p.N, p.K, "fp16", p.codes,
                           np.zeros_like(p.scales), p.biases, p.x_bits, p.seed)
    assert_within_tolerance(run(ps, variant), expected, bound, "zero scales")


@pytest.mark.parametrize("variant", ALL, ids=ALL_IDS)
def test_ones_row(variant):
    bits, K, N = 4, 1024, 40
    p = workloads.make_problem("t", bits, N, K, 1, "bf16", seed=12)
    ones = workloads.f32_to_bf16_bits(np.ones((1, K), np.float32))
    p = workloads.Problem(p.name, bits, 1, N, K, "bf16", p.codes, p.scales, p.biases, ones, 0)
    y_ref, bound = reference(p)
    assert_within_tolerance(run(p, variant), y_ref, bound, "ones")


# --------------------------------------------------------------------------
# Invariants and edge behaviour
# --------------------------------------------------------------------------

@pytest.mark.parametrize("variant", ALL, ids=ALL_IDS)
def test_deterministic(variant):
    p = workloads.make_problem("t", 3, 1000, 2048, 5, "bf16", seed=13)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, 3)
    ys = [aq.aq_matmul_variant(variant, x, Wq, s, b, 3).clone() for _ in range(3)]
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


def test_rows_match_single_row_calls():
    p = workloads.make_problem("t", 4, 300, 1024, 6, "fp16", seed=14)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, 4)
    y = y_to_f64(aq.aq_matmul(x, Wq, s, b, 4), "fp16")
    y_ref, bound = reference(p)
    for m in range(p.M):
        ym = y_to_f64(aq.aq_matmul(x[m:m + 1], Wq, s, b, 4), "fp16")
        assert_within_tolerance(ym, y_ref[m:m + 1], bound[m:m + 1], f"row {m}")
        assert np.all(np.abs(ym[0] - y[m]) <= 2 * oracle.tolerance(bound[m]))


@pytest.mark.parametrize("variant", ALL, ids=ALL_IDS)
def test_no_writes_outside_output(variant):
    M, N, K, bits = 3, 45, 1024, 4
    p = workloads.make_problem("t", bits, N, K, M, "fp16", seed=15)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, bits)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 12345, dtype=torch.int16, device="cuda")
    out = buf[guard:guard + M * N].view(torch.float16).view(M, N)
    aq.aq_matmul_variant(variant, x, Wq, s, b, bits, out=out)
    torch.cuda.synchronize()
    host = buf.cpu()
    assert torch.all(host[:guard] == 12345) and torch.all(host[guard + M * N:] == 12345)
    y_ref, bound = reference(p)
    assert_within_tolerance(y_to_f64(out, "fp16"), y_ref, bound, "canary")


def test_unsupported_variant_queues_nothing():
    p = workloads.make_problem("t", 4, 16, 576, 1, "fp16", seed=16)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, 4)
    with pytest.raises(aq.AqError) as e:
        aq.aq_matmul_variant(QMV, x, Wq, s, b, 4)
    assert e.value.status == 2


def test_dispatch_counters():
    p = workloads.make_problem("t", 4, 64, 512, 1, "fp16", seed=17)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, 4)
    aq.aq_stats(reset=True)
    aq.aq_matmul(x, Wq, s, b, 4)
    aq.aq_matmul_variant(GENERIC, x, Wq, s, b, 4)
    torch.cuda.synchronize()
    calls = aq.aq_stats()
    assert calls[GEMV] == 1 and calls[GENERIC] == 1


def test_host_entry_point():
    p = workloads.make_problem("t", 4, 200, 1024, 2, "bf16", seed=18)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, 4)
    x_host = x.cpu().pin_memory()
    out_host = torch.empty((2, 200), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    out_dev = torch.empty((2, 200), dtype=torch.bfloat16, device="cuda")
    aq.aq_matmul_host(x_host, Wq, s, b, 4, out_host, x_dev, out_dev)
    y_ref, bound = reference(p)
    assert_within_tolerance(y_to_f64(out_host, "bf16"), y_ref, bound, "host")
