"""GPU parity for the other code widths (2, 3, 4, 5, 6, 8 bits) and group
sizes (32, 64, 128): aq_pack bit-exact against the oracle's packer,
aq_matmul_ex within the matmul tolerance of the oracle's general matmul,
aq_quantize_ex bit-exact against the oracle's general quantiser.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._gpu import assert_within_tolerance, bf16_tile_tolerance, y_to_f64

pytestmark = pytest.mark.gpu

aq = pytest.importorskip("quantized_matmul_affine_gb300")

WIDTHS = [2, 3, 4, 5, 6, 8]
GROUPS = [32, 64, 128]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _problem(bits, group, M, N, K, dtype, seed):
    """Codes, fp16 scales/biases centred like the workloads, x of dtype."""
    rng = np.random.default_rng(seed)
    G = K // group
    codes = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
    s = (np.abs(rng.standard_normal((N, G))) * (0.16 / (1 << bits)) + 1e-3).astype(np.float16)
    b = (-(1 << (bits - 1)) * s.astype(np.float64) + rng.standard_normal((N, G)) * 1e-3).astype(
        np.float16)
    x_bits = workloads.make_x(M, K, dtype, seed + 1)
    return codes, s, b, x_bits


def _x(x_bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("N,K", [(1, 32), (7, 96), (33, 1024)])
def test_pack_bit_exact(bits, N, K):
    rng = np.random.default_rng(bits + N + K)
    codes = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    got = aq.aq_pack(torch.from_numpy(codes).cuda(), bits).cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got, oracle.pack_g(codes, bits))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("M,N,K", [(1, 100, 512), (5, 37, 1024), (20, 64, 384)])
def test_matmul_ex_parity(M, N, K, bits, group, dtype):
    codes, s, b, x_bits = _problem(bits, group, M, N, K, dtype, seed=bits * 100 + group + M)
    Wq = aq.aq_pack(torch.from_numpy(codes).cuda(), bits)
    y = aq.aq_matmul_ex(_x(x_bits, dtype), Wq, torch.from_numpy(s).cuda(),
                        torch.from_numpy(b).cuda(), bits, group)
    torch.cuda.synchronize()
    y_ref, bound = oracle.matmul_g(workloads.to_f64(x_bits, dtype), oracle.pack_g(codes, bits),
                                   s, b, bits, group, threads=8)
    on_tc = M > 4 and K % 512 == 0 and not (bits in (3, 4) and group == 64)  # bf16 weight tiles
    tol = bf16_tile_tolerance(bound, y_ref) if dtype == "bf16" and on_tc else None
    assert_within_tolerance(y_to_f64(y, dtype), y_ref, bound, f"bits={bits} group={group}", tol)


# Past 4 rows (K % 512 == 0, aligned operands): the tensor-core kernel with
# the general-width dequantisation.  64-, 128- and 256-row x tiles, several x
# tiles, ragged N and M, few weight tiles (each split in K over two CTAs),
# and N = 20000 (157 weight tiles: one round over the SMs plus five tiles
# split in K).
TC_SHAPES = [(5, 90, 512), (33, 300, 1024), (64, 700, 2048), (100, 129, 512),
             (256, 520, 1024), (300, 140, 512), (40, 20000, 512)]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("M,N,K", TC_SHAPES)
def test_matmul_ex_tensor_core(M, N, K, bits, group, dtype):
    if bits in (3, 4) and group == 64:
        pytest.skip("the 3/4-bit group-64 format runs as aq_matmul")
    codes, s, b, x_bits = _problem(bits, group, M, N, K, dtype, seed=bits * 7 + group + M + N)
    Wq = aq.aq_pack(torch.from_numpy(codes).cuda(), bits)
    st, bt = torch.from_numpy(s).cuda(), torch.from_numpy(b).cuda()
    x = _x(x_bits, dtype)
    torch.cuda.synchronize()
    aq.aq_stats(reset=True)
    y = aq.aq_matmul_ex(x, Wq, st, bt, bits, group)
    torch.cuda.synchronize()
    calls = aq.aq_stats()
    assert calls[aq.AQ_VARIANT_TC] == 1 and calls[aq.AQ_VARIANT_GENERIC] == 0, calls
    y_ref, bound = oracle.matmul_g(workloads.to_f64(x_bits, dtype), oracle.pack_g(codes, bits),
                                   s, b, bits, group, threads=8)
    tol = bf16_tile_tolerance(bound, y_ref) if dtype == "bf16" else None
    assert_within_tolerance(y_to_f64(y, dtype), y_ref, bound, f"bits={bits} group={group}", tol)
    assert aq.aq_device_error() == 0


def test_matmul_ex_tensor_core_is_deterministic():
    M, N, K, bits, group = 200, 20000, 512, 5, 32
    codes, s, b, x_bits = _problem(bits, group, M, N, K, "bf16", seed=99)
    Wq = aq.aq_pack(torch.from_numpy(codes).cuda(), bits)
    st, bt = torch.from_numpy(s).cuda(), torch.from_numpy(b).cuda()
    x = _x(x_bits, "bf16")
    y1 = aq.aq_matmul_ex(x, Wq, st, bt, bits, group)
    y2 = aq.aq_matmul_ex(x, Wq, st, bt, bits, group)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_matmul_ex_at_the_format_is_aq_matmul():
    # 4 bits, groups of 64: the same kernels and bits as aq_matmul_bf16
    p = workloads.make_problem("t", 4, 300, 2048, 3, "bf16", seed=8)
    Wq = aq.aq_pack(torch.from_numpy(p.codes).cuda(), 4)
    s, b = torch.from_numpy(p.scales).cuda(), torch.from_numpy(p.biases).cuda()
    x = _x(p.x_bits, "bf16")
    y1 = aq.aq_matmul_ex(x, Wq, s, b, 4, 64)
    y2 = aq.aq_matmul_bf16(x, Wq, s, b, 4)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_matmul_ex_rejects_bad_group():
    codes, s, b, x_bits = _problem(4, 32, 1, 8, 96, "fp16", seed=1)
    Wq = aq.aq_pack(torch.from_numpy(codes).cuda(), 4)
    with pytest.raises(aq.AqError) as e:
        aq.aq_matmul_ex(_x(x_bits, "fp16"), Wq, torch.from_numpy(s).cuda(),
                        torch.from_numpy(b).cuda(), 4, 48)
    assert e.value.status == 1


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", WIDTHS)
def test_quantize_ex_bit_exact(bits, group, dtype):
    N, K = 45, 512
    b16, vals = workloads.make_weights(N, K, dtype, seed=bits + group)
    w = torch.from_numpy(b16.view(np.int16)).cuda().view(
        torch.bfloat16 if dtype == "bf16" else torch.float16)
    Wq, s, b = aq.aq_quantize_ex(w, bits, group)
    torch.cuda.synchronize()
    codes, sb, bb = oracle.quantize_g(vals, bits, group)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint16), sb)
    np.testing.assert_array_equal(b.cpu().numpy().view(np.uint16), bb)
    np.testing.assert_array_equal(Wq.cpu().numpy().view(np.uint32), oracle.pack_g(codes, bits))


@pytest.mark.parametrize("bits,group", [(2, 32), (3, 128), (5, 64), (6, 32), (8, 128)])
@pytest.mark.parametrize("M,N,K", [(2, 1001, 4096), (4, 50, 2048), (8, 33, 1280), (9, 64, 1280),
                                   (32, 40, 640), (33, 17, 256), (1, 3, 32 * 33)])
def test_matmul_ex_small_m_shapes(M, N, K, bits, group):
    # the segment kernel: row blocks of 1/2/4/8 activation rows, a long row,
    # ragged N (past 4 rows only where K % 512 != 0 keeps the call off the
    # tensor cores), and M = 33 with K = 256 (the plain kernel)
    if K % group:
        pytest.skip("K not a multiple of the group")
    codes, s, b, x_bits = _problem(bits, group, M, N, K, "bf16", seed=bits + group + M + N)
    Wq = aq.aq_pack(torch.from_numpy(codes).cuda(), bits)
    torch.cuda.synchronize()
    aq.aq_stats(reset=True)
    y = aq.aq_matmul_ex(_x(x_bits, "bf16"), Wq, torch.from_numpy(s).cuda(),
                        torch.from_numpy(b).cuda(), bits, group)
    torch.cuda.synchronize()
    calls = aq.aq_stats()
    assert calls[aq.AQ_VARIANT_GENERIC] == 1 and calls[aq.AQ_VARIANT_TC] == 0, calls
    y_ref, bound = oracle.matmul_g(workloads.to_f64(x_bits, "bf16"), oracle.pack_g(codes, bits),
                                   s, b, bits, group, threads=8)
    assert_within_tolerance(y_to_f64(y, "bf16"), y_ref, bound, f"bits={bits} group={group}")


def test_matmul_ex_unaligned_x_takes_the_plain_kernel():
    # x 2-byte aligned only: the small-M kernel stages x with 16-byte loads,
    # so the call runs on the plain kernel, with the same results
    M, N, K, bits, group = 3, 70, 512, 5, 64
    codes, s, b, x_bits = _problem(bits, group, M, N, K, "fp16", seed=77)
    flat = torch.zeros(M * K + 1, dtype=torch.int16, device="cuda")
    flat[1:] = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16).reshape(-1)).cuda()
    x = flat[1:].view(M, K).view(torch.float16)
    assert x.data_ptr() % 16 != 0
    Wq = aq.aq_pack(torch.from_numpy(codes).cuda(), bits)
    y = aq.aq_matmul_ex(x, Wq, torch.from_numpy(s).cuda(), torch.from_numpy(b).cuda(), bits,
                        group)
    torch.cuda.synchronize()
    y_ref, bound = oracle.matmul_g(workloads.to_f64(x_bits, "fp16"), oracle.pack_g(codes, bits),
                                   s, b, bits, group)
    assert_within_tolerance(y_to_f64(y, "fp16"), y_ref, bound, "unaligned x")
