"""GPU parity of the quantiser (aq_quantize / aq_quantize_bf16) against the
oracle's quantiser, through the C ABI: codes (packed words), scales and
biases bit-exact.  Both sides decide the codes in single precision with the
same operations, so the integer decisions agree exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

aq = pytest.importorskip("quantized_matmul_affine_gb300")


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _device_weights(bits16: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits16).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def _check(vals: np.ndarray, bits16: np.ndarray, dtype: str, bits: int, what: str):
    q = aq.aq_quantize_bf16 if dtype == "bf16" else aq.aq_quantize
    Wq, s, b = q(_device_weights(bits16, dtype), bits)
    torch.cuda.synchronize()
    codes, sb, bb = oracle.quantize(vals, bits)
    got_w = Wq.cpu().numpy().view(np.uint32)
    want_w = oracle.pack(codes, bits)
    got_s = s.cpu().numpy().view(np.uint16)
    got_b = b.cpu().numpy().view(np.uint16)
    for name, got, want in (("scales", got_s, sb), ("biases", got_b, bb), ("words", got_w, want_w)):
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{what}: {name} differ at {bad[:4].tolist()} ({len(bad)} total)"


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("N,K", [(1, 64), (3, 192), (37, 576), (300, 1024), (5, 4096),
                                 (1000, 320)])
def test_quantize_bit_exact(N, K, bits, dtype):
    # ragged group counts (N*K/64 not a multiple of the four groups a warp takes)
    b16, vals = workloads.make_weights(N, K, dtype, seed=N + K + bits)
    _check(vals, b16, dtype, bits, f"{N}x{K} bits={bits} {dtype}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
def test_quantize_special_groups(bits, dtype):
    # constant groups, exact power-of-two grids, a group spanning zero, wide
    # and tiny ranges, ties in (w - bias) / scale
    K = 64 * 8
    rng = np.random.default_rng(7)
    qmax = (1 << bits) - 1
    rows = []
    rows.append(np.full(K, 0.5))
    grid = rng.integers(0, qmax + 1, size=K).astype(np.float64)
    grid[::64] = 0
    grid[1::64] = qmax
    rows.append(grid * 2.0**-5 - 1.0)
    rows.append(np.linspace(-3, 3, K))
    rows.append(rng.standard_normal(K) * 100)
    rows.append(rng.standard_normal(K) * 1e-3)
    half = (np.arange(K) % (2 * qmax + 1)) * 0.5 * 2.0**-4  # multiples of half a level
    half[::64] = 0
    half[1::64] = qmax * 2.0**-4
    rows.append(half)
    w = np.stack(rows).astype(np.float32)
    conv = workloads.f32_to_bf16_bits if dtype == "bf16" else workloads.f32_to_fp16_bits
    b16 = conv(w)
    vals = workloads.to_f64(b16, dtype).astype(np.float32)
    _check(vals, b16, dtype, bits, "special groups")


@pytest.mark.parametrize("index", range(len(workloads.QUANTIZE_WORKLOADS["quantize"])))
def test_quantize_workloads_full_size(index):
    # every group of the full-size shapes the benchmark times
    bits, N, K, dtype, seed = workloads.QUANTIZE_WORKLOADS["quantize"][index]
    b16, vals = workloads.make_weights(N, K, dtype, seed)
    _check(vals, b16, dtype, bits, f"quantize[{index}]")


@pytest.mark.parametrize("bits", [3, 4])
def test_quantize_then_matmul(bits):
    # quantised weights go straight into the matmul; the result equals the
    # oracle's matmul on the oracle's quantisation
    N, K, M = 200, 1024, 3
    b16, vals = workloads.make_weights(N, K, "bf16", seed=99)
    Wq, s, b = aq.aq_quantize_bf16(_device_weights(b16, "bf16"), bits)
    x_bits = workloads.make_x(M, K, "bf16", seed=5)
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    y = aq.aq_matmul_bf16(x, Wq, s, b, bits)
    torch.cuda.synchronize()
    codes, sb, bb = oracle.quantize(vals, bits)
    y_ref, bound = oracle.matmul(workloads.to_f64(x_bits, "bf16"), oracle.pack(codes, bits),
                                 sb.view(np.float16), bb.view(np.float16), bits)
    got = workloads.to_f64(y.view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    assert np.all(np.abs(got - y_ref) <= oracle.tolerance(bound))
