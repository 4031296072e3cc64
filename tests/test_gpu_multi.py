"""GPU parity of the fused multi-projection calls against the fp64 oracle,
through the C ABI.

aq_matmul_multi: every projection's y within the matmul tolerance
|y - y_ref| <= 2e-3 * sum_k |x_k w_nk| + 1e-5.

aq_matmul_gate_up: h = silu(g) * u with g, u the gate and up products, against
oracle.gate_up (the float64 operator, pinned in tests/test_oracle_gate_up.py).  With
tg, tu the matmul tolerances of g and u and |silu'| <= 1.1,
|h - h_ref| <= 1.1 tg (|u| + tu) + (|silu(g)| + 1.1 tg) tu, plus one rounding
of h to the output type (2^-8 relative for bf16, 2^-11 for fp16).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._gpu import assert_within_tolerance, dev_tensors, y_to_f64

pytestmark = pytest.mark.gpu

aq = pytest.importorskip("quantized_matmul_affine_gb300")


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    aq.aq_device_error(clear=True)
    yield
    assert aq.aq_device_error() == 0


def _problems(bits, Ns, K, M, dtype, seed):
    """One problem per projection, all with the same x (drawn with the first)."""
    ps = [workloads.make_problem("m", bits, n, K, M, dtype, seed=seed + 17 * j)
          for j, n in enumerate(Ns)]
    return ps, ps[0].x_bits


def _weights(p):
    codes, s, b, _ = dev_tensors(p)
    return aq.aq_pack(codes, p.bits), s, b


def _x(x_bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def _ref(p, x_bits, dtype, cols=None):
    x = workloads.to_f64(x_bits, dtype)
    words = oracle.pack(p.codes, p.bits)
    if cols is None:
        return oracle.matmul(x, words, p.scales, p.biases, p.bits, threads=8)
    return oracle.matmul_cols(x, words, p.scales, p.biases, p.bits, cols)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("Ns,K,M", [
    ((300, 64, 100), 1024, 1),        # q, k, v in miniature
    ((257, 33, 1000, 5), 512, 5),     # four projections, ragged rows
    ((700, 700), 2048, 12),           # two column blocks
    ((96, 3000), 1536, 24),           # four column blocks
    ((20000, 4000), 512, 2),          # several passes per CTA
    ((128,), 1024, 3),                # one projection: as aq_matmul
    ((300, 64), 1024, 40),            # M > 32: one launch per projection
    ((300, 64), 576, 1),              # K % 512 != 0: one launch per projection
])
def test_multi_parity(Ns, K, M, bits, dtype):
    ps, x_bits = _problems(bits, Ns, K, M, dtype, seed=sum(Ns) + K + M + bits)
    x = _x(x_bits, dtype)
    ys = aq.aq_matmul_multi(x, [_weights(p) for p in ps], bits)
    torch.cuda.synchronize()
    for j, (p, y) in enumerate(zip(ps, ys)):
        y_ref, bound = _ref(p, x_bits, dtype)
        assert_within_tolerance(y_to_f64(y, dtype), y_ref, bound, f"projection {j} of {Ns}")


def test_multi_matches_single_calls_bitwise():
    # the same kernel arithmetic per projection: identical bits to aq_matmul
    # on a shape that aq_matmul also sends to the resident kernel
    ps, x_bits = _problems(4, (512, 200), 2048, 1, "bf16", seed=3)
    x = _x(x_bits, "bf16")
    ws = [_weights(p) for p in ps]
    ys = aq.aq_matmul_multi(x, ws, 4)
    singles = [aq.aq_matmul_bf16(x, *w, 4) for w in ws]
    torch.cuda.synchronize()
    assert aq.aq_select(1, 512, 2048, 4, aq.AQ_BF16) == aq.AQ_VARIANT_GEMV
    for y, z in zip(ys, singles):
        assert torch.equal(y.view(torch.int16), z.view(torch.int16))


def _check_gate_up(h, pg, pu, x_bits, dtype, cols=None):
    x = workloads.to_f64(x_bits, dtype)
    r = oracle.gate_up(x, (oracle.pack(pg.codes, pg.bits), pg.scales, pg.biases),
                       (oracle.pack(pu.codes, pu.bits), pu.scales, pu.biases), pg.bits, cols)
    h_ref, u, s = r["h"], r["u"], r["silu"]
    tg, tu = oracle.tolerance(r["bound_g"]), oracle.tolerance(r["bound_u"])
    e1 = 1.1 * tg * (np.abs(u) + tu) + (np.abs(s) + 1.1 * tg) * tu
    rnd = 2.0**-8 if dtype == "bf16" else 2.0**-11
    tol = e1 + rnd * (np.abs(h_ref) + e1) + 1e-7
    err = np.abs(h - h_ref)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, [(int(i), int(j), float(h[i, j]), float(h_ref[i, j]), float(tol[i, j]))
                           for i, j in bad[:4]]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("N,K,M", [(100, 512, 1), (700, 2048, 3), (3000, 1024, 9),
                                   (1000, 1536, 20), (19456, 512, 1)])
def test_gate_up_parity(N, K, M, bits, dtype):
    (pg, pu), x_bits = _problems(bits, (N, N), K, M, dtype, seed=N + K + M)
    x = _x(x_bits, dtype)
    h = aq.aq_matmul_gate_up(x, _weights(pg), _weights(pu), bits)
    torch.cuda.synchronize()
    _check_gate_up(y_to_f64(h, dtype), pg, pu, x_bits, dtype)


def test_gate_up_layer_shape_sampled():
    # the 13824 x 5120 gate/up pair of the decoder-layer workload, one bf16 row
    (pg, pu), x_bits = _problems(4, (13824, 13824), 5120, 1, "bf16", seed=34)
    x = _x(x_bits, "bf16")
    h = aq.aq_matmul_gate_up(x, _weights(pg), _weights(pu), 4)
    torch.cuda.synchronize()
    cols = np.random.default_rng(0).choice(13824, 512, replace=False)
    _check_gate_up(y_to_f64(h, "bf16")[:, cols], pg, pu, x_bits, "bf16", cols)


def test_gate_up_unsupported_queues_nothing():
    (pg, pu), x_bits = _problems(4, (64, 64), 512, 40, "bf16", seed=1)
    x = _x(x_bits, "bf16")
    out = torch.full((40, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(aq.AqError) as e:
        aq.aq_matmul_gate_up(x, _weights(pg), _weights(pu), 4, out=out)
    assert e.value.status == 2
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
