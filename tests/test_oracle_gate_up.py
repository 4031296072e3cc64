"""Pins for the oracle's gated MLP input h = silu(g) * u (oracle.gate_up).

The operator is the gate/up epilogue of the mlx-bun 0.4.0 -> 1.0.0 page
(src/model/trellis-shared-m.ts): sigmoid(gate) = 1 / (1 + exp(-gate)),
silu = gate * sigmoid, h = silu * up, with gate and up the two affine
group-64 products of the same activations.  The checks here hold by
mathematics, not by the oracle's own code:

* hand-computed values (tests/golden/gate_up_examples.txt) from published
  constants of the exponential, including both large-argument limits (a wrong
  sign in the exponent fails them);
* closed forms: all-zero up weights give h = 0; all-zero gate weights give
  silu(0) = 0, so h = 0;
* the odd part of SiLU: silu(g) - silu(-g) = g, so negating every gate scale
  and bias (which negates g exactly) changes h by exactly g * u (an exchange
  of the gate and up operands fails this);
* g and u equal the pinned matmul oracle on the gate and up weights.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests import _golden


def _weights(codes, scales, biases, bits):
    return oracle.pack(codes, bits), scales, biases


@pytest.mark.parametrize("case", list(_golden.gate_up_examples()), ids=lambda c: c[0])
def test_golden_gate_up_examples(case):
    name, bits, K, (gc, gs, gb), (uc, us, ub), x, h_expected = case
    r = oracle.gate_up(x[None, :], _weights(gc, gs, gb, bits), _weights(uc, us, ub, bits), bits)
    h = r["h"][0, 0]
    if h_expected == 0.0:
        assert h == 0.0, name
    else:
        assert abs(h - h_expected) <= 1e-14 * abs(h_expected), (name, h, h_expected)


def _problem(bits, N, K, M, dtype, seed):
    pg = workloads.make_problem("g", bits, N, K, M, dtype, seed=seed)
    pu = workloads.make_problem("u", bits, N, K, M, dtype, seed=seed + 1)
    return pg, pu, pg.x_f64()


def _w(p):
    return oracle.pack(p.codes, p.bits), p.scales, p.biases


@pytest.mark.parametrize("bits", [3, 4])
def test_zero_up_weights_give_zero(bits):
    pg, pu, x = _problem(bits, 7, 192, 3, "bf16", seed=11)
    zero = np.zeros_like(pu.codes)
    up = (oracle.pack(zero, bits), pu.scales, np.zeros_like(pu.biases))
    r = oracle.gate_up(x, _w(pg), up, bits)
    assert np.all(r["u"] == 0.0)
    assert np.all(r["h"] == 0.0)
    assert np.any(r["g"] != 0.0)


@pytest.mark.parametrize("bits", [3, 4])
def test_zero_gate_weights_give_zero(bits):
    pg, pu, x = _problem(bits, 5, 128, 2, "fp16", seed=12)
    gate = (oracle.pack(np.zeros_like(pg.codes), bits), pg.scales, np.zeros_like(pg.biases))
    r = oracle.gate_up(x, gate, _w(pu), bits)
    assert np.all(r["g"] == 0.0)
    assert np.all(r["silu"] == 0.0)
    assert np.all(r["h"] == 0.0)


@pytest.mark.parametrize("bits", [3, 4])
def test_odd_part_of_silu(bits):
    # negating the gate scales and biases negates g exactly; silu(g) - silu(-g) = g
    pg, pu, x = _problem(bits, 9, 256, 4, "bf16", seed=13)
    r = oracle.gate_up(x, _w(pg), _w(pu), bits)
    neg = (oracle.pack(pg.codes, bits), -pg.scales, -pg.biases)
    rn = oracle.gate_up(x, neg, _w(pu), bits)
    np.testing.assert_array_equal(rn["g"], -r["g"])
    g, u = r["g"], r["u"]
    diff = r["h"] - rn["h"]
    scale = (np.abs(g) + 1.0) * np.abs(u) + 1e-300
    assert np.all(np.abs(diff - g * u) <= 1e-13 * scale)
    # and the sigmoid's own symmetry: silu(g) + silu(-g) = g * tanh(g / 2)
    assert np.all(np.abs(r["silu"] + rn["silu"] - g * np.tanh(g / 2)) <= 1e-13 * (np.abs(g) + 1))


@pytest.mark.parametrize("bits", [3, 4])
def test_products_are_the_matmul_oracle(bits):
    pg, pu, x = _problem(bits, 33, 320, 3, "fp16", seed=14)
    r = oracle.gate_up(x, _w(pg), _w(pu), bits)
    g, bg = oracle.matmul(x, *_w(pg), bits)
    u, bu = oracle.matmul(x, *_w(pu), bits)
    np.testing.assert_array_equal(r["g"], g)
    np.testing.assert_array_equal(r["u"], u)
    np.testing.assert_array_equal(r["bound_g"], bg)
    np.testing.assert_array_equal(r["bound_u"], bu)


def test_columns_match_full():
    pg, pu, x = _problem(4, 40, 256, 2, "bf16", seed=15)
    full = oracle.gate_up(x, _w(pg), _w(pu), 4)
    cols = np.array([39, 0, 17, 17, 5])
    part = oracle.gate_up(x, _w(pg), _w(pu), 4, cols=cols)
    for k in ("h", "g", "u", "silu", "bound_g", "bound_u"):
        np.testing.assert_array_equal(part[k], full[k][:, cols])
