"""Pins that tie the fp64 oracle to something other than itself.

Each test checks the oracle against values or properties that the format's
definition and plain mathematics fix (mlx-bun pages, @mlx-bun/inference
1.0.0, kernels/quantization/*: the LSB-first 64-value group stream, 2*B words
per group, w = scale*q + bias):

* hand-derived packed words and hand-computed matmul values (tests/golden/);
* an independent bit-by-bit unpacker and an exact rational-arithmetic matmul
  on tiny shapes;
* pack/unpack round trips in both directions;
* closed forms (all-zero codes, zero scales, unit activation rows, all-ones
  activations);
* invariants (permuting whole groups together with x, linearity in x, row
  independence, thread-count independence).

A plausible slip in the oracle (a wrong shift or word index at a straddle, a
dropped bias, a scale read from the wrong group, a transposed operand, a sign
error) breaks at least one of these.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from tests import _golden


# --------------------------------------------------------------------------
# Hand-derived fixtures
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", list(_golden.pack_vectors()), ids=lambda c: c[0])
def test_golden_pack_vectors(case):
    name, bits, K, codes, words = case
    got = oracle.pack(codes[None, :], bits)[0]
    np.testing.assert_array_equal(got, words, err_msg=name)
    back = oracle.unpack(words[None, :], K, bits)[0]
    np.testing.assert_array_equal(back, codes & ((1 << bits) - 1), err_msg=name)


@pytest.mark.parametrize("case", list(_golden.matmul_examples()), ids=lambda c: c[0])
def test_golden_matmul_examples(case):
    name, bits, K, codes, scales, biases, x, y_expected = case
    words = oracle.pack(codes, bits)
    y, bound = oracle.matmul(x[None, :], words, scales, biases, bits)
    # Every value involved is dyadic and small: the fp64 result is exact.
    np.testing.assert_array_equal(y[0], y_expected, err_msg=name)
    assert np.all(bound[0] >= np.abs(y[0]))


# --------------------------------------------------------------------------
# Independent brute force
# --------------------------------------------------------------------------

def _bit_by_bit_codes(words_row, K, bits):
    """Read code v as bits v*B .. v*B+B-1 of the row, one bit at a time."""
    codes = []
    for v in range(K):
        q = 0
        for j in range(bits):
            i = v * bits + j
            q |= ((int(words_row[i // 32]) >> (i % 32)) & 1) << j
        codes.append(q)
    return codes


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("K", [64, 128, 192])
def test_bruteforce_exact(bits, K):
    rng = np.random.default_rng(100 + 10 * bits + K // 64)
    M, N = 3, 4
    G = K // 64
    words = rng.integers(0, 2**32, size=(N, K * bits // 32), dtype=np.uint64).astype(np.uint32)
    scales = rng.standard_normal((N, G)).astype(np.float16).astype(np.float64)
    biases = rng.standard_normal((N, G)).astype(np.float16).astype(np.float64)
    x = rng.standard_normal((M, K)).astype(np.float16).astype(np.float64)
    y, bound = oracle.matmul(x, words, scales, biases, bits)
    for n in range(N):
        q = _bit_by_bit_codes(words[n], K, bits)
        np.testing.assert_array_equal(oracle.unpack(words[n:n + 1], K, bits)[0], q)
        w = [Fraction(scales[n, k // 64]) * q[k] + Fraction(biases[n, k // 64]) for k in range(K)]
        for m in range(M):
            exact = sum(Fraction(x[m, k]) * w[k] for k in range(K))
            mag = sum(abs(Fraction(x[m, k]) * w[k]) for k in range(K))
            # fp64 summation of K terms: |error| <= K * 2^-53 * sum|terms|
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(K, 2**52) * mag
            assert abs(Fraction(bound[m, n]) - mag) <= Fraction(K, 2**52) * mag


def test_dequant_matches_bitwise_codes():
    rng = np.random.default_rng(7)
    for bits in (3, 4):
        K, N = 128, 3
        words = rng.integers(0, 2**32, size=(N, K * bits // 32), dtype=np.uint64).astype(np.uint32)
        s = rng.standard_normal((N, 2)).astype(np.float16)
        b = rng.standard_normal((N, 2)).astype(np.float16)
        W = oracle.dequant(words, s, b, K, bits)
        for n in range(N):
            q = _bit_by_bit_codes(words[n], K, bits)
            for k in range(K):
                assert W[n, k] == float(s[n, k // 64]) * q[k] + float(b[n, k // 64])


# --------------------------------------------------------------------------
# Round trips
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [3, 4])
def test_roundtrip_codes(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(17, 320), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.unpack(oracle.pack(codes, bits), 320, bits), codes)


@pytest.mark.parametrize("bits", [3, 4])
def test_roundtrip_words(bits):
    # Every bit of a row is a code bit (64*B bits = 2*B whole words per group),
    # so unpack followed by pack is the identity on arbitrary words.
    rng = np.random.default_rng(50 + bits)
    words = rng.integers(0, 2**32, size=(5, 512 * bits // 32), dtype=np.uint64).astype(np.uint32)
    np.testing.assert_array_equal(oracle.pack(oracle.unpack(words, 512, bits), bits), words)


@pytest.mark.parametrize("bits", [3, 4])
def test_pack_masks_high_bits(bits):
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 256, size=(3, 128), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.pack(codes, bits),
                                  oracle.pack(codes & ((1 << bits) - 1), bits))


def test_words_per_row():
    assert oracle.words_per_row(64, 3) == 6 and oracle.words_per_row(64, 4) == 8
    assert oracle.words_per_row(5120, 3) == 480 and oracle.words_per_row(8192, 4) == 1024


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.pack(np.zeros((2, 100), np.uint8), 4)  # K not a multiple of 64
    with pytest.raises(ValueError):
        oracle.pack(np.zeros((2, 64), np.uint8), 5)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def _random_problem(bits, M=3, N=5, K=256, seed=0):
    p = workloads.make_problem("pin", bits, N, K, M, "fp16", seed)
    return p, oracle.pack(p.codes, bits)


@pytest.mark.parametrize("bits", [3, 4])
def test_closed_form_zero_codes(bits):
    p, _ = _random_problem(bits)
    words = oracle.pack(np.zeros_like(p.codes), bits)
    x = p.x_f64()
    y, _ = oracle.matmul(x, words, p.scales, p.biases, bits)
    xs = x.reshape(p.M, p.G, 64).sum(axis=2)  # sum of x over each group
    expected = xs @ p.biases.astype(np.float64).T
    np.testing.assert_allclose(y, expected, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bits", [3, 4])
def test_closed_form_zero_scales(bits):
    p, words = _random_problem(bits, seed=1)
    x = p.x_f64()
    y, _ = oracle.matmul(x, words, np.zeros_like(p.scales), p.biases, bits)
    xs = x.reshape(p.M, p.G, 64).sum(axis=2)
    np.testing.assert_allclose(y, xs @ p.biases.astype(np.float64).T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bits", [3, 4])
def test_closed_form_unit_rows(bits):
    # x = e_k reads back exactly one dequantised weight per output.
    p, words = _random_problem(bits, N=4, K=192, seed=2)
    K = p.K
    y, _ = oracle.matmul(np.eye(K), words, p.scales, p.biases, bits)
    s = p.scales.astype(np.float64)
    b = p.biases.astype(np.float64)
    for k in range(K):
        g = k // 64
        np.testing.assert_array_equal(y[k], s[:, g] * p.codes[:, k] + b[:, g])


@pytest.mark.parametrize("bits", [3, 4])
def test_closed_form_ones(bits):
    p, words = _random_problem(bits, seed=3)
    y, _ = oracle.matmul(np.ones((1, p.K)), words, p.scales, p.biases, bits)
    qsum = p.codes.reshape(p.N, p.G, 64).astype(np.int64).sum(axis=2)
    expected = (p.scales.astype(np.float64) * qsum + 64 * p.biases.astype(np.float64)).sum(axis=1)
    np.testing.assert_allclose(y[0], expected, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [3, 4])
def test_group_permutation_equivariance(bits):
    p, words = _random_problem(bits, K=320, seed=4)
    perm = np.random.default_rng(5).permutation(p.G)
    kperm = (perm[:, None] * 64 + np.arange(64)[None, :]).reshape(-1)
    y, bound = oracle.matmul(p.x_f64(), words, p.scales, p.biases, bits)
    words_p = oracle.pack(p.codes[:, kperm], bits)
    y2, _ = oracle.matmul(p.x_f64()[:, kperm], words_p, p.scales[:, perm], p.biases[:, perm], bits)
    assert np.all(np.abs(y - y2) <= 1e-13 * bound + 1e-300)


@pytest.mark.parametrize("bits", [3, 4])
def test_linearity_in_x(bits):
    p, words = _random_problem(bits, seed=6)
    x1 = p.x_f64()
    x2 = np.random.default_rng(8).standard_normal(x1.shape)
    y1, b1 = oracle.matmul(x1, words, p.scales, p.biases, bits)
    y2, b2 = oracle.matmul(x2, words, p.scales, p.biases, bits)
    y12, _ = oracle.matmul(x1 - 2 * x2, words, p.scales, p.biases, bits)
    assert np.all(np.abs(y12 - (y1 - 2 * y2)) <= 1e-12 * (b1 + 2 * b2))


def test_rows_independent_and_threads_identical():
    p, words = _random_problem(4, M=4, N=37, K=256, seed=10)
    x = p.x_f64()
    y, bound = oracle.matmul(x, words, p.scales, p.biases, 4)
    for m in range(p.M):
        ym, _ = oracle.matmul(x[m:m + 1], words, p.scales, p.biases, 4)
        np.testing.assert_array_equal(ym[0], y[m])
    yt, bt = oracle.matmul(x, words, p.scales, p.biases, 4, threads=5)
    np.testing.assert_array_equal(yt, y)
    np.testing.assert_array_equal(bt, bound)
    cols = [36, 0, 17, 17]
    yc, bc = oracle.matmul_cols(x, words, p.scales, p.biases, 4, cols)
    np.testing.assert_array_equal(yc, y[:, cols])
    np.testing.assert_array_equal(bc, bound[:, cols])


def test_bf16_inputs_widen_exactly():
    # The bf16 widening used to feed the oracle is exact: round trip the bits.
    rng = np.random.default_rng(11)
    bits16 = workloads.f32_to_bf16_bits(rng.standard_normal(1000).astype(np.float32))
    back = workloads.f32_to_bf16_bits(workloads.to_f64(bits16, "bf16").astype(np.float32))
    np.testing.assert_array_equal(back, bits16)
    # and matches the definition value = (bits << 16) reinterpreted as float32
    v = workloads.to_f64(np.array([0x3F80, 0xC000, 0x4049], np.uint16), "bf16")
    np.testing.assert_array_equal(v, [1.0, -2.0, 3.140625])
