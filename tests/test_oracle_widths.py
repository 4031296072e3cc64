"""Pins for the oracle's other code widths (2, 3, 4, 5, 6, 8 bits) and group
sizes (32, 64, 128), CPU only.

The bit stream is the one of the 3/4-bit format (mlx-bun pages,
affine-split-mma.ts helper affine_unit: code v at bits [v*B, v*B+B) of the
row's LSB-first stream); scales and biases come one per group.  These tests
tie the general functions to hand-derived words, an independent bit-by-bit
unpacker, exact rational arithmetic, closed forms and the quantiser's exact
recovery, so a wrong straddle, a group index taken with the wrong group size
or a dropped bias fails one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import _golden

WIDTHS = [2, 3, 4, 5, 6, 8]
GROUPS = [32, 64, 128]


@pytest.mark.parametrize("case", list(_golden.pack_vectors("pack_vectors_widths.txt")),
                         ids=lambda c: c[0])
def test_golden_words(case):
    name, bits, K, codes, words = case
    got = oracle.pack_g(codes[None, :], bits)[0]
    assert np.array_equal(got, words), (name, [hex(w) for w in got])


def _unpack_bitwise(words, K, bits):
    # independent: walk the stream one bit at a time
    out = np.zeros(K, np.uint8)
    for v in range(K):
        q = 0
        for i in range(bits):
            b = v * bits + i
            q |= ((int(words[b // 32]) >> (b % 32)) & 1) << i
        out[v] = q
    return out


@pytest.mark.parametrize("bits", WIDTHS)
def test_bitwise_unpack_and_round_trip(bits):
    rng = np.random.default_rng(bits)
    K = 160
    codes = rng.integers(0, 256, size=(3, K)).astype(np.uint8)
    words = oracle.pack_g(codes, bits)
    masked = codes & np.uint8((1 << bits) - 1)
    for n in range(3):
        assert np.array_equal(_unpack_bitwise(words[n], K, bits), masked[n])
    assert np.array_equal(oracle.unpack_g(words, K, bits), masked)
    assert np.array_equal(oracle.pack_g(oracle.unpack_g(words, K, bits), bits), words)


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", [2, 5, 8])
def test_bruteforce_exact(bits, group):
    rng = np.random.default_rng(bits * 1000 + group)
    M, N, K = 2, 3, 2 * group
    G = K // group
    codes = rng.integers(0, 1 << bits, size=(N, K)).astype(np.uint8)
    s = rng.integers(1, 64, size=(N, G)) / 256.0
    b = rng.integers(-64, 64, size=(N, G)) / 128.0
    x = rng.integers(-8, 8, size=(M, K)) / 4.0
    y, _ = oracle.matmul_g(x, oracle.pack_g(codes, bits), s, b, bits, group)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                g = k // group
                w = Fraction(s[n, g]) * int(codes[n, k]) + Fraction(b[n, g])
                acc += Fraction(x[m, k]) * w
            assert y[m, n] == float(acc)


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", WIDTHS)
def test_zero_codes_closed_form(bits, group):
    rng = np.random.default_rng(7)
    M, N, K = 3, 4, 384
    G = K // group
    x = rng.standard_normal((M, K))
    b = rng.standard_normal((N, G))
    s = rng.standard_normal((N, G))
    words = oracle.pack_g(np.zeros((N, K), np.uint8), bits)
    y, _ = oracle.matmul_g(x, words, s, b, bits, group)
    xs = x.reshape(M, G, group).sum(axis=2)
    np.testing.assert_allclose(y, xs @ b.T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", WIDTHS)
def test_dequant_matches_codes(bits, group):
    rng = np.random.default_rng(bits + group)
    N, K = 3, 256
    codes = rng.integers(0, 1 << bits, size=(N, K)).astype(np.uint8)
    s = rng.standard_normal((N, K // group))
    b = rng.standard_normal((N, K // group))
    W = oracle.dequant_g(oracle.pack_g(codes, bits), s, b, K, bits, group)
    g = np.arange(K) // group
    np.testing.assert_array_equal(W, s[:, g] * codes + b[:, g])


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", WIDTHS)
def test_quantize_exact_recovery(bits, group):
    rng = np.random.default_rng(100 + bits + group)
    N, K = 3, 2 * group
    qmax = (1 << bits) - 1
    codes = rng.integers(0, qmax + 1, size=(N, K)).astype(np.uint8)
    codes[:, ::group] = 0
    codes[:, 1::group] = qmax
    e = rng.integers(4, 9, size=(N, K // group))
    s = 2.0 ** (-e.astype(np.float64))
    b = rng.integers(-16, 16, size=(N, K // group)) * s
    g = np.arange(K) // group
    w = (s[:, g] * codes + b[:, g]).astype(np.float32)
    assert np.array_equal(w.astype(np.float16).astype(np.float32), w)
    q, sb, bb = oracle.quantize_g(w, bits, group)
    assert np.array_equal(q, codes)
    assert np.array_equal(sb, s.astype(np.float16).view(np.uint16))
    assert np.array_equal(bb, b.astype(np.float16).view(np.uint16))


def test_group64_equals_the_format_functions():
    # the 3/4-bit group-64 entry points and the general ones agree
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, size=(4, 256)).astype(np.uint8)
    for bits in (3, 4):
        c = codes & np.uint8((1 << bits) - 1)
        assert np.array_equal(oracle.pack(c, bits), oracle.pack_g(c, bits))
    w = rng.standard_normal((4, 256)).astype(np.float16).astype(np.float32)
    a = oracle.quantize(w, 4)
    bq = oracle.quantize_g(w, 4, 64)
    for u, v in zip(a, bq):
        assert np.array_equal(u, v)


def test_general_functions_reject_bad_shapes():
    with pytest.raises(ValueError):
        oracle.pack_g(np.zeros((1, 48), np.uint8), 4)      # K not a multiple of 32
    with pytest.raises(ValueError):
        oracle.pack_g(np.zeros((1, 32), np.uint8), 7)      # width outside the set
    with pytest.raises(ValueError):
        oracle.quantize_g(np.zeros((1, 64), np.float32), 4, 48)  # group size outside the set
