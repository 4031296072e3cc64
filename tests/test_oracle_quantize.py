"""Pins for the oracle's quantiser (float weights -> affine group-64 codes,
fp16 scale and bias), CPU only.

The pages fix the stored format and w = scale*q + bias but not the
quantiser's rounding rules; the oracle takes the plain reading (min/max per
group, scale = (max - min) / (2^B - 1), bias = min, both rounded to fp16,
q = clamp(rint((w - bias) / scale))).  These tests tie it to things outside
itself:

* its binary16 conversions against numpy's IEEE conversions, on every fp16
  value, every midpoint between neighbours and the values just around them;
* exact recovery of (codes, scale, bias) from weights built as s*q + b with
  a power-of-two scale and both end codes present in every group;
* the nearest-level property by brute force over all 2^B levels;
* closed forms (a constant group) and the error bound of the levels.

A slip such as a code taken from the wrong group, an unrounded scale, a
biased rounding or a wrong clamp breaks one of them.
"""
import numpy as np
import pytest

import oracle


def _all_finite_f16() -> np.ndarray:
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    return np.concatenate([h, h | 0x8000])


def test_f16_to_f32_exact_on_every_pattern():
    h = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_bits_to_f32(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_f32_to_f16_matches_ieee_rne():
    f = _all_finite_f16().view(np.float16).astype(np.float64)
    pos = np.sort(np.unique(np.abs(f)))
    mids = (pos[:-1] + pos[1:]) / 2  # ties: must go to the even neighbour
    vals = np.concatenate([f, mids, -mids, [65504.0, 65519.0, 65520.0, 1e9, 2.0**-26, 2.0**-25]])
    v32 = vals.astype(np.float32)
    # the float32 just below and above each value (breaks ties the other way)
    v32 = np.concatenate([v32, np.nextafter(v32, np.float32(np.inf)),
                          np.nextafter(v32, np.float32(-np.inf))])
    with np.errstate(over="ignore"):
        want = v32.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16_bits(v32)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(v32[i]), int(got[i]), int(want[i])) for i in bad[:5]]


@pytest.mark.parametrize("bits", [3, 4])
def test_exact_recovery(bits):
    # w = s*q + b with s = 2^-e, b on the same grid, codes 0 and 2^B - 1 in
    # every group: max - min = (2^B - 1) s exactly, so the quantiser must give
    # back s, b and the codes themselves.
    rng = np.random.default_rng(bits)
    N, K = 5, 320
    qmax = (1 << bits) - 1
    codes = rng.integers(0, qmax + 1, size=(N, K)).astype(np.uint8)
    codes[:, ::64] = 0
    codes[:, 1::64] = qmax
    e = rng.integers(3, 9, size=(N, K // 64))
    s = 2.0 ** (-e.astype(np.float64))
    b = rng.integers(-64, 64, size=(N, K // 64)) * s
    w = (s[:, np.arange(K) // 64] * codes + b[:, np.arange(K) // 64]).astype(np.float32)
    assert np.array_equal(w.astype(np.float16).astype(np.float32), w)  # fp16 weights
    got_q, sb, bb = oracle.quantize(w, bits)
    assert np.array_equal(got_q, codes)
    assert np.array_equal(sb, s.astype(np.float16).view(np.uint16))
    assert np.array_equal(bb, b.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("bits", [3, 4])
def test_constant_group(bits):
    w = np.full((2, 128), 0.3125, np.float32)
    w[1, 64:] = -7.0
    q, sb, bb = oracle.quantize(w, bits)
    assert np.all(q == 0)
    assert np.all(sb == 0)
    assert bb[0, 0] == bb[0, 1] == np.float16(0.3125).view(np.uint16)
    assert bb[1, 1] == np.float16(-7.0).view(np.uint16)


def _levels(sb, bb, bits):
    s = sb.view(np.float16).astype(np.float64)
    b = bb.view(np.float16).astype(np.float64)
    lv = np.arange(1 << bits, dtype=np.float64)
    return s, b, lv


@pytest.mark.parametrize("dtype", [np.float16, "bf16"])
@pytest.mark.parametrize("bits", [3, 4])
def test_nearest_level_bruteforce(bits, dtype):
    rng = np.random.default_rng(10 + bits)
    N, K = 7, 256
    w = (rng.standard_normal((N, K)) * rng.uniform(0.01, 3, size=(N, 1))).astype(np.float32)
    if dtype == "bf16":
        w = (w.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)  # bf16 values
    else:
        w = w.astype(np.float16).astype(np.float32)
    q, sb, bb = oracle.quantize(w, bits)
    s, b, lv = _levels(sb, bb, bits)
    G = K // 64
    for n in range(N):
        for g in range(G):
            wg = w[n, 64 * g:64 * g + 64].astype(np.float64)
            dist = np.abs(s[n, g] * lv[None, :] + b[n, g] - wg[:, None])  # [64, levels]
            chosen = dist[np.arange(64), q[n, 64 * g:64 * g + 64]]
            # the chosen level is a nearest one (single-precision ties aside)
            assert np.all(chosen <= dist.min(axis=1) + s[n, g] * 2.0**-18), (n, g)


@pytest.mark.parametrize("bits", [3, 4])
def test_error_bound(bits):
    rng = np.random.default_rng(20 + bits)
    N, K = 16, 512
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float16).astype(np.float32)
    q, sb, bb = oracle.quantize(w, bits)
    s, b, _ = _levels(sb, bb, bits)
    G = K // 64
    qmax = (1 << bits) - 1
    wh = w.astype(np.float64)
    lo = wh.reshape(N, G, 64).min(axis=2)
    hi = wh.reshape(N, G, 64).max(axis=2)
    # the levels cover [b, b + qmax s]; fp16 rounding of s and b moves the
    # ends by at most |hi - (b + qmax s)| and |lo - b|
    slack = np.maximum(np.abs(hi - (b + qmax * s)), np.abs(lo - b))
    deq = oracle.dequant(oracle.pack(q, bits), s, b, K, bits)
    err = np.abs(deq - wh).reshape(N, G, 64).max(axis=2)
    assert np.all(err <= s / 2 + slack + s * 2.0**-18)
    assert np.all(q <= qmax)


def test_quantize_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((2, 100), np.float32), 4)
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((2, 64), np.float32), 5)
