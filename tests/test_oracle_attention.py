"""Pins for the oracle's decode attention over a quantised KV cache, CPU only.

The oracle computes o = softmax(q . Kd^T) . Vd per query head in fp64, head
h reading KV head h / (H/KV), K and V dequantised as scale * q + bias per
group along d (the operator of the fused decode kernel of the mlx-bun
0.0.4 page, src/model/fused-decode-kernel.ts).  The tests tie it to an
mpmath evaluation at 50 digits over an independent bit-by-bit unpacker, to closed forms (one token,
a zero query), and to invariants (token order, a constant shift of every
score of a head, the grouped-query head mapping), so a wrong head index,
group index, missing max subtraction or normalisation fails one of them.
"""
import numpy as np
import pytest

import oracle

mpmath = pytest.importorskip("mpmath")


def _cache(rng, KV, N, D, bits, group, scale=0.05):
    R = KV * N
    codes = rng.integers(0, 1 << bits, size=(R, D)).astype(np.uint8)
    s = (np.abs(rng.standard_normal((R, D // group))) * scale + 1e-3).astype(np.float16)
    b = (-(1 << (bits - 1)) * s.astype(np.float64) + rng.standard_normal((R, D // group)) * 1e-2
         ).astype(np.float16)
    return codes, s.astype(np.float64), b.astype(np.float64)


def _bitwise_dequant(words, s, b, D, bits, group):
    R = words.shape[0]
    out = np.zeros((R, D), np.float64)
    for r in range(R):
        for d in range(D):
            q = 0
            for i in range(bits):
                bit = d * bits + i
                q |= ((int(words[r, bit // 32]) >> (bit % 32)) & 1) << i
            out[r, d] = s[r, d // group] * q + b[r, d // group]
    return out


def _run(q, kc, ks, kb, vc, vs, vb, KV, N, bits, group):
    return oracle.attention(q, oracle.pack_g(kc, bits), ks, kb, oracle.pack_g(vc, bits), vs, vb,
                            KV, N, bits, group)


@pytest.mark.parametrize("bits,group", [(4, 32), (4, 64), (8, 64), (8, 128)])
def test_mpmath_reference(bits, group):
    rng = np.random.default_rng(bits + group)
    H, KV, N, D = 4, 2, 6, 128
    kc, ks, kb = _cache(rng, KV, N, D, bits, group)
    vc, vs, vb = _cache(rng, KV, N, D, bits, group)
    q = rng.standard_normal((H, D))
    o, _, _ = _run(q, kc, ks, kb, vc, vs, vb, KV, N, bits, group)
    Kd = _bitwise_dequant(oracle.pack_g(kc, bits), ks, kb, D, bits, group)
    Vd = _bitwise_dequant(oracle.pack_g(vc, bits), vs, vb, D, bits, group)
    mpmath.mp.dps = 50
    for h in range(H):
        kv = h // (H // KV)
        sc = [mpmath.fsum(mpmath.mpf(q[h, d]) * mpmath.mpf(Kd[kv * N + n, d]) for d in range(D))
              for n in range(N)]
        e = [mpmath.exp(v) for v in sc]
        den = mpmath.fsum(e)
        for d in range(D):
            ref = mpmath.fsum(e[n] * mpmath.mpf(Vd[kv * N + n, d]) for n in range(N)) / den
            assert abs(o[h, d] - float(ref)) <= 1e-12 * (1 + abs(float(ref)))


def test_single_token_returns_its_value_row():
    rng = np.random.default_rng(1)
    H, KV, N, D, bits, group = 3, 3, 1, 64, 4, 32
    kc, ks, kb = _cache(rng, KV, N, D, bits, group)
    vc, vs, vb = _cache(rng, KV, N, D, bits, group)
    q = rng.standard_normal((H, D)) * 10
    o, _, vmag = _run(q, kc, ks, kb, vc, vs, vb, KV, N, bits, group)
    Vd = _bitwise_dequant(oracle.pack_g(vc, bits), vs, vb, D, bits, group)
    np.testing.assert_array_equal(o, Vd)
    np.testing.assert_array_equal(vmag, np.abs(Vd))


def test_zero_query_averages_the_values():
    rng = np.random.default_rng(2)
    H, KV, N, D, bits, group = 2, 1, 9, 128, 8, 64
    kc, ks, kb = _cache(rng, KV, N, D, bits, group)
    vc, vs, vb = _cache(rng, KV, N, D, bits, group)
    o, smag, _ = _run(np.zeros((H, D)), kc, ks, kb, vc, vs, vb, KV, N, bits, group)
    Vd = _bitwise_dequant(oracle.pack_g(vc, bits), vs, vb, D, bits, group)
    np.testing.assert_allclose(o, np.tile(Vd.mean(axis=0), (H, 1)), rtol=1e-14, atol=1e-15)
    assert np.all(smag == 0)


def test_token_order_does_not_matter():
    rng = np.random.default_rng(3)
    H, KV, N, D, bits, group = 4, 2, 11, 64, 4, 64
    kc, ks, kb = _cache(rng, KV, N, D, bits, group)
    vc, vs, vb = _cache(rng, KV, N, D, bits, group)
    q = rng.standard_normal((H, D)) * 3
    o, _, _ = _run(q, kc, ks, kb, vc, vs, vb, KV, N, bits, group)
    perm = np.concatenate([kv * N + rng.permutation(N) for kv in range(KV)])
    o2, _, _ = _run(q, kc[perm], ks[perm], kb[perm], vc[perm], vs[perm], vb[perm], KV, N, bits,
                    group)
    np.testing.assert_allclose(o2, o, rtol=1e-13, atol=1e-14)


def test_constant_score_shift_cancels():
    # adding c to every key bias of a group adds c * sum(q over the group) to
    # every score of a head alike; the softmax must not move
    rng = np.random.default_rng(4)
    H, KV, N, D, bits, group = 2, 1, 13, 64, 4, 32
    kc, ks, kb = _cache(rng, KV, N, D, bits, group)
    vc, vs, vb = _cache(rng, KV, N, D, bits, group)
    q = rng.standard_normal((H, D))
    o, _, _ = _run(q, kc, ks, kb, vc, vs, vb, KV, N, bits, group)
    o2, _, _ = _run(q, kc, ks, kb + 0.75, vc, vs, vb, KV, N, bits, group)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)


def test_grouped_query_heads_read_their_kv_head():
    rng = np.random.default_rng(5)
    H, KV, N, D, bits, group = 6, 3, 7, 64, 8, 32
    kc, ks, kb = _cache(rng, KV, N, D, bits, group)
    vc, vs, vb = _cache(rng, KV, N, D, bits, group)
    q = rng.standard_normal((H, D))
    o, _, _ = _run(q, kc, ks, kb, vc, vs, vb, KV, N, bits, group)
    rep = H // KV
    for h in range(H):
        kv = h // rep
        sl = slice(kv * N, (kv + 1) * N)
        oh, _, _ = _run(q[h:h + 1], kc[sl], ks[sl], kb[sl], vc[sl], vs[sl], vb[sl], 1, N, bits,
                        group)
        np.testing.assert_array_equal(o[h], oh[0])


def test_attention_rejects_bad_shapes():
    rng = np.random.default_rng(6)
    kc, ks, kb = _cache(rng, 2, 3, 64, 4, 64)
    with pytest.raises(ValueError):  # H not a multiple of KV
        _run(np.zeros((3, 64)), kc, ks, kb, kc, ks, kb, 2, 3, 4, 64)
