"""The Python binding refuses buffers whose size or dtype differs from what
the call reads or writes, before any launch (CPU tensors, no GPU needed)."""
import pytest
import torch

import quantized_matmul_affine_gb300 as aq


def _w(N, K, bits, group):
    return (torch.zeros((N, K * bits // 32), dtype=torch.int32),
            torch.zeros((N, K // group), dtype=torch.float16),
            torch.zeros((N, K // group), dtype=torch.float16))


def test_matmul_checks_weight_and_output_sizes():
    x = torch.zeros((2, 512), dtype=torch.float16)
    Wq, s, b = _w(64, 512, 4, 64)
    with pytest.raises(ValueError, match="Wq holds"):
        aq.aq_matmul(x, Wq[:-1], s, b, 4)
    with pytest.raises(ValueError, match="biases"):
        aq.aq_matmul(x, Wq, s, b[:-1], 4)
    with pytest.raises(ValueError, match="out holds"):
        aq.aq_matmul(x, Wq, s, b, 4, out=torch.zeros((2, 63), dtype=torch.float16))
    with pytest.raises(ValueError, match="out must be"):
        aq.aq_matmul(x, Wq, s, b, 4, out=torch.zeros((2, 64), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA tensor"):   # sizes right: reaches the device check
        aq.aq_matmul(x, Wq, s, b, 4)


def test_matmul_ex_checks_sizes_for_its_width_and_group():
    x = torch.zeros((1, 384), dtype=torch.bfloat16)
    Wq, s, b = _w(10, 384, 6, 128)
    with pytest.raises(ValueError, match="scales must be"):
        aq.aq_matmul_ex(x, Wq, s.float(), b, 6, 128)
    with pytest.raises(ValueError, match="Wq holds"):
        aq.aq_matmul_ex(x, Wq, s, b, 5, 128)        # the words of 6 bits, not 5
    with pytest.raises(ValueError, match="CUDA tensor"):
        aq.aq_matmul_ex(x, Wq, s, b, 6, 128)


def test_attention_checks_every_cache_tensor():
    H, KV, N, D, bits, group = 4, 2, 10, 64, 4, 32
    q = torch.zeros((H, D), dtype=torch.bfloat16)

    def cache(n):
        return (torch.zeros((KV, n, D * bits // 32), dtype=torch.int32),
                torch.zeros((KV, n, D // group), dtype=torch.float16),
                torch.zeros((KV, n, D // group), dtype=torch.float16))

    with pytest.raises(ValueError, match="v_words"):
        aq.aq_attention_decode(q, cache(N), cache(N - 1), bits, group)
    k = cache(N)
    with pytest.raises(ValueError, match="k_biases"):
        aq.aq_attention_decode(q, (k[0], k[1], k[2][:, :-1]), cache(N), bits, group)
    with pytest.raises(ValueError, match="q must be"):
        aq.aq_attention_decode(q.float(), cache(N), cache(N), bits, group)
    with pytest.raises(ValueError, match="out holds"):
        aq.aq_attention_decode(q, cache(N), cache(N), bits, group,
                               out=torch.zeros((H, D - 1), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA tensor"):
        aq.aq_attention_decode(q, cache(N), cache(N), bits, group)


def test_multi_and_gate_up_check_each_projection():
    x = torch.zeros((1, 512), dtype=torch.bfloat16)
    a, b = _w(64, 512, 4, 64), _w(32, 512, 4, 64)
    with pytest.raises(ValueError, match=r"Wq\[1\]"):
        aq.aq_matmul_multi(x, [a, (b[0][:-1], b[1], b[2])], 4)
    with pytest.raises(ValueError, match="one output per projection"):
        aq.aq_matmul_multi(x, [a, b], 4, outs=[torch.zeros((1, 64), dtype=torch.bfloat16)])
    with pytest.raises(ValueError, match=r"scales \(up\)"):
        aq.aq_matmul_gate_up(x, a, (a[0], a[1][:-1], a[2]), 4)


def test_pack_checks_the_words_buffer():
    codes = torch.zeros((4, 64), dtype=torch.uint8)
    with pytest.raises(ValueError, match="words holds"):
        aq.aq_pack(codes, 3, words=torch.zeros((4, 5), dtype=torch.int32))


def test_attention_wants_three_dimensional_caches():
    q = torch.zeros((4, 64), dtype=torch.bfloat16)
    flat = (torch.zeros((20, 8), dtype=torch.int32), torch.zeros((20, 2), dtype=torch.float16),
            torch.zeros((20, 2), dtype=torch.float16))
    with pytest.raises(ValueError, match=r"\[KV, N"):
        aq.aq_attention_decode(q, flat, flat, 4, 32)
