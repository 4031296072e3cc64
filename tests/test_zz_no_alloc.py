"""aq_attention_decode_static, the entry point that allocates nothing: the
several-cluster attention plan with the library's fixed scratch in place of
a caller workspace.  It must give the same bits as aq_attention_decode_ws
with a workspace of the size that plan asks for, call after call (the
counters at the start of the scratch return to zero after each call), and
refuse plans whose workspace exceeds the scratch.

This file is collected last, so that it runs both alone and after every
other test has used the library in the same process."""
import os
import re

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

aq = pytest.importorskip("quantized_matmul_affine_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _scratch_bytes():
    text = open(os.path.join(ROOT, "include", "aq.h")).read()
    return int(re.search(r"#define AQ_ATTENTION_STATIC_SCRATCH_BYTES (\d+)", text).group(1))


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _problem(H, KV, N, D, bits, group, seed):
    rng = np.random.default_rng(seed)
    R, G = KV * N, D // group

    def side():
        codes = rng.integers(0, 1 << bits, size=(R, D), dtype=np.uint8)
        s = (np.abs(rng.standard_normal((R, G))) * (0.16 / (1 << bits)) + 1e-3).astype(np.float16)
        b = (-(1 << (bits - 1)) * s.astype(np.float64)).astype(np.float16)
        return (aq.aq_pack(torch.from_numpy(codes).cuda(), bits).view(KV, N, D * bits // 32),
                torch.from_numpy(s).cuda().view(KV, N, G), torch.from_numpy(b).cuda().view(KV, N, G))

    k, v = side(), side()
    q = (torch.from_numpy(rng.standard_normal((H, D)).astype(np.float32)) * 2).to(
        torch.bfloat16).cuda()
    return q, k, v


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_static_scratch_matches_the_workspace_path_two_calls_in_a_row():
    H, KV, N, D, bits, group = 16, 8, 32768, 256, 4, 64  # several clusters a KV head
    need = aq.aq_attention_workspace_bytes(H, KV, N, D, bits, group)
    assert 0 < need <= _scratch_bytes()
    q, k, v = _problem(H, KV, N, D, bits, group, seed=1)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    got, want = [], []
    for _ in range(2):
        want.append(aq.aq_attention_decode_ws(q, k, v, bits, group, workspace=ws))
        got.append(aq.aq_attention_decode_static(q, k, v, bits, group))
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        assert _same(g, w)
    assert _same(got[0], got[1])
    assert aq.aq_device_error() == 0


def test_static_scratch_one_cluster_plan_is_aq_attention_decode():
    H, KV, N, D, bits, group = 16, 8, 2048, 256, 4, 64  # one cluster a KV head
    assert aq.aq_attention_workspace_bytes(H, KV, N, D, bits, group) == 0
    q, k, v = _problem(H, KV, N, D, bits, group, seed=2)
    got = [aq.aq_attention_decode_static(q, k, v, bits, group) for _ in range(2)]
    want = aq.aq_attention_decode(q, k, v, bits, group)
    torch.cuda.synchronize()
    assert _same(got[0], want) and _same(got[1], want)


def test_static_scratch_refuses_a_larger_workspace():
    cap = _scratch_bytes()
    for H, KV, N, D in [(64, 8, 65536, 512), (64, 8, 262144, 512), (32, 4, 262144, 512)]:
        need = aq.aq_attention_workspace_bytes(H, KV, N, D, 4, 64)
        if need > cap:
            break
    else:
        pytest.skip("no plan on this device needs more than the static scratch")
    # refused before anything is read or queued: small placeholder tensors
    q = torch.zeros((H, D), dtype=torch.bfloat16, device="cuda")
    words = torch.zeros((KV, N, D // 8), dtype=torch.int32, device="cuda")
    sb = torch.zeros((KV, N, D // 64), dtype=torch.float16, device="cuda")
    with pytest.raises(aq.AqError) as e:
        aq.aq_attention_decode_static(q, (words, sb, sb), (words, sb, sb), 4, 64)
    assert e.value.status == 2  # AQ_ERR_UNSUPPORTED
