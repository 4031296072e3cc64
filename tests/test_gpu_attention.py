"""GPU parity of decode attention over a quantised KV cache
(aq_attention_decode) against the fp64 oracle, through the C ABI.

Tolerance per output element: the GPU keeps the scores in fp32, so a score
is off by at most tau = 1e-4 * sum_d |q k| + 1e-5 (two orders above fp32
rounding); a softmax weight then moves by a factor within exp(+-2 tau),
giving |o - o_ref| <= (exp(2 max tau) - 1) * sum_n p |v|, plus fp32
accumulation over the rows (2^-24 per row), plus one rounding of o to the
output type (2^-8 relative bf16, 2^-11 fp16).  The value product takes
p * scale as fp16 (the pages' kernel rounds even the scores to the input
type): 2^-11 relative per term of sum_n p |scale * code|, which is at most
sum_n p |v| + max_n |bias| of the group; 2^-10 of that is allowed.
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


def _cache(rng, KV, N, D, bits, group, ramp=0.0):
    R = KV * N
    codes = rng.integers(0, 1 << bits, size=(R, D)).astype(np.uint8)
    c = 0.16 / (1 << bits)
    # ramp > 0: scales grow by 2^ramp from the first cached row to the last
    grow = 2.0 ** (ramp * (np.arange(R) % N) / max(1, N - 1))[:, None]
    s = ((np.abs(rng.standard_normal((R, D // group))) * c + 1e-3) * grow).astype(np.float16)
    b = (-(1 << (bits - 1)) * s.astype(np.float64) + rng.standard_normal((R, D // group)) * 1e-3
         ).astype(np.float16)
    return codes, s, b


def _dev_cache(codes, s, b, KV, N, D, bits):
    words = aq.aq_pack(torch.from_numpy(codes).cuda(), bits).view(KV, N, D * bits // 32)
    return (words, torch.from_numpy(s).cuda().view(KV, N, -1),
            torch.from_numpy(b).cuda().view(KV, N, -1))


def _case(H, KV, N, D, bits, group, dtype, seed, qscale=2.0, ramp=0.0):
    rng = np.random.default_rng(seed)
    kc, ks, kb = _cache(rng, KV, N, D, bits, group)
    vc, vs, vb = _cache(rng, KV, N, D, bits, group, ramp)
    qf = (rng.standard_normal((H, D)) * qscale).astype(np.float32)
    q_bits = workloads.f32_to_bf16_bits(qf) if dtype == "bf16" else workloads.f32_to_fp16_bits(qf)
    return (kc, ks, kb), (vc, vs, vb), q_bits


def _check(H, KV, N, D, bits, group, dtype, seed, qscale=2.0, ramp=0.0, workspace=False):
    """workspace=True: aq_attention_decode_ws with a zeroed workspace of the
    size its plan wants; returns that workspace (its counters checked zero)."""
    (kc, ks, kb), (vc, vs, vb), q_bits = _case(H, KV, N, D, bits, group, dtype, seed, qscale,
                                               ramp)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(tdt)
    kd, vd = _dev_cache(kc, ks, kb, KV, N, D, bits), _dev_cache(vc, vs, vb, KV, N, D, bits)
    ws = None
    if workspace:
        n = aq.aq_attention_workspace_bytes(H, KV, N, D, bits, group)
        ws = torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")
        o = aq.aq_attention_decode_ws(q, kd, vd, bits, group, workspace=ws)
    else:
        o = aq.aq_attention_decode(q, kd, vd, bits, group)
    torch.cuda.synchronize()
    if ws is not None and ws.numel() >= 4 * KV:  # a several-cluster plan: its counters
        assert int(ws[:4 * KV].view(torch.int32).abs().sum()) == 0, "counters not back to zero"
    got = workloads.to_f64(o.view(torch.int16).cpu().numpy().view(np.uint16), dtype)
    ref, smag, vmag = oracle.attention(workloads.to_f64(q_bits, dtype), oracle.pack_g(kc, bits),
                                       ks, kb, oracle.pack_g(vc, bits), vs, vb, KV, N, bits, group)
    tau = (1e-4 * smag + 1e-5).max(axis=1, keepdims=True)
    rnd = 2.0**-8 if dtype == "bf16" else 2.0**-11
    # largest |value bias| of each (query head, dimension)'s KV head and group
    vbmax = np.abs(vb.astype(np.float64)).reshape(KV, N, D // group).max(axis=1)
    vbmax = np.repeat(np.repeat(vbmax, H // KV, axis=0), group, axis=1)
    tol = ((np.expm1(2 * tau) + 2.0**-24 * N) * vmag + 2.0**-10 * (vmag + vbmax)
           + rnd * np.abs(ref) + 1e-6)
    bad = np.argwhere(~(np.abs(got - ref) <= tol))
    assert bad.size == 0, [(int(h), int(d), float(got[h, d]), float(ref[h, d]), float(tol[h, d]))
                           for h, d in bad[:4]]
    return ws


@pytest.mark.parametrize("H,KV,N,D,bits,group,dtype", [
    (4, 4, 1, 64, 4, 32, "bf16"),         # one cached row
    (8, 2, 100, 128, 4, 64, "bf16"),      # four query heads per KV head
    (16, 8, 1000, 256, 8, 64, "bf16"),    # several CTAs per cluster
    (8, 1, 777, 128, 8, 32, "fp16"),      # eight query heads, ragged blocks
    (2, 2, 5000, 64, 4, 64, "fp16"),      # 16 blocks of a KV head
    (32, 8, 4096, 128, 4, 128, "bf16"),
    (6, 6, 70, 256, 4, 32, "bf16"),       # rows fewer than warps x blocks
    (8, 8, 300, 256, 8, 128, "fp16"),     # 256-byte rows: two TMA boxes per stage
    (4, 2, 1531, 64, 8, 32, "bf16"),      # 64-byte rows, ragged last stage
    (2, 1, 16, 128, 4, 128, "bf16"),      # one full tile
    (16, 2, 2053, 256, 4, 64, "fp16"),    # eight query heads over 256 dims
    (8, 8, 129, 128, 4, 32, "bf16"),      # one row past a stage
    (8, 1, 1000, 256, 8, 32, "fp16"),     # eight heads, 8-bit 256-byte rows, groups of 32
    (16, 2, 700, 256, 8, 64, "bf16"),
    (8, 2, 1000, 512, 4, 64, "bf16"),     # 512 dimensions: a warp pair per tile
    (8, 8, 333, 512, 8, 128, "fp16"),     # 512-byte rows, one-stage ring
    (16, 2, 1500, 512, 4, 32, "bf16"),    # eight heads, sixteen groups per row
    (2, 2, 97, 512, 8, 32, "bf16"),
])
def test_attention_parity(H, KV, N, D, bits, group, dtype):
    _check(H, KV, N, D, bits, group, dtype, seed=H + KV + N + D + bits + group)


def test_attention_sharp_softmax():
    # large scores: one row dominates each head
    _check(8, 4, 333, 128, 8, 64, "bf16", seed=9, qscale=40.0)


@pytest.mark.parametrize("ramp", [12.0, -12.0])
def test_attention_value_scale_range(ramp):
    # value scales over 4096x from the first row to the last (or back): the
    # fp16 headroom exponent of each warp is lowered as larger scales appear
    _check(8, 2, 3000, 128, 4, 64, "bf16", seed=11, ramp=ramp)


def test_attention_describe():
    d = aq.aq_attention_describe(16, 8, 8192, 256, 4, 64)
    fields = dict(kv.split("=") for kv in d.split()[1:])
    assert d.startswith("attn ") and 1 <= int(fields["cluster"]) <= 16
    assert int(fields["block"]) * int(fields["cluster"]) >= 8192 and int(fields["block"]) % 16 == 0
    assert int(fields["grid"]) == 8 * int(fields["cluster"])
    assert aq.aq_attention_describe(16, 8, 8192, 96, 4, 32) == "unsupported"


def test_attention_workload_shape():
    # 16 query heads over 8 KV heads of 256 dims, 8192 cached rows, 4-bit
    _check(16, 8, 8192, 256, 4, 64, "bf16", seed=10)


def test_attention_unsupported_head_dim():
    (kc, ks, kb), (vc, vs, vb), q_bits = _case(2, 2, 10, 96, 4, 32, "bf16", seed=1)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    with pytest.raises(aq.AqError) as e:
        aq.aq_attention_decode(q, _dev_cache(kc, ks, kb, 2, 10, 96, 4),
                               _dev_cache(vc, vs, vb, 2, 10, 96, 4), 4, 32)
    assert e.value.status == 2


def test_attention_deterministic():
    (kc, ks, kb), (vc, vs, vb), q_bits = _case(16, 8, 3000, 128, 4, 64, "bf16", seed=2)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    k = _dev_cache(kc, ks, kb, 8, 3000, 128, 4)
    v = _dev_cache(vc, vs, vb, 8, 3000, 128, 4)
    outs = [aq.aq_attention_decode(q, k, v, 4, 64).clone() for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


# aq_attention_decode_ws: a KV head's rows over several clusters, partials
# merged by the cluster that arrives last (counters in the workspace).
@pytest.mark.parametrize("H,KV,N,D,bits,group,dtype", [
    (16, 8, 32768, 256, 4, 64, "bf16"),   # the 32k workload shape: four clusters a head
    (16, 8, 8192, 256, 4, 64, "bf16"),    # the 8k workload shape
    (16, 8, 2048, 256, 4, 64, "bf16"),
    (16, 8, 8192, 256, 8, 64, "bf16"),
    (32, 8, 8192, 128, 4, 64, "bf16"),
    (16, 8, 8192, 512, 4, 64, "bf16"),    # warp pairs
    (8, 2, 5000, 128, 4, 32, "fp16"),     # few KV heads: many clusters a head
    (4, 1, 20000, 64, 8, 64, "fp16"),
    (8, 8, 300, 128, 4, 128, "bf16"),     # few rows: one cluster a head
])
def test_attention_ws_parity(H, KV, N, D, bits, group, dtype):
    _check(H, KV, N, D, bits, group, dtype, seed=3 * H + KV + N + D + bits + group,
           workspace=True)


def test_attention_ws_plan_spreads_the_heads():
    # 8 KV heads of 32768 rows: one cluster per head holds at most ~12 CTAs;
    # with a workspace the plan takes several clusters a head
    n = aq.aq_attention_workspace_bytes(16, 8, 32768, 256, 4, 64)
    assert n > 0
    d = aq.aq_attention_describe_ws(16, 8, 32768, 256, 4, 64, n)
    fields = dict(kv.split("=") for kv in d.split()[1:])
    assert int(fields["clusters_per_kv_head"]) > 1 and int(fields["workspace"]) <= n
    assert int(fields["grid"]) == 8 * int(fields["cluster"]) * int(fields["clusters_per_kv_head"])
    assert int(fields["grid"]) > 8 * int(dict(kv.split("=") for kv in aq.aq_attention_describe(
        16, 8, 32768, 256, 4, 64).split()[1:])["cluster"])
    # too small a workspace: the one-cluster plan
    d1 = aq.aq_attention_describe_ws(16, 8, 32768, 256, 4, 64, 64)
    assert "clusters_per_kv_head=1" in d1


def test_attention_ws_deterministic_and_reusable():
    H, KV, N, D, bits, group = 16, 8, 32768, 256, 4, 64
    (kc, ks, kb), (vc, vs, vb), q_bits = _case(H, KV, N, D, bits, group, "bf16", seed=5)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    kd, vd = _dev_cache(kc, ks, kb, KV, N, D, bits), _dev_cache(vc, vs, vb, KV, N, D, bits)
    n = aq.aq_attention_workspace_bytes(H, KV, N, D, bits, group)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    outs = [aq.aq_attention_decode_ws(q, kd, vd, bits, group, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert int(ws[:4 * KV].view(torch.int32).abs().sum()) == 0


def test_attention_ws_small_workspace_runs_one_cluster():
    _check(16, 8, 4096, 256, 4, 64, "bf16", seed=12)  # reference for the shape
    H, KV, N, D, bits, group = 16, 8, 4096, 256, 4, 64
    (kc, ks, kb), (vc, vs, vb), q_bits = _case(H, KV, N, D, bits, group, "bf16", seed=12)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    kd, vd = _dev_cache(kc, ks, kb, KV, N, D, bits), _dev_cache(vc, vs, vb, KV, N, D, bits)
    o1 = aq.aq_attention_decode(q, kd, vd, bits, group)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")  # too small for several clusters
    o2 = aq.aq_attention_decode_ws(q, kd, vd, bits, group, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
