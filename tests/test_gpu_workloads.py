"""Parity at the workloads' full sizes, in the launch configuration the
benchmark uses (automatic dispatch).  The packed words are compared bit for
bit with the oracle's; outputs are checked against the fp64 oracle on a
seeded sample of output columns (all activation rows), or in full where the
oracle finishes in seconds."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._gpu import assert_within_tolerance, dev_tensors, y_to_f64

pytestmark = pytest.mark.gpu

aq = pytest.importorskip("quantized_matmul_affine_gb300")

CASES = [(name, i) for name, cfgs in workloads.WORKLOADS.items() for i in range(len(cfgs))]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    aq.aq_device_error(clear=True)
    yield
    assert aq.aq_device_error() == 0


@pytest.mark.parametrize("name,index", CASES, ids=[f"{n}[{i}]" for n, i in CASES])
def test_workload(name, index):
    p = workloads.workload(name, index)
    codes, s, b, x = dev_tensors(p)
    Wq = aq.aq_pack(codes, p.bits)
    del codes
    words_ref = oracle.pack(p.codes, p.bits)
    np.testing.assert_array_equal(Wq.cpu().numpy().view(np.uint32), words_ref)
    fn = aq.aq_matmul_bf16 if p.x_dtype == "bf16" else aq.aq_matmul
    y = y_to_f64(fn(x, Wq, s, b, p.bits), p.x_dtype)
    if p.M * p.N * p.K <= 64 * 1024 * 1024:
        y_ref, bound = oracle.matmul(p.x_f64(), words_ref, p.scales, p.biases, p.bits, threads=8)
        assert_within_tolerance(y, y_ref, bound, p.name)
    else:
        rng = np.random.default_rng(1000 + index)
        cols = np.unique(np.concatenate([[0, p.N - 1], rng.integers(0, p.N, 62)]))
        y_ref, bound = oracle.matmul_cols(p.x_f64(), words_ref, p.scales, p.biases, p.bits,
                                          cols)
        assert_within_tolerance(y[:, cols], y_ref, bound, p.name)
    assert np.all(np.isfinite(y))
