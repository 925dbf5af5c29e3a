"""GPU parity at the full workload sizes, with the plans the benchmark uses.

Each case runs the whole GEMM on the GPU through the C ABI and checks a sample
of rows (spread over every tile row and the ragged end) against the oracle
element by element, under the same bound as the small cases; amax is checked
bit-for-bit against max |C| over the GPU's entire output.
"""
import numpy as np
import pytest
import torch

import precision_matmul_gb300 as pm
from precision_matmul_gb300 import synth

from parity import check, run_gpu

pytestmark = pytest.mark.gpu


def _rows(M, n=12):
    """Sample rows: both ends, tile-row boundaries and a spread in between."""
    cand = {0, 1, M - 1, M // 2, min(M - 1, 127), min(M - 1, 128)}
    cand.update(int(x) for x in np.linspace(0, M - 1, n))
    return sorted(r for r in cand if 0 <= r < M)


def _full(p, rows=None):
    c, amax, plan = run_gpu(p)
    torch.cuda.synchronize()
    assert pm.fp8mm_device_error(0) == 0
    check(p, c, amax, rows=_rows(p.M) if rows is None else rows)
    return plan


def test_tiny_per_tensor_full_check():
    c, amax, _ = run_gpu(synth.tiny_per_tensor())
    torch.cuda.synchronize()
    check(synth.tiny_per_tensor(), c, amax)


@pytest.mark.parametrize("fast", [True, False])
def test_llm_4096(fast):
    _full(synth.llm_per_tensor(fast_accum=fast))


def test_blockwise_8192_7168_2048():
    _full(synth.blockwise())


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
def test_mx_batched_4x4096(fmt):
    _full(synth.mx_batched(fmt=fmt), rows=_rows(4096, 6))


@pytest.mark.parametrize("M,data,fast", [
    (16, "gauss40", True), (16, "gauss40", False), (64, "adversarial", False), (256, "gauss40", True),
    (1024, "gauss40", False), (2048, "adversarial", True), (8192, "gauss40", True),
])
def test_skinny_sweep_28672_8192(M, data, fast):
    p = synth.skinny(M=M, data=data, fast_accum=fast)
    _full(p, rows=_rows(M, 8))
