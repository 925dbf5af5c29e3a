"""GPU parity at the full workload sizes, with the plans the benchmark uses.

Each case runs the whole GEMM on the GPU through the C ABI.  The per-tensor
256^3 and 4096^3 GEMMs and the 8192 x 7168 x 2048 block-scaled GEMM are
compared with the oracle on every element of C; the MX batch and the skinny
sweep (N = 28672, K = 8192) on a sample of rows spread over every tile row and
the ragged end, under the same bound as the small cases.  amax is checked bit
for bit against max |C| over the GPU's entire output.
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


def _full(p, rows="all"):
    c, amax, plan = run_gpu(p)
    torch.cuda.synchronize()
    assert pm.fp8mm_device_error(0) == 0
    check(p, c, amax, rows=None if rows == "all" else rows)
    return plan


def test_tiny_per_tensor_full_check():
    _full(synth.tiny_per_tensor())


@pytest.mark.parametrize("fast", [True, False])
def test_llm_4096(fast):
    _full(synth.llm_per_tensor(fast_accum=fast))


def test_blockwise_8192_7168_2048():
    _full(synth.blockwise())


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
def test_mx_batched_4x4096(fmt):
    _full(synth.mx_batched(fmt=fmt), rows=_rows(4096, 6))


_SKINNY = {}


def _skinny(M, data):
    """Inputs shared by the fast and slow calls of one (M, data) pair."""
    key = (M, data)
    if key not in _SKINNY:
        _SKINNY.clear()
        _SKINNY[key] = synth.skinny(M=M, data=data)
    return _SKINNY[key]


@pytest.mark.parametrize("M", [16, 64, 256, 1024, 2048, 8192])
@pytest.mark.parametrize("data", ["gauss40", "adversarial"])
@pytest.mark.parametrize("fast", [True, False])
def test_skinny_sweep_28672_8192(M, data, fast):
    p = _skinny(M, data)
    p.fast_accum = fast
    _full(p, rows=_rows(M, 8))
