"""The kernels' abort path, exercised on the GPU without a fault or a hang.

With fp8mm_test_withhold_loads enabled the producer issues no operand loads,
so the MMA issuer's first wait for a stage and the epilogue's wait for the
accumulator (each bounded at 2^31 SM cycles) run out: the first to give up
records its code in the abort word, every role leaves its loop, in-flight work
drains, TMEM is freed and the kernel returns.
The test then checks that the CUDA context is still usable: the same call,
with loads, matches the oracle.  (The failure is made on purpose by a flag
that nothing sets, as a bounded wait; nothing traps or faults.)
"""
import pytest
import torch

import precision_matmul_gb300 as pm
from precision_matmul_gb300 import _binding as B
from precision_matmul_gb300 import synth

from parity import check, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fast", [True, False])
def test_a_wait_that_runs_out_aborts_and_the_context_stays_usable(fast):
    p = synth.llm_per_tensor(M=256, N=512, K=512, seed=90, fast_accum=fast)
    assert pm.fp8mm_device_error(0, clear=True) == 0
    B.fp8mm_test_withhold_loads(True)
    try:
        run_gpu(p, cta_pair=2)  # one-CTA tiles
        torch.cuda.synchronize()
    finally:
        B.fp8mm_test_withhold_loads(False)
    code = pm.fp8mm_device_error(0, clear=True)
    # the MMA issuer's stage wait (2) or the epilogue's accumulator wait (8) gave up first
    assert code != 0 and (code & ~(2 | 8)) == 0, f"abort word {code:#x}"
    assert pm.fp8mm_device_error(0) == 0  # cleared
    c, amax, plan = run_gpu(p, cta_pair=2)
    torch.cuda.synchronize()
    assert pm.fp8mm_device_error(0) == 0
    check(p, c, amax)
