"""The no-allocation entry point, fp8mm_run_static_workspace.

Callers such as plugin or custom-call hosts own every device buffer and hand
an operation only its inputs and outputs, so they cannot give fp8mm_run a
workspace.  This entry point takes its split-K scratch from a fixed array
inside the library instead.  The test calls it through the C ABI on a plan
that needs scratch, twice in a row with different inputs, and compares each
result with fp8mm_run's output for the same inputs (and with the oracle's
bound); it also checks that a plan needing more scratch than the array holds
is refused before anything runs.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from precision_matmul_gb300 import _binding as B
from precision_matmul_gb300 import synth

from parity import check

pytestmark = pytest.mark.gpu


def _desc_for(p):
    return B.make_desc(p.M, p.N, p.K, p.L, a_fmt=p.a_fmt, b_fmt=p.b_fmt, scale_mode=p.scale_mode,
                       out_dtype=p.out_dtype, fast_accum=1 if p.fast_accum else 0, device=0)


def test_static_workspace_matches_caller_workspace_twice():
    dev = torch.device("cuda:0")
    probs = [synth.skinny(M=40, N=2048, K=4096, seed=101, fast_accum=True),
             synth.skinny(M=40, N=2048, K=4096, seed=102, fast_accum=True)]
    plan = B.Plan(_desc_for(probs[0]))
    ws_bytes = plan.workspace_size()
    assert plan.info()["splitk"] > 1 and 0 < ws_bytes <= B.FP8MM_STATIC_WORKSPACE_BYTES
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for p in probs:
        a, b = p.a[0].to(dev), p.b[0].to(dev)
        sa, sb = p.scale_a.to(dev), p.scale_b.to(dev)
        c_ref = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)
        m_ref = torch.empty(1, dtype=torch.float32, device=dev)
        B.fp8mm_run(plan, a.data_ptr(), b.data_ptr(), sa.data_ptr(), sb.data_ptr(), c_ref.data_ptr(),
                    m_ref.data_ptr(), ws.data_ptr(), ws_bytes, stream)
        c = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device=dev)
        m = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
        B.fp8mm_run_static_workspace(plan, a.data_ptr(), b.data_ptr(), sa.data_ptr(), sb.data_ptr(),
                                     c.data_ptr(), m.data_ptr(), stream)
        torch.cuda.synchronize()
        assert B.fp8mm_device_error(0) == 0
        # the same kernel, the same split order: identical bits, and both within the oracle's bound
        assert torch.equal(c.view(torch.int16), c_ref.view(torch.int16))
        assert torch.equal(m.view(torch.int32), m_ref.view(torch.int32))
        check(p, c, m)


def test_static_workspace_refuses_oversized_plans():
    p = synth.skinny(M=64, N=28672, K=8192, seed=103)
    d = _desc_for(p)
    d.splitk = 8
    plan = B.Plan(d)
    assert plan.workspace_size() > B.FP8MM_STATIC_WORKSPACE_BYTES
    with pytest.raises(B.FP8MMError) as e:
        B.fp8mm_run_static_workspace(plan, 16, 16, 16, 16, 16, 16, None)
    assert e.value.status == B.FP8MM_ERR_WORKSPACE
    np.testing.assert_equal(B.fp8mm_device_error(0), 0)


def test_static_workspace_slow_block_scaled_split_k_swapped():
    # the promoted (slow) path of a block-scaled, swapped, split-K plan: partial
    # tiles of promoted sums go through the library's array instead of a caller buffer
    dev = torch.device("cuda:0")
    p = synth.blockwise(M=48, N=1024, K=2048, seed=104)
    d = _desc_for(p)
    d.splitk, d.swap_ab = 3, 1
    plan = B.Plan(d)
    info = plan.info()
    ws_bytes = plan.workspace_size()
    assert info["slow"] == 1 and info["swap_ab"] == 1 and info["splitk"] == 3
    assert 0 < ws_bytes <= B.FP8MM_STATIC_WORKSPACE_BYTES
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    a, b = p.a[0].to(dev), p.b[0].to(dev)
    sa, sb = p.scale_a.to(dev), p.scale_b.to(dev)
    c_ref = torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)
    m_ref = torch.empty(1, dtype=torch.float32, device=dev)
    B.fp8mm_run(plan, a.data_ptr(), b.data_ptr(), sa.data_ptr(), sb.data_ptr(), c_ref.data_ptr(),
                m_ref.data_ptr(), ws.data_ptr(), ws_bytes, stream)
    for _ in range(2):
        c = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device=dev)
        m = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
        B.fp8mm_run_static_workspace(plan, a.data_ptr(), b.data_ptr(), sa.data_ptr(), sb.data_ptr(),
                                     c.data_ptr(), m.data_ptr(), stream)
        torch.cuda.synchronize()
        assert B.fp8mm_device_error(0) == 0
        assert torch.equal(c.view(torch.int16), c_ref.view(torch.int16))
        assert torch.equal(m.view(torch.int32), m_ref.view(torch.int32))
        check(p, c, m)
