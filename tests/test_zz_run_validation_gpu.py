"""fp8mm_run's own checks on the GPU: each bad buffer returns its status
before anything is enqueued, so the output and amax keep their prior
contents; the same plan then runs with good buffers."""
import ctypes

import pytest
import torch

from precision_matmul_gb300 import _binding as B

pytestmark = pytest.mark.gpu

SENTINEL = 0x1234


def _run(plan, stream, a, b, sa, sb, c, amax, ws, ws_bytes):
    return B.load().fp8mm_run(plan.handle, a, b, sa, sb, c, amax, ws, ctypes.c_size_t(ws_bytes), stream)


def test_bad_buffers_are_refused_and_nothing_runs():
    dev = "cuda:0"
    M, N, K = 64, 256, 1024                    # swap-AB, 64-wide tiles, split in two along K
    plan = B.Plan(B.make_desc(M, N, K, 1, out_dtype=B.FP8MM_OUT_BF16, fast_accum=1, splitk=2))
    assert plan.info()["splitk"] == 2
    ws_bytes = plan.workspace_size()
    assert ws_bytes > 0
    a = torch.zeros(M * K + 64, dtype=torch.uint8, device=dev)
    b = torch.zeros(N * K + 64, dtype=torch.uint8, device=dev)
    s = torch.ones(4, dtype=torch.float32, device=dev)
    c = torch.full((M * N + 64,), SENTINEL, dtype=torch.int16, device=dev)
    amax = torch.full((4,), SENTINEL, dtype=torch.int32, device=dev)
    ws = torch.empty(ws_bytes + 512, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    good = dict(a=a.data_ptr(), b=b.data_ptr(), sa=s.data_ptr(), sb=s.data_ptr(), c=c.data_ptr(),
                amax=amax.data_ptr(), ws=ws.data_ptr(), ws_bytes=ws_bytes)

    def run(**over):
        args = dict(good)
        args.update(over)
        return _run(plan, stream, **args)

    cases = [
        (dict(a=good["a"] + 1), B.FP8MM_ERR_ALIGNMENT),
        (dict(b=good["b"] + 8), B.FP8MM_ERR_ALIGNMENT),
        (dict(c=good["c"] + 2), B.FP8MM_ERR_ALIGNMENT),
        (dict(sa=good["sa"] + 2), B.FP8MM_ERR_ALIGNMENT),
        (dict(amax=good["amax"] + 2), B.FP8MM_ERR_ALIGNMENT),
        (dict(ws=good["ws"] + 16), B.FP8MM_ERR_ALIGNMENT),
        (dict(ws=None), B.FP8MM_ERR_WORKSPACE),
        (dict(ws_bytes=ws_bytes - 1), B.FP8MM_ERR_WORKSPACE),
        (dict(c=None), B.FP8MM_ERR_INVALID),
        (dict(a=None), B.FP8MM_ERR_INVALID),
        (dict(sb=None), B.FP8MM_ERR_INVALID),
        (dict(amax=None), B.FP8MM_ERR_INVALID),
    ]
    for over, want in cases:
        assert run(**over) == want, over
    torch.cuda.synchronize()
    assert (c == SENTINEL).all() and (amax == SENTINEL).all()
    assert B.fp8mm_device_error(0) == 0

    assert run() == B.FP8MM_OK                 # zero operands: C = +0 everywhere, amax = +0
    torch.cuda.synchronize()
    assert (c[:M * N] == 0).all() and (c[M * N:] == SENTINEL).all()
    assert int(amax[0]) == 0 and (amax[1:] == SENTINEL).all()


def test_mx_factors_need_16_byte_alignment():
    dev = "cuda:0"
    plan = B.Plan(B.make_desc(128, 128, 128, 1, scale_mode=B.FP8MM_SCALE_MX32_UE8M0, out_dtype=B.FP8MM_OUT_F32))
    a = torch.zeros(128 * 128, dtype=torch.uint8, device=dev)
    sf = torch.full((512 + 64,), 127, dtype=torch.uint8, device=dev)
    c = torch.full((128 * 128,), SENTINEL, dtype=torch.int32, device=dev)
    amax = torch.full((1,), SENTINEL, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for off in (4, 8):
        st = _run(plan, stream, a.data_ptr(), a.data_ptr(), sf.data_ptr() + off, sf.data_ptr(), c.data_ptr(),
                  amax.data_ptr(), None, 0)
        assert st == B.FP8MM_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert (c == SENTINEL).all() and int(amax[0]) == SENTINEL
