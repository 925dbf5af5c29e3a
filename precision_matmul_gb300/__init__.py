"""GB300-native (sm_103a) FP8 scaled matrix multiply with a fused global amax.

``scaled_mm`` is the torch-facing call: it marshals tensors into the C ABI of
``include/fp8mm.h`` (``fp8mm_plan`` / ``fp8mm_run``), whose CUDA kernels do all
of the arithmetic.  torch supplies device memory and streams only.  There is
no host or library fallback: without the built CUDA library every call raises.

Semantics (mmaemu "API reference (v0.1)", mmaemu.scaled_mm; TileOPs "Linear
Algebra Operators", GemmFP8FwdOp; cuDNN "GEMM + Amax (SM100)")::

    C = (A * s_a) @ (B * s_b)^T  in out_dtype,   amax = max |C|

with A [M, K] (or [L, M, K]) and B [N, K] (or [L, N, K]) FP8 (E4M3 or E5M2),
per-tensor, 1x128 / 128x128 block, or MX (UE8M0 per 32 along K) scales, and
fast (one fp32 chain over K) or slow (128-K chunks promoted in fp32)
accumulation.
"""
from __future__ import annotations

import threading

from . import _binding
from ._binding import (FP8MM_E4M3, FP8MM_E5M2, FP8MM_OUT_BF16, FP8MM_OUT_F16, FP8MM_OUT_F32,
                       FP8MM_SCALE_A1x128_B1x128, FP8MM_SCALE_A1x128_B128x128, FP8MM_SCALE_MX32_UE8M0,
                       FP8MM_SCALE_TENSOR, FP8MMError, Plan, fp8mm_device_error, fp8mm_gemm, fp8mm_plan,
                       fp8mm_run, fp8mm_status_string, make_desc)

__all__ = ["scaled_mm", "plan_for", "Plan", "FP8MMError", "fp8mm_plan", "fp8mm_run", "fp8mm_gemm",
           "fp8mm_device_error", "fp8mm_status_string", "make_desc", "FP8MM_E4M3", "FP8MM_E5M2",
           "FP8MM_OUT_F32", "FP8MM_OUT_BF16", "FP8MM_OUT_F16", "FP8MM_SCALE_TENSOR",
           "FP8MM_SCALE_A1x128_B1x128", "FP8MM_SCALE_A1x128_B128x128", "FP8MM_SCALE_MX32_UE8M0"]

_lock = threading.Lock()
_plans: dict = {}
_workspaces: dict = {}


def _torch():
    import torch
    return torch


def _fmt_of(t, explicit):
    torch = _torch()
    if explicit is not None:
        return int(explicit)
    if t.dtype == torch.float8_e4m3fn:
        return FP8MM_E4M3
    if t.dtype == torch.float8_e5m2:
        return FP8MM_E5M2
    raise TypeError(f"operand dtype {t.dtype}: pass float8_e4m3fn / float8_e5m2, or uint8 codes with a_fmt/b_fmt")


def _out_code(dtype):
    torch = _torch()
    table = {torch.float32: FP8MM_OUT_F32, torch.bfloat16: FP8MM_OUT_BF16, torch.float16: FP8MM_OUT_F16}
    if dtype not in table:
        raise TypeError(f"out_dtype {dtype}: float32, bfloat16 or float16")
    return table[dtype]


def _infer_scale_mode(scale_a, scale_b, L, M, N, K):
    torch = _torch()
    if scale_a.dtype in (torch.uint8, getattr(torch, "float8_e8m0fnu", torch.uint8)):
        return FP8MM_SCALE_MX32_UE8M0
    if scale_a.numel() == 1 and scale_b.numel() == 1:
        return FP8MM_SCALE_TENSOR
    kb = (K + 127) // 128
    if scale_b.numel() == L * N * kb and scale_a.numel() == L * M * kb:
        return FP8MM_SCALE_A1x128_B1x128
    if scale_b.numel() == L * ((N + 127) // 128) * kb and scale_a.numel() == L * M * kb:
        return FP8MM_SCALE_A1x128_B128x128
    raise ValueError("cannot infer the scale form from the scale shapes; pass scale_mode")


def plan_for(desc_key: tuple) -> Plan:
    """Cached plan for a description tuple (see ``scaled_mm``)."""
    with _lock:
        p = _plans.get(desc_key)
        if p is None:
            p = Plan(make_desc(*desc_key[:4], a_fmt=desc_key[4], b_fmt=desc_key[5], scale_mode=desc_key[6],
                               out_dtype=desc_key[7], fast_accum=desc_key[8], splitk=desc_key[9],
                               swap_ab=desc_key[10], block_n=desc_key[11], device=desc_key[12],
                               cta_pair=desc_key[13] if len(desc_key) > 13 else 0,
                               epi_warps=desc_key[14] if len(desc_key) > 14 else 0))
            _plans[desc_key] = p
        return p


def _workspace(device, stream_handle, nbytes):
    torch = _torch()
    if nbytes == 0:
        return None
    key = (device, stream_handle)
    with _lock:
        ws = _workspaces.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=f"cuda:{device}")
            _workspaces[key] = ws
        return ws


def scaled_mm(a, b, scale_a, scale_b, *, out_dtype=None, use_fast_accum=False, a_fmt=None, b_fmt=None,
              scale_mode=None, out=None, amax=None, splitk=0, swap_ab=0, block_n=0, cta_pair=0, epi_warps=0):
    """C = (a * scale_a) @ (b * scale_b)^T and amax = max |C|, on a's CUDA device.

    a: [M, K] or [L, M, K]; b: [N, K] or [L, N, K]; both K-contiguous FP8
    (float8_e4m3fn / float8_e5m2, or uint8 codes with a_fmt / b_fmt).
    Scales are device tensors: fp32 one-element (per-tensor), fp32 1x128 /
    128x128 block scales, or uint8 / float8_e8m0fnu MX factor atoms.
    Returns (C, amax) with C of out_dtype (default bfloat16) and amax a
    one-element fp32 tensor.  splitk, swap_ab, block_n, cta_pair and
    epi_warps override the planner's choices (0 leaves them to it; meanings as
    in fp8mm_desc).  Enqueued on the current stream; nothing is
    synchronised.  One workspace per (device, stream) is reused, so calls on
    one stream must not overlap with calls of another thread on that stream.
    """
    torch = _torch()
    if out_dtype is None:
        out_dtype = torch.bfloat16
    batched = a.dim() == 3
    if a.dim() not in (2, 3) or b.dim() != a.dim():
        raise ValueError("a and b must both be [M, K] or both [L, M, K]")
    if not (a.is_cuda and b.is_cuda and scale_a.is_cuda and scale_b.is_cuda):
        raise ValueError("all inputs must be CUDA tensors")
    L = a.shape[0] if batched else 1
    M, K = a.shape[-2], a.shape[-1]
    N = b.shape[-2]
    if b.shape[-1] != K or (batched and b.shape[0] != L):
        raise ValueError("a and b disagree on K or L")
    if not (a.is_contiguous() and b.is_contiguous() and scale_a.is_contiguous() and scale_b.is_contiguous()):
        raise ValueError("a, b and the scales must be contiguous (K innermost)")
    fa, fb = _fmt_of(a, a_fmt), _fmt_of(b, b_fmt)
    oc = _out_code(out_dtype)
    mode = scale_mode if scale_mode is not None else _infer_scale_mode(scale_a, scale_b, L, M, N, K)
    device = a.device.index if a.device.index is not None else torch.cuda.current_device()
    fast = 1 if use_fast_accum else 0
    key = (M, N, K, L, fa, fb, int(mode), oc, fast, int(splitk), int(swap_ab), int(block_n), device, int(cta_pair),
           int(epi_warps))
    plan = plan_for(key)
    shape = (L, M, N) if batched else (M, N)
    if out is None:
        out = torch.empty(shape, dtype=out_dtype, device=a.device)
    elif tuple(out.shape) != shape or out.dtype != out_dtype or not out.is_contiguous():
        raise ValueError("out has the wrong shape, dtype or layout")
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=a.device)
    stream = torch.cuda.current_stream(a.device).cuda_stream
    nbytes = plan.workspace_size()
    ws = _workspace(device, stream, nbytes)
    plan.run(a.data_ptr(), b.data_ptr(), scale_a.data_ptr(), scale_b.data_ptr(), out.data_ptr(),
             amax.data_ptr(), ws.data_ptr() if ws is not None else None, nbytes, stream)
    return out, amax
