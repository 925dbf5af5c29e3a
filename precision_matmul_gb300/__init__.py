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
from ._binding import (FP8MM_E2M1, FP8MM_E4M3, FP8MM_E5M2, FP8MM_OUT_BF16, FP8MM_OUT_E4M3, FP8MM_OUT_E5M2, FP8MM_OUT_F16,
                       FP8MM_OUT_F32, FP8MM_SCALE_A1x128_B1x128, FP8MM_SCALE_A1x128_B128x128,
                       FP8MM_SCALE_MX32_UE8M0, FP8MM_SCALE_NV16_E4M3, FP8MM_SCALE_TENSOR, FP8MMError, Plan, fp8mm_device_error,
                       fp8mm_gemm, fp8mm_plan, fp8mm_run, fp8mm_run_ex, fp8mm_status_string, make_desc)

__all__ = ["scaled_mm", "torch_scaled_mm", "bmm_fp8", "describe", "operand_majors", "plan_for", "Plan", "FP8MMError",
           "fp8mm_plan", "fp8mm_run", "fp8mm_run_ex", "fp8mm_gemm",
           "fp8mm_device_error", "fp8mm_status_string", "make_desc", "FP8MM_E4M3", "FP8MM_E5M2", "FP8MM_E2M1",
           "FP8MM_SCALE_NV16_E4M3",
           "FP8MM_OUT_F32", "FP8MM_OUT_BF16", "FP8MM_OUT_F16", "FP8MM_OUT_E4M3", "FP8MM_OUT_E5M2", "FP8MM_SCALE_TENSOR",
           "FP8MM_SCALE_A1x128_B1x128", "FP8MM_SCALE_A1x128_B128x128", "FP8MM_SCALE_MX32_UE8M0"]

_lock = threading.Lock()
_plans: dict = {}
_workspaces: dict = {}


def _torch():
    import torch
    return torch


def _fmt_of(t, explicit):
    torch = _torch()
    table = {torch.float8_e4m3fn: FP8MM_E4M3, torch.float8_e5m2: FP8MM_E5M2}
    if hasattr(torch, "float4_e2m1fn_x2"):
        table[torch.float4_e2m1fn_x2] = FP8MM_E2M1
    native = table.get(t.dtype)
    if native is None and t.dtype != torch.uint8:
        raise TypeError(f"operand dtype {t.dtype}: pass float8_e4m3fn / float8_e5m2 / float4_e2m1fn_x2, or uint8 "
                        "codes with a_fmt/b_fmt")
    if explicit is None:
        if native is None:
            raise TypeError("uint8 operand codes need their format (a_fmt / b_fmt)")
        return native
    if int(explicit) not in (FP8MM_E4M3, FP8MM_E5M2, FP8MM_E2M1):
        raise ValueError(f"format {explicit}: FP8MM_E4M3, FP8MM_E5M2 or FP8MM_E2M1")
    if native is not None and int(explicit) != native:
        raise ValueError(f"operand dtype {t.dtype} contradicts format {explicit}")
    return int(explicit)


def _out_code(dtype):
    torch = _torch()
    table = {torch.float32: FP8MM_OUT_F32, torch.bfloat16: FP8MM_OUT_BF16, torch.float16: FP8MM_OUT_F16,
             torch.float8_e4m3fn: FP8MM_OUT_E4M3, torch.float8_e5m2: FP8MM_OUT_E5M2}
    if dtype not in table:
        raise TypeError(f"out_dtype {dtype}: float32, bfloat16, float16, float8_e4m3fn or float8_e5m2")
    return table[dtype]


def _major(t, name):
    """0 if t ([.., rows, K]) has K contiguous; 1 if it is the transposed view
    of a contiguous [.., K, rows] tensor (rows contiguous)."""
    if t.is_contiguous():
        return 0
    if t.transpose(-1, -2).is_contiguous():
        return 1
    raise ValueError(f"{name} must be contiguous along K, or the transpose of a tensor contiguous along its rows")


def operand_majors(a, b):
    """(a_major, b_major) of fp8mm_desc from the operands' strides: a [.., M, K]
    and b [.., N, K] views are K-major when K is contiguous, M/N-major when
    they are transposed views of tensors stored [.., K, M] / [.., K, N]."""
    return _major(a, "a"), _major(b, "b")


def _mx_dtypes():
    torch = _torch()
    return (torch.uint8,) + ((torch.float8_e8m0fnu,) if hasattr(torch, "float8_e8m0fnu") else ())


def _scale_elems(mode, L, M, N, K):
    """Elements of (scale_a, scale_b) that the kernels read for a scale form:
    one fp32 each per tensor; fp32 [L][M][ceil(K/128)] for 1x128 A scales and
    [L][N][..] / [L][ceil(N/128)][..] for B; one 512-byte atom per 128 rows
    and 4 factors along K for the factor forms (128 K for UE8M0 per 32, 64 K
    for E4M3 per 16)."""
    kb = (K + 127) // 128
    if mode == FP8MM_SCALE_TENSOR:
        return 1, 1
    if mode == FP8MM_SCALE_A1x128_B1x128:
        return L * M * kb, L * N * kb
    if mode == FP8MM_SCALE_A1x128_B128x128:
        return L * M * kb, L * ((N + 127) // 128) * kb
    if mode == FP8MM_SCALE_MX32_UE8M0:
        return L * ((M + 127) // 128) * kb * 512, L * ((N + 127) // 128) * kb * 512
    if mode == FP8MM_SCALE_NV16_E4M3:
        k64 = (K + 63) // 64
        return L * ((M + 127) // 128) * k64 * 512, L * ((N + 127) // 128) * k64 * 512
    raise ValueError(f"scale_mode {mode}: one of the FP8MM_SCALE_* forms")


def _infer_scale_mode(scale_a, scale_b, L, M, N, K):
    torch = _torch()
    if scale_a.dtype == torch.float8_e4m3fn:
        return FP8MM_SCALE_NV16_E4M3
    if scale_a.dtype in _mx_dtypes():
        return FP8MM_SCALE_MX32_UE8M0
    if scale_a.numel() == 1 and scale_b.numel() == 1:
        return FP8MM_SCALE_TENSOR
    for mode in (FP8MM_SCALE_A1x128_B1x128, FP8MM_SCALE_A1x128_B128x128):
        if (scale_a.numel(), scale_b.numel()) == _scale_elems(mode, L, M, N, K):
            return mode
    raise ValueError("cannot infer the scale form from the scale shapes; pass scale_mode")


def describe(a, b, scale_a, scale_b, *, out_dtype=None, a_fmt=None, b_fmt=None, scale_mode=None, out=None,
             amax=None, bias=None, scale_result=None):
    """Check the arguments of ``scaled_mm`` on the host and return
    ``(L, M, N, K, a_fmt, b_fmt, scale_mode, out_code, out_shape)``.

    Everything the kernels will read or write is checked here, because the C
    ABI only sees pointers: operand formats, that every tensor sits on one
    device and is contiguous, and that the scale tensors hold exactly the
    elements their form reads (a short scale tensor would be read past its
    end on the device).  a and b may also be transposed views of tensors
    stored K-outermost (``operand_majors``); their rows must then be 16-byte
    multiples.  A bias is [N] of out_dtype (not for FP8 outputs);
    scale_result is one fp32 (FP8 outputs).  Raises TypeError or ValueError."""
    torch = _torch()
    if out_dtype is None:
        out_dtype = torch.bfloat16
    batched = a.dim() == 3
    if a.dim() not in (2, 3) or b.dim() != a.dim():
        raise ValueError("a and b must both be [M, K] or both [L, M, K]")
    L = a.shape[0] if batched else 1
    fa, fb = _fmt_of(a, a_fmt), _fmt_of(b, b_fmt)
    M, K = a.shape[-2], a.shape[-1]
    N = b.shape[-2]
    if b.shape[-1] != K or (batched and b.shape[0] != L):
        raise ValueError("a and b disagree on K or L")
    if fa == FP8MM_E2M1 or fb == FP8MM_E2M1:
        if fa != fb:
            raise ValueError("FP4 operands go in pairs (A and B of one format)")
        K *= 2  # packed: two elements per byte
    others = [scale_a, scale_b] + [t for t in (out, amax, bias, scale_result) if t is not None]
    if any(t.device != a.device for t in [a, b] + others):
        raise ValueError("all tensors must be on one device")
    if not all(t.is_contiguous() for t in others):
        raise ValueError("the scales, out, amax and bias must be contiguous")
    am, bm = operand_majors(a, b)
    if (am and M % 16) or (bm and N % 16):
        raise ValueError("a K-outermost operand needs rows (M or N) that are multiples of 16")
    oc = _out_code(out_dtype)
    mode = int(scale_mode) if scale_mode is not None else _infer_scale_mode(scale_a, scale_b, L, M, N, K)
    want_a, want_b = _scale_elems(mode, L, M, N, K)
    if mode == FP8MM_SCALE_MX32_UE8M0:
        if scale_a.dtype not in _mx_dtypes() or scale_b.dtype not in _mx_dtypes():
            raise TypeError("MX factors are uint8 / float8_e8m0fnu UE8M0 codes")
        if fa != fb:
            raise ValueError("the MX form needs A and B of one format")
    elif mode == FP8MM_SCALE_NV16_E4M3:
        if scale_a.dtype not in (torch.uint8, torch.float8_e4m3fn) or scale_b.dtype != scale_a.dtype:
            raise TypeError("per-16 factors are uint8 / float8_e4m3fn E4M3 codes")
        if fa != FP8MM_E2M1:
            raise ValueError("factors per 16 elements go with FP4 operands")
    elif scale_a.dtype != torch.float32 or scale_b.dtype != torch.float32:
        raise TypeError("per-tensor and block scales are float32")
    if (scale_a.numel(), scale_b.numel()) != (want_a, want_b):
        raise ValueError(f"scale form {mode} reads {want_a} / {want_b} scale elements for A / B; "
                         f"got {scale_a.numel()} / {scale_b.numel()}")
    shape = (L, M, N) if batched else (M, N)
    if out is not None and (tuple(out.shape) != shape or out.dtype != out_dtype):
        raise ValueError("out has the wrong shape or dtype")
    if amax is not None and (amax.dtype != torch.float32 or amax.numel() < 1):
        raise ValueError("amax must hold at least one float32")
    if bias is not None:
        if oc in (FP8MM_OUT_E4M3, FP8MM_OUT_E5M2):
            raise ValueError("a bias is not defined for FP8 outputs")
        if bias.dtype != out_dtype or bias.numel() != N:
            raise ValueError("bias must hold N values of out_dtype")
    if scale_result is not None and (scale_result.dtype != torch.float32 or scale_result.numel() != 1):
        raise ValueError("scale_result must be one float32")
    return L, M, N, K, fa, fb, mode, oc, shape


_KEY_LEN = 19


def normalize_key(desc_key: tuple) -> tuple:
    """The canonical plan key: (M, N, K, L, a_fmt, b_fmt, scale_mode, out_dtype,
    fast_accum, splitk, swap_ab, block_n, device, cta_pair, epi_warps,
    strict_torch, bias, a_major, b_major), with fields left off the end taken
    as 0."""
    key = tuple(int(x) for x in desc_key)
    if not 13 <= len(key) <= _KEY_LEN:
        raise ValueError(f"plan key of {len(key)} fields")
    return key + (0,) * (_KEY_LEN - len(key))


def plan_for(desc_key: tuple) -> Plan:
    """Cached plan for a description tuple (see ``normalize_key``)."""
    k = normalize_key(desc_key)
    with _lock:
        p = _plans.get(k)
        if p is None:
            p = Plan(make_desc(*k[:4], a_fmt=k[4], b_fmt=k[5], scale_mode=k[6], out_dtype=k[7], fast_accum=k[8],
                               splitk=k[9], swap_ab=k[10], block_n=k[11], device=k[12], cta_pair=k[13],
                               epi_warps=k[14], strict_torch=k[15], bias=k[16], a_major=k[17], b_major=k[18]))
            _plans[k] = p
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
              scale_mode=None, out=None, amax=None, splitk=0, swap_ab=0, block_n=0, cta_pair=0, epi_warps=0,
              strict_torch=False, bias=None, scale_result=None):
    """C = (a * scale_a) @ (b * scale_b)^T (+ bias) and amax = max |C|, on a's CUDA device.

    a: [M, K] or [L, M, K]; b: [N, K] or [L, N, K]; FP8 (float8_e4m3fn /
    float8_e5m2, or uint8 codes with a_fmt / b_fmt), each either K-contiguous
    or the transposed view of a tensor stored K-outermost ([.., K, M] /
    [.., K, N]: the NN / TN / TT layouts, copied into K-major workspace by the
    library before the GEMM).  Scales are device tensors: fp32 one-element
    (per-tensor), fp32 1x128 / 128x128 block scales, or uint8 / float8_e8m0fnu
    MX factor atoms.  out_dtype (default bfloat16) may be float32, bfloat16,
    float16, float8_e4m3fn or float8_e5m2; FP8 outputs are multiplied by
    scale_result (one fp32 device tensor, default 1) before their saturating
    rounding, and their amax is max |C| before scale_result.  bias: [N] of
    out_dtype added to every row (not for FP8 outputs).
    Returns (C, amax) with amax a one-element fp32 tensor.  splitk, swap_ab,
    block_n, cta_pair and epi_warps override the planner's choices (0 leaves
    them to it; meanings as in fp8mm_desc).  strict_torch=True refuses
    (FP8MMError, FP8MM_ERR_REJECTED) what torch._scaled_mm refuses.  Enqueued
    on the current stream; nothing is synchronised.  One workspace per
    (device, stream) is reused, so calls on one stream must not overlap with
    calls of another thread on that stream.
    """
    torch = _torch()
    if out_dtype is None:
        out_dtype = torch.bfloat16
    if not a.is_cuda:
        raise ValueError("all inputs must be CUDA tensors")
    L, M, N, K, fa, fb, mode, oc, shape = describe(a, b, scale_a, scale_b, out_dtype=out_dtype, a_fmt=a_fmt,
                                                   b_fmt=b_fmt, scale_mode=scale_mode, out=out, amax=amax,
                                                   bias=bias, scale_result=scale_result)
    am, bm = operand_majors(a, b)
    device = a.device.index if a.device.index is not None else torch.cuda.current_device()
    fast = 1 if use_fast_accum else 0
    key = (M, N, K, L, fa, fb, int(mode), oc, fast, int(splitk), int(swap_ab), int(block_n), device, int(cta_pair),
           int(epi_warps), int(bool(strict_torch)), 1 if bias is not None else 0, am, bm)
    plan = plan_for(key)
    if out is None:
        out = torch.empty(shape, dtype=out_dtype, device=a.device)
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=a.device)
    stream = torch.cuda.current_stream(a.device).cuda_stream
    nbytes = plan.workspace_size()
    ws = _workspace(device, stream, nbytes)
    ws_ptr = ws.data_ptr() if ws is not None else None
    if bias is None and scale_result is None:
        plan.run(a.data_ptr(), b.data_ptr(), scale_a.data_ptr(), scale_b.data_ptr(), out.data_ptr(),
                 amax.data_ptr(), ws_ptr, nbytes, stream)
    else:
        plan.run_ex(a.data_ptr(), b.data_ptr(), scale_a.data_ptr(), scale_b.data_ptr(),
                    scale_result.data_ptr() if scale_result is not None else None,
                    bias.data_ptr() if bias is not None else None, out.data_ptr(), amax.data_ptr(), ws_ptr, nbytes,
                    stream)
    return out, amax


def torch_scaled_mm(input, mat2, scale_a, scale_b, bias=None, scale_result=None, out_dtype=None,
                    use_fast_accum=False, *, out=None):
    """The same GEMM in torch._scaled_mm's calling convention (mmaemu "API
    reference (v0.1)", mmaemu.scaled_mm, argument table).

    input [M, K] row-major FP8; mat2 [K, N] FP8 in column-major storage (the
    ``w.t()`` of a row-major [N, K] weight); scale_a, scale_b one-element fp32
    tensors that multiply the result; bias [N] of out_dtype; scale_result a
    one-element fp32 tensor, read only for FP8 outputs; out_dtype defaults to
    input's dtype and may be float32, bfloat16, float16, float8_e4m3fn or
    float8_e5m2.  Returns the [M, N] result (use ``scaled_mm`` for the fused
    amax as well).

    As in torch, E5M2 x E5M2 and E4M3 x E4M3 -> E5M2 are refused (FP8MMError
    with FP8MM_ERR_REJECTED), as are row-major mat2 (ValueError) and a bias
    with an FP8 output (ValueError).  Row-wise scales raise NotImplementedError.
    """
    torch = _torch()
    if out_dtype is None:
        out_dtype = input.dtype
    if input.dim() != 2 or mat2.dim() != 2:
        raise ValueError("input must be [M, K] and mat2 [K, N]")
    if mat2.shape[0] != input.shape[1]:
        raise ValueError("input and mat2 disagree on K")
    if scale_a.numel() != 1 or scale_b.numel() != 1:
        raise NotImplementedError("only tensor-wise (one-element) scales")
    if not input.is_contiguous():
        raise ValueError("input must be row-major ([M, K] with K contiguous)")
    b = mat2.t()  # [N, K]
    if not b.is_contiguous():
        raise ValueError("mat2 must be column-major ([K, N] with K contiguous, e.g. w.t() of a row-major weight)")
    fp8_out = out_dtype in (torch.float8_e4m3fn, torch.float8_e5m2)
    if scale_result is not None and not fp8_out:
        scale_result = None  # read only for FP8 outputs
    c, _ = scaled_mm(input, b, scale_a.reshape(1), scale_b.reshape(1), out_dtype=out_dtype,
                     use_fast_accum=use_fast_accum, scale_mode=FP8MM_SCALE_TENSOR, out=out, strict_torch=True,
                     bias=bias, scale_result=scale_result.reshape(1) if scale_result is not None else None)
    return c


def bmm_fp8(a, b, scale_a, scale_b, *, trans_b=False, out_dtype=None, use_fast_accum=False, out=None):
    """Batched FP8 GEMM d[i] = (a[i] @ b[i]) * scale_a * scale_b (TileOPs
    "Linear Algebra Operators", BmmFP8FwdOp).

    a is [B, M, K]; b is [B, K, N] (trans_b False, torch.bmm's order) or
    [B, N, K] (trans_b True); scale_a and scale_b are per-tensor fp32 (0-dim or
    one element); out_dtype defaults to bfloat16.  As on that page, b's
    strides, not trans_b, decide whether b is read in place: a b whose K axis
    is innermost goes to the GEMM as it is; a b stored [B, K, N] with N
    innermost is first copied into a K-major buffer by the library's
    transposing kernel (one extra read and write of b).  Other strides raise
    ValueError.  Returns d, [B, M, N] (use ``scaled_mm`` for the fused amax).
    """
    torch = _torch()
    if out_dtype is None:
        out_dtype = torch.bfloat16
    if a.dim() != 3 or b.dim() != 3:
        raise ValueError("a must be [B, M, K] and b [B, K, N] (or [B, N, K] with trans_b)")
    bnk = b if trans_b else b.transpose(1, 2)
    if bnk.shape[0] != a.shape[0] or bnk.shape[2] != a.shape[2]:
        raise ValueError("a and b disagree on the batch or on K")
    d, _ = scaled_mm(a, bnk, scale_a.reshape(1), scale_b.reshape(1), out_dtype=out_dtype,
                     use_fast_accum=use_fast_accum, scale_mode=FP8MM_SCALE_TENSOR, out=out)
    return d
