"""Shared helpers for the GPU parity tests: run a synthetic problem through the
C ABI and compare it with the CPU oracle under the stated error bound.

Bound (per element, finite oracle values):
    |C_gpu - C_exact| <= K * 2^-23 * sum_k |a_hat_k b_hat_k| + ulp_out(max(|C_exact|, |C_gpu|)) / 2
where C_exact is the oracle's unrounded float64 value.  With a bias the fp32
rounding of the addition adds 2^-23 |bias[n]|.  FP8 outputs compare with the
saturated target clip(scale_result * C_exact) and scale the accumulation term
by scale_result (see ``fp8_bound``).  Non-finite oracle values are compared
by class (NaN, +Inf, -Inf); NaN outputs must carry the canonical bit pattern.
Amax must equal max |C| over the GPU's own C bit for bit (for FP8 outputs:
the FP8 rounding of fp32(amax * scale_result) must equal max |C|, because
amax is taken before scale_result), and lie within the largest element bound
of the oracle's max |C_exact|.

Every check records its worst error / bound ratio; the test session prints
them (tests/conftest.py), so how close a case comes to the bound is visible.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import precision_matmul_gb300 as pm
from precision_matmul_gb300 import synth

# (significand bits incl. the implicit one, exponent of the smallest normal)
_FMT = {synth.OUT_F32: (24, -126), synth.OUT_BF16: (8, -126), synth.OUT_F16: (11, -14),
        synth.OUT_E4M3: (4, -6), synth.OUT_E5M2: (3, -14)}
_NAN_BITS = {synth.OUT_F32: 0x7FFFFFFF, synth.OUT_BF16: 0x7FFF, synth.OUT_F16: 0x7FFF}
_FP8_OUT = (synth.OUT_E4M3, synth.OUT_E5M2)

# (test id, worst error / bound, elements compared)
REPORT: list = []


def half_ulp(out_dtype: int, x: np.ndarray) -> np.ndarray:
    p, emin = _FMT[out_dtype]
    ax = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.where(ax > 0, np.maximum(e, emin), emin)
    return np.exp2(e - (p - 1)) / 2


def element_bound(out_dtype: int, K: int, ce: np.ndarray, absum: np.ndarray, got: np.ndarray,
                  bias: np.ndarray | None = None) -> np.ndarray:
    mag = np.maximum(np.abs(ce), np.nan_to_num(np.abs(got), posinf=0.0))
    tol = K * 2.0 ** -23 * absum + half_ulp(out_dtype, mag)
    if bias is not None:
        tol = tol + 2.0 ** -23 * np.abs(bias)
    return tol


def fp8_bound(out_dtype: int, K: int, target: np.ndarray, sr: float, absum: np.ndarray, got: np.ndarray,
              ce: np.ndarray) -> np.ndarray:
    """Bound for an FP8 output against target = clip(sr * C_exact, +-fmax): the
    accumulation error scaled by sr, the fp32 roundings of alpha * acc and of
    the product with sr (2^-23 |sr C_exact|), and half an FP8 ulp.  Clipping is
    1-Lipschitz, so the saturated GPU value stays inside the same bound."""
    mag = np.maximum(np.abs(target), np.nan_to_num(np.abs(got), posinf=0.0))
    return sr * K * 2.0 ** -23 * absum + 2.0 ** -23 * np.abs(sr * ce) + half_ulp(out_dtype, mag)


def to_device(p: synth.Problem, device="cuda:0"):
    dev = torch.device(device)
    return (p.a.to(dev), p.b.to(dev), p.scale_a.to(dev), p.scale_b.to(dev))


def run_gpu(p: synth.Problem, *, splitk=0, swap_ab=0, block_n=0, cta_pair=0, epi_warps=0, device="cuda:0",
            tensors=None, scale_result=None, bias=None):
    """One fp8mm_run through the C ABI; returns (C on device [L][M][N], amax tensor, plan)."""
    a, b, sa, sb = tensors if tensors is not None else to_device(p, device)
    dev = torch.device(device)
    kw = {}
    if scale_result is not None:
        kw["scale_result"] = torch.tensor([float(scale_result)], dtype=torch.float32, device=dev)
    if bias is not None:
        kw["bias"] = bias.to(dev)
    c, amax = pm.scaled_mm(a, b, sa, sb, out_dtype=synth.OUT_TORCH[p.out_dtype],
                           use_fast_accum=p.fast_accum, a_fmt=p.a_fmt, b_fmt=p.b_fmt,
                           scale_mode=p.scale_mode, splitk=splitk, swap_ab=swap_ab, block_n=block_n,
                           cta_pair=cta_pair, epi_warps=epi_warps, **kw)
    key = (p.M, p.N, p.K, p.L, p.a_fmt, p.b_fmt, p.scale_mode, p.out_dtype, 1 if p.fast_accum else 0,
           splitk, swap_ab, block_n, torch.device(device).index or 0, cta_pair, epi_warps, 0,
           1 if bias is not None else 0)
    return c, amax, pm.plan_for(key)


def amax_bits_of(c: torch.Tensor) -> int:
    """Bits of max |C| over a tensor, NaN -> canonical 0x7FFFFFFF, empty -> 0."""
    if c.numel() == 0:
        return 0
    f = c.float()
    if torch.isnan(f).any():
        return 0x7FFFFFFF
    return int(f.abs().max().view(torch.int32).item())


def _fp8_value(out_dtype: int, x: float) -> float:
    """The FP8 rounding (nearest even, saturating) of an fp32 number, via torch's cast."""
    fmax = 448.0 if out_dtype == synth.OUT_E4M3 else 57344.0
    t = torch.tensor([x], dtype=torch.float32).clamp(-fmax, fmax)
    return float(t.to(synth.OUT_TORCH[out_dtype]).float().item())


def _record(worst: float, count: int):
    name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    REPORT.append((name, worst, count))


def check(p: synth.Problem, c: torch.Tensor, amax: torch.Tensor, *, rows=None, oracle_threads=None,
          full_amax=True, block_rows=512, scale_result=None, bias=None):
    """Compare GPU output with the oracle on all rows (in blocks of
    ``block_rows``) or on the given row indices; with full_amax (the default)
    also check amax against the GPU's own C and the oracle's max.  Returns the
    worst error / bound ratio over the compared elements."""
    c = c.reshape(p.L, p.M, p.N)
    a, b = p.a.numpy(), p.b.numpy()
    sa, sb = p.scale_a.numpy(), p.scale_b.numpy()
    fp8_out = p.out_dtype in _FP8_OUT
    sr = 1.0 if scale_result is None else float(np.float32(scale_result))
    bias_np = None if bias is None else bias.double().numpy().reshape(-1)
    if rows is None:
        rows_list = [(r, min(p.M, r + block_rows)) for r in range(0, p.M, block_rows)]
    else:
        rows_list = [(int(r), int(r) + 1) for r in rows]
    worst = 0.0
    compared = 0
    global_tol = 0.0
    acc_tol = 0.0  # accumulation part of the bound alone (amax of an FP8 output is taken before the rounding)
    oracle_max = 0.0
    all_finite = True
    any_nan_exact = False
    for (r0, r1) in rows_list:
        ce, co, ab = oracle.scaled_gemm(a, b, sa, sb, a_fmt=p.a_fmt, b_fmt=p.b_fmt,
                                        scale_mode=p.scale_mode, out_dtype=p.out_dtype, rows=(r0, r1),
                                        nthreads=oracle_threads, scale_result=scale_result, bias=bias_np)
        got_t = c[:, r0:r1, :].cpu()
        got = got_t.float().double().numpy()
        if fp8_out:
            fmax = 448.0 if p.out_dtype == synth.OUT_E4M3 else 57344.0
            target = np.clip(sr * ce, -fmax, fmax)
            finite = np.isfinite(ce)
            tol = fp8_bound(p.out_dtype, p.K, target, sr, ab, got, ce)
            err = np.abs(got - target)
        else:
            finite = np.isfinite(co)
            tol = element_bound(p.out_dtype, p.K, ce, ab, got, bias_np)
            err = np.abs(got - ce)
        bad = finite & ~(err <= tol)
        if bad.any():
            idx = np.argwhere(bad)[:8]
            det = [(tuple(int(v) for v in i), float(got[tuple(i)]), float(ce[tuple(i)]), float(tol[tuple(i)]))
                   for i in idx]
            raise AssertionError(f"{int(bad.sum())} of {bad.size} elements outside the bound "
                                 f"(rows {r0}:{r1}); first (idx, gpu, oracle, tol): {det}")
        # non-finite classes (FP8 outputs saturate Inf to +-fmax; NaN stays NaN)
        nf = ~finite
        if nf.any():
            if fp8_out:
                assert np.array_equal(np.isnan(got[nf]), np.isnan(ce[nf])), "NaN positions differ"
                inf_or = np.isinf(ce[nf])
                assert np.array_equal(got[nf][inf_or], np.sign(sr * ce[nf][inf_or]) * fmax), "saturation of Inf"
            else:
                assert np.array_equal(np.isnan(got[nf]), np.isnan(co[nf])), "NaN positions differ"
                inf_or = np.isinf(co[nf])
                assert np.array_equal(got[nf][inf_or], co[nf][inf_or]), "Inf signs differ"
        # (a finite oracle value that became non-finite on the GPU fails the bound above)
        nan_mask = torch.isnan(got_t.float())
        if nan_mask.any() and not fp8_out:
            ib = got_t.view(torch.int32 if p.out_dtype == synth.OUT_F32 else torch.int16)
            bits = ib[nan_mask].to(torch.int64) & (0xFFFFFFFF if p.out_dtype == synth.OUT_F32 else 0xFFFF)
            assert (bits == _NAN_BITS[p.out_dtype]).all(), "non-canonical NaN payload"
        if finite.any():
            worst = max(worst, float(np.max(np.where(finite, err / np.maximum(tol, 1e-300), 0))))
            global_tol = max(global_tol, float(np.max(np.where(finite, tol, 0))))
            at = p.K * 2.0 ** -23 * ab + 2.0 ** -23 * np.abs(ce)
            acc_tol = max(acc_tol, float(np.max(np.where(finite, at, 0))))
            oracle_max = max(oracle_max, float(np.max(np.where(finite, np.abs(ce), 0))))
        compared += int(finite.sum())
        all_finite = all_finite and bool(np.isfinite(co).all())
        any_nan_exact = any_nan_exact or bool(np.isnan(ce).any())
    got_amax_bits = int(amax.view(torch.int32).item())
    if full_amax:
        if fp8_out:
            # amax is max |C| before scale_result and the FP8 rounding; rounding is
            # monotone, so the largest stored magnitude is the rounding of amax * sr
            am = float(amax.item())
            if any_nan_exact:
                assert got_amax_bits == 0x7FFFFFFF
            else:
                stored = float(c.float().abs().max().item()) if c.numel() else 0.0
                want = _fp8_value(p.out_dtype, float(np.float32(np.float32(am) * np.float32(sr))))
                assert abs(want) == stored, (am, sr, want, stored)
        else:
            # bit-equal to max |C| over the GPU's own output
            assert got_amax_bits == amax_bits_of(c), (hex(got_amax_bits), hex(amax_bits_of(c)))
    if full_amax and rows is None and all_finite and not any_nan_exact:
        # within the bound of the oracle's max |C_exact| (when every stored value is finite: an
        # exact value that rounds to +-Inf in out_dtype makes amax +Inf on both sides)
        am = float(amax.item())
        slack = global_tol if not fp8_out else acc_tol
        assert abs(am - oracle_max) <= slack + 1e-300, (am, oracle_max, slack)
    _record(worst, compared)
    return worst
