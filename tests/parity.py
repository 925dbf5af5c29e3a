"""Shared helpers for the GPU parity tests: run a synthetic problem through the
C ABI and compare it with the CPU oracle under the stated error bound.

Bound (per element, finite oracle values):
    |C_gpu - C_exact| <= K * 2^-23 * sum_k |a_hat_k b_hat_k| + ulp_out(max(|C_exact|, |C_gpu|)) / 2
where C_exact is the oracle's unrounded float64 value.  Non-finite oracle
values are compared by class (NaN, +Inf, -Inf); NaN outputs must carry the
canonical bit pattern.  Amax must equal max |C| over the GPU's own C bit for
bit, and lie within the largest element bound of the oracle's max |C_exact|.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import precision_matmul_gb300 as pm
from precision_matmul_gb300 import synth

# (significand bits incl. the implicit one, exponent of the smallest normal)
_FMT = {synth.OUT_F32: (24, -126), synth.OUT_BF16: (8, -126), synth.OUT_F16: (11, -14)}
_NAN_BITS = {synth.OUT_F32: 0x7FFFFFFF, synth.OUT_BF16: 0x7FFF, synth.OUT_F16: 0x7FFF}


def half_ulp(out_dtype: int, x: np.ndarray) -> np.ndarray:
    p, emin = _FMT[out_dtype]
    ax = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.where(ax > 0, np.maximum(e, emin), emin)
    return np.exp2(e - (p - 1)) / 2


def element_bound(out_dtype: int, K: int, ce: np.ndarray, absum: np.ndarray, got: np.ndarray) -> np.ndarray:
    mag = np.maximum(np.abs(ce), np.nan_to_num(np.abs(got), posinf=0.0))
    return K * 2.0 ** -23 * absum + half_ulp(out_dtype, mag)


def to_device(p: synth.Problem, device="cuda:0"):
    dev = torch.device(device)
    return (p.a.to(dev), p.b.to(dev), p.scale_a.to(dev), p.scale_b.to(dev))


def run_gpu(p: synth.Problem, *, splitk=0, swap_ab=0, block_n=0, cta_pair=0, epi_warps=0, device="cuda:0",
            tensors=None):
    """One fp8mm_run through the C ABI; returns (C on device [L][M][N], amax tensor, plan)."""
    a, b, sa, sb = tensors if tensors is not None else to_device(p, device)
    c, amax = pm.scaled_mm(a, b, sa, sb, out_dtype=synth.OUT_TORCH[p.out_dtype],
                           use_fast_accum=p.fast_accum, a_fmt=p.a_fmt, b_fmt=p.b_fmt,
                           scale_mode=p.scale_mode, splitk=splitk, swap_ab=swap_ab, block_n=block_n,
                           cta_pair=cta_pair, epi_warps=epi_warps)
    key = (p.M, p.N, p.K, p.L, p.a_fmt, p.b_fmt, p.scale_mode, p.out_dtype, 1 if p.fast_accum else 0,
           splitk, swap_ab, block_n, torch.device(device).index or 0, cta_pair, epi_warps)
    return c, amax, pm.plan_for(key)


def amax_bits_of(c: torch.Tensor) -> int:
    """Bits of max |C| over a tensor, NaN -> canonical 0x7FFFFFFF, empty -> 0."""
    if c.numel() == 0:
        return 0
    f = c.float()
    if torch.isnan(f).any():
        return 0x7FFFFFFF
    return int(f.abs().max().view(torch.int32).item())


def check(p: synth.Problem, c: torch.Tensor, amax: torch.Tensor, *, rows=None, oracle_threads=None,
          full_amax=True):
    """Compare GPU output with the oracle on all rows (or the given row indices)."""
    c = c.reshape(p.L, p.M, p.N)
    a, b = p.a.numpy(), p.b.numpy()
    sa, sb = p.scale_a.numpy(), p.scale_b.numpy()
    if rows is None:
        rows_list = [(0, p.M)]
    else:
        rows_list = [(int(r), int(r) + 1) for r in rows]
    worst = 0.0
    global_tol = 0.0
    global_max = 0.0
    for (r0, r1) in rows_list:
        ce, co, ab = oracle.scaled_gemm(a, b, sa, sb, a_fmt=p.a_fmt, b_fmt=p.b_fmt,
                                        scale_mode=p.scale_mode, out_dtype=p.out_dtype, rows=(r0, r1),
                                        nthreads=oracle_threads)
        got_t = c[:, r0:r1, :].cpu()
        got = got_t.double().numpy()
        finite = np.isfinite(co)
        tol = element_bound(p.out_dtype, p.K, ce, ab, got)
        err = np.abs(got - ce)
        bad = finite & ~(err <= tol)
        if bad.any():
            idx = np.argwhere(bad)[:8]
            det = [(tuple(int(v) for v in i), float(got[tuple(i)]), float(ce[tuple(i)]), float(tol[tuple(i)]))
                   for i in idx]
            raise AssertionError(f"{int(bad.sum())} of {bad.size} elements outside the bound "
                                 f"(rows {r0}:{r1}); first (idx, gpu, oracle, tol): {det}")
        # non-finite classes
        nf = ~finite
        if nf.any():
            assert np.array_equal(np.isnan(got[nf]), np.isnan(co[nf])), "NaN positions differ"
            inf_or = np.isinf(co[nf])
            assert np.array_equal(got[nf][inf_or], co[nf][inf_or]), "Inf signs differ"
        # (a finite oracle value that became non-finite on the GPU fails the bound above)
        nan_mask = torch.isnan(got_t.float())
        if nan_mask.any():
            ib = got_t.view(torch.int32 if p.out_dtype == synth.OUT_F32 else torch.int16)
            bits = ib[nan_mask].to(torch.int64) & (0xFFFFFFFF if p.out_dtype == synth.OUT_F32 else 0xFFFF)
            assert (bits == _NAN_BITS[p.out_dtype]).all(), "non-canonical NaN payload"
        if finite.any():
            worst = max(worst, float(np.max(np.where(finite, err / np.maximum(tol, 1e-300), 0))))
            global_tol = max(global_tol, float(np.max(np.where(finite, tol, 0))))
            global_max = max(global_max, float(np.max(np.where(finite, np.abs(ce), 0))))
    # amax: bit-equal to max |C| over the GPU's own output
    got_amax_bits = int(amax.view(torch.int32).item())
    if full_amax:
        assert got_amax_bits == amax_bits_of(c), (hex(got_amax_bits), hex(amax_bits_of(c)))
    if rows is None:
        # within the bound of the oracle's max |C_exact| (when every stored value is finite: an
        # exact value that rounds to +-Inf in out_dtype makes amax +Inf on both sides)
        ce_all, co_all, _ = oracle.scaled_gemm(a, b, sa, sb, a_fmt=p.a_fmt, b_fmt=p.b_fmt,
                                               scale_mode=p.scale_mode, out_dtype=p.out_dtype,
                                               nthreads=oracle_threads)
        if np.isfinite(co_all).all():
            am = float(amax.item())
            assert abs(am - float(np.abs(ce_all).max())) <= global_tol + 1e-300
    return worst
