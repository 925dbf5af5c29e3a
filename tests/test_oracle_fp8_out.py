"""Pins for the oracle's FP8 outputs and scale_result.

The pages allow float8_e4m3fn / float8_e5m2 as out_dtype and use scale_result
for FP8 outputs only (mmaemu "API reference (v0.1)", mmaemu.scaled_mm).  The
readings pinned here: the result is multiplied by scale_result and rounded once
to nearest even on the FP8 grid, saturating at the largest finite value (Inf
included); NaN stays NaN; other outputs ignore scale_result.  The independent
routes are torch's float32 -> float8 casts (round to nearest even) on inputs
exact in float32, and the FP8 value tables.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from precision_matmul_gb300 import synth

_FP8 = {oracle.OUT_E4M3: (torch.float8_e4m3fn, 448.0, oracle.FMT_E4M3),
        oracle.OUT_E5M2: (torch.float8_e5m2, 57344.0, oracle.FMT_E5M2)}


def _torch_round(out, x):
    """torch's cast of float32 values already inside the format's range."""
    dt, fmax, _ = _FP8[out]
    t = torch.tensor(np.asarray(x, dtype=np.float64), dtype=torch.float32)
    assert (t.abs() <= fmax).all()
    return t.to(dt).to(torch.float64).numpy()


def _finite_values(out):
    _, _, fmt = _FP8[out]
    v = oracle.decode(fmt, np.arange(256, dtype=np.uint8))
    return np.unique(v[np.isfinite(v)])


@pytest.mark.parametrize("out", [oracle.OUT_E4M3, oracle.OUT_E5M2])
def test_every_fp8_value_rounds_to_itself(out):
    v = _finite_values(out)
    assert np.array_equal(oracle.round_out(out, v), v)


@pytest.mark.parametrize("out", [oracle.OUT_E4M3, oracle.OUT_E5M2])
def test_midpoints_and_neighbours_match_torch(out):
    v = _finite_values(out)
    v = v[v >= 0]
    mids = (v[1:] + v[:-1]) / 2          # ties: to the even neighbour
    eps = np.diff(v) / 8
    x = np.concatenate([mids, mids + eps, mids - eps])
    x = np.concatenate([x, -x])
    ours = oracle.round_out(out, x)
    assert np.array_equal(ours, _torch_round(out, x))


@pytest.mark.parametrize("out", [oracle.OUT_E4M3, oracle.OUT_E5M2])
def test_saturation_and_special_values(out):
    _, fmax, _ = _FP8[out]
    big = [fmax * 1.03, fmax * 1.5, fmax * 1e6, math.inf]
    assert list(oracle.round_out(out, big)) == [fmax] * 4
    assert list(oracle.round_out(out, [-b for b in big])) == [-fmax] * 4
    assert math.isnan(oracle.round_out(out, [math.nan])[0])
    z = oracle.round_out(out, [-0.0, 2.0 ** -40])
    assert z[0] == 0.0 and math.copysign(1.0, z[0]) == -1.0 and z[1] == 0.0


@pytest.mark.parametrize("out", [oracle.OUT_E4M3, oracle.OUT_E5M2])
@pytest.mark.parametrize("sr", [0.125, 0.75, 3.0, 16384.0])
def test_scale_result_multiplies_before_the_rounding(out, sr):
    # Integer operands in [-8, 8] (exact in E4M3) and K = 64 give integer sums
    # below 2^12; with power-of-two tensor scales and these scale_result values
    # C * sr is exact in float32, so torch's float32 -> FP8 cast rounds it once.
    g = torch.Generator().manual_seed(51)
    M, N, K = 24, 40, 64
    a = synth.cast_fp8(torch.randint(-8, 9, (1, M, K), generator=g).float(), synth.E4M3).numpy()
    b = synth.cast_fp8(torch.randint(-8, 9, (1, N, K), generator=g).float(), synth.E4M3).numpy()
    sa, sb = np.array([2.0 ** -6], np.float32), np.array([2.0 ** -5], np.float32)
    ce, co, _ = oracle.scaled_gemm(a, b, sa, sb, out_dtype=out, scale_result=sr)
    _, fmax, _ = _FP8[out]
    x = ce * sr
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)
    inside = np.abs(x) <= fmax
    assert inside.any()
    assert np.array_equal(co[inside], _torch_round(out, x[inside]))
    assert np.all(co[~inside] == np.sign(x[~inside]) * fmax)
    if sr == 16384.0 and out == oracle.OUT_E4M3:
        assert (~inside).any()                        # saturation is exercised
    # a divided (or ignored) scale_result gives other values
    assert not np.array_equal(co, oracle.round_out(out, ce / sr))


def test_other_outputs_ignore_scale_result():
    p = synth.llm_per_tensor(M=16, N=24, K=128, seed=52, out_dtype=synth.OUT_BF16)
    a, b, sa, sb = p.a.numpy(), p.b.numpy(), p.scale_a.numpy(), p.scale_b.numpy()
    for out in (oracle.OUT_F32, oracle.OUT_BF16, oracle.OUT_F16):
        ref = oracle.scaled_gemm(a, b, sa, sb, out_dtype=out)
        got = oracle.scaled_gemm(a, b, sa, sb, out_dtype=out, scale_result=4.0)
        for x, y in zip(ref, got):
            assert np.array_equal(x, y)


def test_amax_before_quantization():
    p = synth.llm_per_tensor(M=16, N=24, K=128, seed=53)
    ce, co, _ = oracle.scaled_gemm(p.a.numpy(), p.b.numpy(), p.scale_a.numpy(), p.scale_b.numpy(),
                                   out_dtype=oracle.OUT_E4M3, scale_result=0.5)
    am = oracle.amax_before_quantization(ce)
    assert am == float(np.float32(np.abs(ce).max()))
    assert am != oracle.amax(co)                      # not the amax of the stored FP8 values
    assert math.isnan(oracle.amax_before_quantization(np.array([1.0, math.nan])))
