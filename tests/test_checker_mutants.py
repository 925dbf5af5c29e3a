"""The parity checker against mutated results (CPU only).

The GPU parity tests pass a result when every element lies within
K 2^-23 sum|a b| + half an ulp of the oracle's exact value, NaNs are canonical,
non-finite values match by class and amax equals max |C| of the stored result
bit for bit.  Here the "GPU" result is the oracle's own rounded output, which
must pass, and each mutant class of an epilogue (rounding, sign, dropped scale,
dropped K step, saturation, NaN payload, amax) must fail.  Mutants that stay
inside the bound are recorded as such: the order in which the scales are
applied, the accumulation order (fast against slow) and the sign of zero are
not part of the contract.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_matmul_gb300 import synth

from parity import check

_TORCH = {synth.OUT_F32: torch.float32, synth.OUT_BF16: torch.bfloat16, synth.OUT_F16: torch.float16}


def _oracle_out(p):
    ce, co, ab = oracle.scaled_gemm(p.a.numpy(), p.b.numpy(), p.scale_a.numpy(), p.scale_b.numpy(),
                                    a_fmt=p.a_fmt, b_fmt=p.b_fmt, scale_mode=p.scale_mode, out_dtype=p.out_dtype)
    return ce, co, ab


def _as_result(p, values):
    c = torch.as_tensor(np.asarray(values, dtype=np.float64)).to(_TORCH[p.out_dtype]).reshape(p.L, p.M, p.N)
    return c


def _amax_of(c):
    f = c.float()
    if torch.isnan(f).any():
        return torch.tensor([float("nan")]).view(torch.int32).fill_(0x7FFFFFFF).view(torch.float32)
    return f.abs().max().reshape(1)


def _passes(p, c, amax=None):
    try:
        check(p, c, _amax_of(c) if amax is None else amax)
        return True
    except AssertionError:
        return False


@pytest.fixture(scope="module")
def prob():
    return synth.llm_per_tensor(M=48, N=40, K=384, seed=41, fast_accum=True, out_dtype=synth.OUT_BF16)


def test_the_oracles_own_result_passes(prob):
    _, co, _ = _oracle_out(prob)
    assert _passes(prob, _as_result(prob, co))


def test_truncation_instead_of_round_to_nearest_is_caught(prob):
    ce, co, _ = _oracle_out(prob)
    # bf16 by truncating the fp32 value toward zero (drop the low 16 bits)
    t = torch.as_tensor(ce).to(torch.float32).view(torch.int32) & ~0xFFFF
    c = t.view(torch.float32).to(torch.bfloat16).reshape(prob.L, prob.M, prob.N)
    assert not torch.equal(c.float().double().flatten(), torch.as_tensor(co).flatten())  # the mutant differs
    assert not _passes(prob, c)


def test_one_flipped_sign_is_caught(prob):
    _, co, _ = _oracle_out(prob)
    v = co.copy().reshape(-1)
    i = int(np.argmax(np.abs(v)))
    v[i] = -v[i]
    assert not _passes(prob, _as_result(prob, v.reshape(co.shape)))


def test_a_dropped_scale_is_caught(prob):
    _, co, _ = _oracle_out(prob)
    s_b = float(prob.scale_b[0])
    assert s_b != 1.0
    assert not _passes(prob, _as_result(prob, co / s_b))


def test_a_dropped_k_step_is_caught(prob):
    q = synth.Problem(prob.name, prob.L, prob.M, prob.N, prob.K, prob.a.clone(), prob.b, prob.scale_a, prob.scale_b,
                      prob.a_fmt, prob.b_fmt, prob.scale_mode, prob.out_dtype, prob.fast_accum)
    q.a[..., -1] = 0  # the last K element of every row left out
    _, co_short, _ = _oracle_out(q)
    assert not _passes(prob, _as_result(prob, co_short))


def test_saturating_instead_of_overflowing_is_caught():
    p = synth.llm_per_tensor(M=16, N=16, K=256, seed=42, fast_accum=True, out_dtype=synth.OUT_F16)
    p.scale_a.fill_(16.0)
    p.scale_b.fill_(16.0)  # |C| far beyond fp16's 65504
    _, co, _ = _oracle_out(p)
    assert np.isinf(co).any()
    sat = np.where(np.isinf(co), np.sign(co) * 65504.0, co)
    assert _passes(p, _as_result(p, co))
    assert not _passes(p, _as_result(p, sat))


def test_non_canonical_nan_payload_is_caught():
    g = torch.Generator().manual_seed(43)
    a = synth.cast_fp8(torch.randn(1, 8, 32, generator=g), synth.E5M2)
    b = synth.cast_fp8(torch.randn(1, 8, 32, generator=g), synth.E5M2)
    a[0, 2, 3] = 0x7F  # a NaN code
    one = torch.tensor([1.0])
    p = synth.Problem("nan", 1, 8, 8, 32, a, b, one, one.clone(), synth.E5M2, synth.E5M2, synth.SCALE_TENSOR,
                      synth.OUT_BF16, True)
    _, co, _ = _oracle_out(p)
    c = _as_result(p, co)
    bits = c.view(torch.int16)
    bits[torch.isnan(c)] = 0x7FC1  # a quiet NaN with another payload
    assert torch.isnan(c.float()).any()
    assert not _passes(p, c)


def test_amax_of_the_unrounded_values_is_caught(prob):
    ce, co, _ = _oracle_out(prob)
    c = _as_result(prob, co)
    unrounded = torch.tensor([float(np.abs(ce).max())], dtype=torch.float32)
    assert int(unrounded.view(torch.int32)) != int(_amax_of(c).view(torch.int32))
    assert not _passes(prob, c, unrounded)


def test_inside_the_bound_scale_order(prob):
    # not part of the contract: alpha applied in another order
    ce, co, ab = _oracle_out(prob)
    s_a, s_b = float(prob.scale_a[0]), float(prob.scale_b[0])
    raw = ce / (s_a * s_b)
    other_order = (raw.astype(np.float32) * np.float32(s_a)).astype(np.float32) * np.float32(s_b)
    assert _passes(prob, _as_result(prob, oracle.round_out(prob.out_dtype, other_order.astype(np.float64))))


def _fp32_chain(a, b, chunk):
    """fp32 accumulation over K: one chain (chunk = K) or 128-K chunks whose
    fp32 partials are added into an fp32 accumulator."""
    M, K = a.shape
    acc = np.zeros((M, b.shape[0]), dtype=np.float32)
    for c0 in range(0, K, chunk):
        part = np.zeros_like(acc)
        for k in range(c0, min(K, c0 + chunk)):
            part = (part + np.outer(a[:, k], b[:, k]).astype(np.float32)).astype(np.float32)
        acc = (acc + part).astype(np.float32)
    return acc


@pytest.mark.parametrize("chunk", [384, 128])
def test_inside_the_bound_accumulation_order(prob, chunk):
    # fast (one fp32 chain) and slow (128-K chunks) orders of fp32 rounding both pass
    dt = torch.float8_e4m3fn
    a = prob.a[0].view(dt).to(torch.float64).numpy()
    b = prob.b[0].view(dt).to(torch.float64).numpy()
    acc = _fp32_chain(a, b, chunk).astype(np.float64)
    alpha = float(np.float32(float(prob.scale_a[0]) * float(prob.scale_b[0])))
    vals = oracle.round_out(prob.out_dtype, (np.float32(alpha) * acc.astype(np.float32)).astype(np.float64))
    assert _passes(prob, _as_result(prob, vals[None]))


def test_inside_the_bound_zero_sign():
    p = synth.llm_per_tensor(M=8, N=8, K=32, seed=44, fast_accum=True, out_dtype=synth.OUT_F32)
    p.a[0, 1, :] = 0  # row 1 of C is exactly zero
    _, co, _ = _oracle_out(p)
    v = co.copy()
    v[0, 1, :] = -0.0
    assert _passes(p, _as_result(p, v))
