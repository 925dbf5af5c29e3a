"""Pins for the oracle's single rounding of a float64 value onto fp32/bf16/fp16.

Each format is checked against a library conversion that rounds once:
C/numpy double -> float32, numpy double -> float16 (rounded directly from the
double's bits), and torch float32 -> bfloat16 on inputs exact in float32.
"""
import math

import numpy as np
import torch

import oracle


def _samples(seed, lo, hi, n=4000):
    rng = np.random.default_rng(seed)
    e = rng.uniform(lo, hi, n)
    m = rng.uniform(1, 2, n)
    s = rng.choice([-1.0, 1.0], n)
    return s * m * np.exp2(e)


def test_round_f32_matches_c_cast():
    x = np.concatenate([_samples(1, -155, 130), [0.0, -0.0, np.inf, -np.inf, 3.4028235677973366e38,
                                                  3.4028235677973366e38 * (1 + 2 ** -25)]])
    ours = oracle.round_out(oracle.OUT_F32, x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float32).astype(np.float64)
    assert np.array_equal(ours, ref)


def test_round_f16_matches_numpy():
    x = np.concatenate([_samples(2, -28, 17), [65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25,
                                                2.0 ** -25 * 1.0001, 3 * 2.0 ** -26]])
    ours = oracle.round_out(oracle.OUT_F16, x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(ours, ref)
    assert oracle.round_out(oracle.OUT_F16, [65520.0])[0] == math.inf  # ties-to-even past max -> Inf


def test_round_bf16_matches_torch_on_f32_exact_inputs():
    x = _samples(3, -140, 127).astype(np.float32).astype(np.float64)
    # bf16 midpoints: exact in float32, so torch's float32 -> bf16 rounding is a single rounding
    base = torch.tensor(_samples(4, -120, 120, 2000), dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    ulp = np.exp2(np.floor(np.log2(np.abs(base))) - 7)
    mids = base + np.sign(base) * ulp / 2
    x = np.concatenate([x, mids, [3.3895313892515355e38, -3.3895313892515355e38]])
    ours = oracle.round_out(oracle.OUT_BF16, x)
    ref = torch.tensor(x, dtype=torch.float64).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    bf16_max = 3.3895313892515355e38
    # the midpoint between the largest finite bf16 and 2^128 ties to even, i.e. to Inf
    assert oracle.round_out(oracle.OUT_BF16, [bf16_max + 2.0 ** 119])[0] == math.inf
    assert oracle.round_out(oracle.OUT_BF16, [bf16_max + 2.0 ** 119 - 2.0 ** 100])[0] == bf16_max


def test_round_is_single_rounding_from_double():
    # 1 + 2^-8 + 2^-30 lies just above the bf16 midpoint 1 + 2^-8; rounding it
    # to fp32 first would land on the midpoint and tie down to 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert oracle.round_out(oracle.OUT_BF16, [x])[0] == 1.0 + 2.0 ** -7
    assert oracle.round_out(oracle.OUT_BF16, [1.0 + 2.0 ** -8])[0] == 1.0
