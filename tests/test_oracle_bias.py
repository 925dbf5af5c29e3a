"""Pins for the oracle's bias term (a row the scope table marks next).

TileOPs "Linear Algebra Operators", GemmFP8FwdOp: d = (a s_a) @ (b s_b)^T + bias
with bias [N] in out_dtype.  Reading: the bias value of column n is added to
the exact scaled product of every row (and every batch), before the one
rounding to out_dtype.  Checked against exact rationals on tiny K, against the
bias alone when A is zero, and against the unbiased result when the bias is 0.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from precision_matmul_gb300 import synth


def _bias(N, out, seed):
    g = torch.Generator().manual_seed(seed)
    v = torch.exp2(torch.randint(-4, 5, (N,), generator=g).float()) * (torch.rand(N, generator=g) * 2 - 1)
    dt = {oracle.OUT_F32: torch.float32, oracle.OUT_BF16: torch.bfloat16, oracle.OUT_F16: torch.float16}[out]
    return v.to(dt).double().numpy()                       # values of the output type


@pytest.mark.parametrize("out", [oracle.OUT_F32, oracle.OUT_BF16, oracle.OUT_F16])
def test_tiny_k_exact_rationals_with_bias(out):
    p = synth.random_codes(M=5, N=7, K=6, seed=61)
    a, b = p.a.numpy()[0], p.b.numpy()[0]
    sa, sb = np.array([0.5], np.float32), np.array([4.0], np.float32)
    bias = _bias(7, out, 62)
    ce, co, _ = oracle.scaled_gemm(a, b, sa, sb, out_dtype=out, bias=bias)
    A = torch.as_tensor(a).view(torch.float8_e4m3fn).double().numpy()
    B = torch.as_tensor(b).view(torch.float8_e4m3fn).double().numpy()
    for m in range(5):
        for n in range(7):
            want = Fraction(2) * sum((Fraction(A[m, k]) * Fraction(B[n, k]) for k in range(6)), Fraction(0))
            want += Fraction(bias[n])                       # column n's bias, every row
            assert Fraction(ce[m, n]) == want
            assert co[m, n] == oracle.round_out(out, [float(want)])[0]


@pytest.mark.parametrize("out", [oracle.OUT_F32, oracle.OUT_BF16, oracle.OUT_F16])
def test_zero_operands_give_the_bias(out):
    L, M, N, K = 2, 3, 9, 32
    a = np.zeros((L, M, K), np.uint8)
    b = np.zeros((L, N, K), np.uint8)
    one = np.array([1.0], np.float32)
    bias = _bias(N, out, 63)
    _, co, _ = oracle.scaled_gemm(a, b, one, one, out_dtype=out, bias=bias)
    assert np.array_equal(co, np.broadcast_to(bias, (L, M, N)))


def test_zero_bias_changes_nothing():
    p = synth.blockwise(M=40, N=136, K=300, seed=64, b_block=128)
    args = (p.a.numpy(), p.b.numpy(), p.scale_a.numpy(), p.scale_b.numpy())
    kw = dict(scale_mode=p.scale_mode, out_dtype=oracle.OUT_BF16)
    ref = oracle.scaled_gemm(*args, **kw)
    got = oracle.scaled_gemm(*args, bias=np.zeros(136), **kw)
    for x, y in zip(ref, got):
        assert np.array_equal(x, y)


def test_bias_arguments():
    p = synth.random_codes(M=4, N=6, K=16, seed=65)
    a, b = p.a.numpy()[0], p.b.numpy()[0]
    one = np.array([1.0], np.float32)
    with pytest.raises(ValueError):
        oracle.scaled_gemm(a, b, one, one, bias=np.zeros(4))           # one value per column
    with pytest.raises(ValueError):                                    # the pages define no FP8 output bias
        oracle.scaled_gemm(a, b, one, one, out_dtype=oracle.OUT_E4M3, bias=np.zeros(6))
