"""Pins for the oracle's scaled GEMM and amax.

Each check reaches the expected value by a route that shares nothing with the
oracle's C code: exact rationals (``fractions.Fraction``) on tiny K, torch's
float64 matmul where the float64 sum is exact, algebraic invariants (power-of-
two scale linearity, layout equivalence, constant block scales = per-tensor,
unit MX factors = per-tensor), the page's own logical-to-physical
permutation of the MX scale-factor atoms and torch's layout routine for the
same factors.
"""
from fractions import Fraction
import math

import numpy as np
import pytest
import torch

import library_refs
import oracle
from precision_matmul_gb300 import synth


def _dec(codes, fmt):
    dt = torch.float8_e5m2 if fmt == oracle.FMT_E5M2 else torch.float8_e4m3fn
    return torch.as_tensor(np.asarray(codes, dtype=np.uint8)).view(dt).to(torch.float64).numpy()


def _np(p):
    return (p.a.numpy(), p.b.numpy(), p.scale_a.numpy(), p.scale_b.numpy())


def _run(p, **kw):
    a, b, sa, sb = _np(p)
    kw.setdefault("a_fmt", p.a_fmt)
    kw.setdefault("b_fmt", p.b_fmt)
    kw.setdefault("scale_mode", p.scale_mode)
    kw.setdefault("out_dtype", p.out_dtype)
    return oracle.scaled_gemm(a, b, sa, sb, **kw)


# ---------------------------------------------------------------------------
# exact rationals on tiny K
# ---------------------------------------------------------------------------

def _fraction_gemm(A, B, fa, fb, scale_fn):
    """Exact sum_c S_A S_B sum_{k in c} a b with a chunk of 128; scale_fn(m, n, c) -> (sa, sb)."""
    Ad, Bd = _dec(A, fa), _dec(B, fb)
    M, K = A.shape
    N = B.shape[0]
    out = np.empty((M, N), dtype=object)
    absum = np.empty((M, N), dtype=object)
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            ab = Fraction(0)
            for c in range((K + 127) // 128):
                sa, sb = scale_fn(m, n, c)
                s = Fraction(sa) * Fraction(sb)
                part = sum((Fraction(Ad[m, k]) * Fraction(Bd[n, k]) for k in range(c * 128, min(K, c * 128 + 128))),
                           Fraction(0))
                apart = sum((abs(Fraction(Ad[m, k]) * Fraction(Bd[n, k])) for k in range(c * 128, min(K, c * 128 + 128))),
                            Fraction(0))
                tot += s * part
                ab += abs(s) * apart
            out[m, n] = tot
            absum[m, n] = ab
    return out, absum


@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E5M2])
@pytest.mark.parametrize("K", [1, 2, 5, 8])
def test_tiny_k_exact_per_tensor_pow2_scales(fmt, K):
    p = synth.random_codes(M=6, N=5, K=K, seed=100 + K, fmt=fmt)
    sa, sb = np.array([0.25], np.float32), np.array([8.0], np.float32)
    a, b = p.a.numpy()[0], p.b.numpy()[0]
    ce, co, ab = oracle.scaled_gemm(a, b, sa, sb, a_fmt=fmt, b_fmt=fmt, out_dtype=oracle.OUT_BF16)
    ref, refab = _fraction_gemm(a, b, fmt, fmt, lambda m, n, c: (0.25, 8.0))
    for m in range(6):
        for n in range(5):
            if fmt == oracle.FMT_E4M3:
                # E4M3 products are multiples of 2^-18 below 2^18: the float64 sum is exact
                assert Fraction(ce[m, n]) == ref[m, n]
                assert Fraction(ab[m, n]) == refab[m, n]
                assert co[m, n] == float(torch.tensor(float(ref[m, n]), dtype=torch.float64)
                                         .to(torch.float32).to(torch.bfloat16).float())
            else:
                # E5M2 products span 2^-32 .. 2^31: float64 rounds each of the K-1 adds
                tol = refab[m, n] * K * Fraction(1, 2 ** 53)
                assert abs(Fraction(ce[m, n]) - ref[m, n]) <= tol
                assert abs(Fraction(ab[m, n]) - refab[m, n]) <= tol


def test_tiny_k_random_scales_one_rounding():
    p = synth.random_codes(M=4, N=4, K=7, seed=7)
    a, b = p.a.numpy()[0], p.b.numpy()[0]
    sa, sb = np.array([0.3711], np.float32), np.array([2.718], np.float32)
    ce, co, ab = oracle.scaled_gemm(a, b, sa, sb)
    ref, _ = _fraction_gemm(a, b, 0, 0, lambda m, n, c: (float(sa[0]), float(sb[0])))
    for m in range(4):
        for n in range(4):
            # s_a*s_b is exact in float64, the sum is exact, one rounding of the product
            assert abs(Fraction(ce[m, n]) - ref[m, n]) <= abs(ref[m, n]) * Fraction(1, 2 ** 53)


@pytest.mark.parametrize("mode", [oracle.SCALE_A1x128_B1x128, oracle.SCALE_A1x128_B128x128])
def test_blockwise_chunks_exact_rationals(mode):
    # K = 300 spans three chunks of 128 with a ragged last chunk of 44; N = 130
    # spans two 128-row blocks of B's scales.
    g = torch.Generator().manual_seed(9)
    M, N, K = 3, 130, 300
    KB = 3
    a = synth.cast_fp8(torch.randn(M, K, generator=g) * 30, synth.E4M3).numpy()
    b = synth.cast_fp8(torch.randn(N, K, generator=g) * 30, synth.E4M3).numpy()
    sa = torch.exp2(torch.randint(-4, 5, (1, M, KB), generator=g).float()).numpy()
    if mode == oracle.SCALE_A1x128_B1x128:
        sb = torch.exp2(torch.randint(-4, 5, (1, N, KB), generator=g).float()).numpy()
        sfn = lambda m, n, c: (float(sa[0, m, c]), float(sb[0, n, c]))
    else:
        sb = torch.exp2(torch.randint(-4, 5, (1, 2, KB), generator=g).float()).numpy()
        sfn = lambda m, n, c: (float(sa[0, m, c]), float(sb[0, n // 128, c]))
    ce, co, ab = oracle.scaled_gemm(a, b, sa, sb, scale_mode=mode)
    cols = [0, 1, 64, 127, 128, 129]
    ref, refab = _fraction_gemm(a, b[cols], 0, 0, lambda m, j, c: sfn(m, cols[j], c))
    for m in range(M):
        for j, n in enumerate(cols):
            assert Fraction(ce[m, n]) == ref[m, j]
            assert Fraction(ab[m, n]) == refab[m, j]


def test_special_values_follow_ieee():
    # E5M2: Inf * 0 = NaN, Inf + finite = Inf, Inf - Inf = NaN; NaN codes propagate
    inf, ninf, one, zero, nan = 0x7C, 0xFC, 0x3C, 0x00, 0x7F
    a = np.array([[inf, zero], [inf, one], [inf, inf], [nan, zero], [one, one]], np.uint8)
    b = np.array([[zero, one], [one, one], [one, zero], [one, one]], np.uint8)
    b[3] = [ninf, one]
    one32 = np.array([1.0], np.float32)
    ce, co, _ = oracle.scaled_gemm(a, b, one32, one32, a_fmt=1, b_fmt=1)
    assert math.isnan(ce[0, 0])                 # inf*0 + 0*1
    assert ce[1, 1] == math.inf                 # inf*1 + 1*1
    assert math.isnan(ce[2, 3])                 # inf*(-inf) + inf*1 -> -inf + inf
    assert all(math.isnan(v) for v in ce[3])    # NaN code
    assert ce[4, 3] == -math.inf
    assert oracle.amax(co) != oracle.amax(co)   # NaN amax


# ---------------------------------------------------------------------------
# cases that reduce to a library routine
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("maker", [
    lambda: synth.random_codes(16, 8, 64),
    lambda: synth.adversarial_codes(64, 64, 256),
    lambda: synth.tiny_per_tensor(M=64, N=48, K=256),
])
def test_e4m3_per_tensor_equals_float64_matmul(maker):
    # E4M3 products are multiples of 2^-18 below 2^18, so any float64 order of
    # summation is exact for these K: torch's float64 matmul must agree bit for bit.
    p = maker()
    ce, co, ab = _run(p)
    A = torch.as_tensor(p.a.numpy()[0]).view(torch.float8_e4m3fn).double()
    B = torch.as_tensor(p.b.numpy()[0]).view(torch.float8_e4m3fn).double()
    acc = (A @ B.T).numpy()
    s = float(p.scale_a[0]) * float(p.scale_b[0])
    assert np.array_equal(ce[0], s * acc)
    assert np.array_equal(ab[0], abs(s) * (A.abs() @ B.abs().T).numpy())
    assert np.array_equal(co[0], (s * acc).astype(np.float32).astype(np.float64))


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_pow2_scale_linearity_bit_exact():
    p = synth.llm_per_tensor(M=40, N=36, K=512, seed=21, out_dtype=synth.OUT_BF16)
    a, b, sa, sb = _np(p)
    base = oracle.scaled_gemm(a, b, sa, sb, out_dtype=oracle.OUT_BF16)
    for pa, pb in [(3, 0), (0, -5), (7, -2)]:
        sa2 = (sa * np.float32(2.0 ** pa)).astype(np.float32)
        sb2 = (sb * np.float32(2.0 ** pb)).astype(np.float32)
        got = oracle.scaled_gemm(a, b, sa2, sb2, out_dtype=oracle.OUT_BF16)
        f = 2.0 ** (pa + pb)
        assert np.array_equal(got[0], base[0] * f)
        assert np.array_equal(got[1], base[1] * f)
        assert np.array_equal(got[2], base[2] * f)


def test_layout_equivalence_nt_nn_tn_tt():
    # TileOPs GemmFwdOp layout table: NT d = a b^T, NN d = a b, TN d = a^T b, TT d = a^T b^T.
    # Feeding the same logical operands through transposed storage must not change a bit.
    p = synth.random_codes(M=20, N=12, K=72, seed=31)
    a, b = p.a.numpy()[0], p.b.numpy()[0]
    one = np.array([1.0], np.float32)
    nt = oracle.scaled_gemm(a, b, one, one)[0]
    a_km = np.ascontiguousarray(a.T)   # stored [K][M] (the "T" of TN/TT)
    b_kn = np.ascontiguousarray(b.T)   # stored [K][N] (the "N" of NN/TN)
    nn = oracle.scaled_gemm(a, b_kn.T, one, one)[0]
    tn = oracle.scaled_gemm(a_km.T, b_kn.T, one, one)[0]
    tt = oracle.scaled_gemm(a_km.T, b, one, one)[0]
    for other in (nn, tn, tt):
        assert np.array_equal(nt, other)
    # and the transposed product really is a different function (a transposed
    # operand would be caught): C^T = B A^T
    ct = oracle.scaled_gemm(b, a, one, one)[0]
    assert np.array_equal(ct, nt.T)


@pytest.mark.parametrize("mode", [oracle.SCALE_A1x128_B1x128, oracle.SCALE_A1x128_B128x128])
def test_constant_block_scales_equal_per_tensor(mode):
    p = synth.llm_per_tensor(M=24, N=130, K=384, seed=41)
    a, b = p.a.numpy()[0], p.b.numpy()[0]
    sa_t, sb_t = np.array([0.5], np.float32), np.array([4.0], np.float32)
    ref = oracle.scaled_gemm(a, b, sa_t, sb_t, out_dtype=oracle.OUT_BF16)
    KB = 3
    sa = np.full((1, 24, KB), 0.5, np.float32)
    sb = np.full((1, 130 if mode == oracle.SCALE_A1x128_B1x128 else 2, KB), 4.0, np.float32)
    got = oracle.scaled_gemm(a, b, sa, sb, scale_mode=mode, out_dtype=oracle.OUT_BF16)
    for x, y in zip(ref, got):
        assert np.array_equal(x, y)


def test_mx_unit_factors_equal_per_tensor():
    # all UE8M0 codes 127 (= 1.0), as in the cuDNN page's JAX example
    p = synth.mx_batched(L=2, M=130, N=72, K=256, seed=51)
    a, b = p.a.numpy(), p.b.numpy()
    sfa = np.full_like(p.scale_a.numpy(), 127)
    sfb = np.full_like(p.scale_b.numpy(), 127)
    one = np.array([1.0], np.float32)
    got = oracle.scaled_gemm(a, b, sfa, sfb, scale_mode=oracle.SCALE_MX32_UE8M0)
    ref = oracle.scaled_gemm(a, b, one, one)
    for x, y in zip(ref, got):
        assert np.array_equal(x, y)


def test_mx_factor_layout_through_page_permutation(facts):
    # Build the factors in the page's LOGICAL shape (32, 4, MB, 4, KB, L) from a
    # known function of (row, factor index), turn them into the physical
    # allocation with torch.permute (the page: logical = physical permuted by
    # (3, 4, 1, 5, 2, 0)), and compare the oracle with a float64 dequantize-
    # then-matmul done by torch on per-element scales.
    assert facts["sf_logical_from_physical_perm"] == "3,4,1,5,2,0"
    perm = (3, 4, 1, 5, 2, 0)
    inv = tuple(perm.index(i) for i in range(6))
    L, M, N, K = 2, 200, 136, 384
    p = synth.mx_batched(L=L, M=M, N=N, K=K, seed=61)
    a, b = p.a.numpy(), p.b.numpy()

    def factors(R, salt):
        MB, KB = (R + 127) // 128, (K + 127) // 128
        i32 = torch.arange(32).view(32, 1, 1, 1, 1, 1)
        i4 = torch.arange(4).view(1, 4, 1, 1, 1, 1)
        mb = torch.arange(MB).view(1, 1, MB, 1, 1, 1)
        j4 = torch.arange(4).view(1, 1, 1, 4, 1, 1)
        kb = torch.arange(KB).view(1, 1, 1, 1, KB, 1)
        ll = torch.arange(L).view(1, 1, 1, 1, 1, L)
        row = i32 + 32 * i4 + 128 * mb          # reading: first logical index fastest
        f = j4 + 4 * kb
        logical = (127 + ((row * 7 + f * 3 + ll * 5 + salt) % 13) - 6).to(torch.uint8)
        physical = logical.permute(*inv).contiguous()
        assert tuple(physical.permute(*perm).shape) == tuple(logical.shape)
        assert torch.equal(physical.permute(*perm), logical)
        per_elem = torch.empty(L, R, K, dtype=torch.float64)
        rr = torch.arange(R).view(R, 1)
        kk = torch.arange(K).view(1, K)
        for l in range(L):
            code = 127 + ((rr * 7 + (kk // 32) * 3 + l * 5 + salt) % 13) - 6
            per_elem[l] = torch.exp2((code - 127).double())
        return physical.numpy(), per_elem

    sfa, ea = factors(M, 1)
    sfb, eb = factors(N, 4)
    ce, co, ab = oracle.scaled_gemm(a, b, sfa, sfb, scale_mode=oracle.SCALE_MX32_UE8M0)
    Ah = torch.as_tensor(a).view(torch.float8_e4m3fn).double() * ea
    Bh = torch.as_tensor(b).view(torch.float8_e4m3fn).double() * eb
    ref = torch.bmm(Ah, Bh.transpose(1, 2)).numpy()
    refab = torch.bmm(Ah.abs(), Bh.abs().transpose(1, 2)).numpy()
    assert np.all(np.abs(ce - ref) <= refab * K * 2.0 ** -52)
    assert np.allclose(ab, refab, rtol=1e-12, atol=0)


def test_mx_factor_layout_matches_the_library_blocked_layout():
    # The row order inside one 128-row atom (row = i32 + 32*i4) is a reading of
    # the page's logical modes.  torch lays out the same hardware factors with
    # an implementation of its own; factors placed by it must give the oracle
    # the per-element dequantize-then-matmul result.
    to_blocked = library_refs.get("to_blocked")
    L, M, N, K = 2, 200, 136, 416  # ragged rows, factor columns padded to a multiple of 4
    p = synth.mx_batched(L=L, M=M, N=N, K=K, seed=62)
    a, b = p.a.numpy(), p.b.numpy()
    g = torch.Generator().manual_seed(63)

    def factors(R):
        codes = torch.randint(121, 134, (L, R, (K + 31) // 32), generator=g, dtype=torch.int32)
        phys = torch.cat([to_blocked(codes[l]) for l in range(L)]).to(torch.uint8)
        per_elem = torch.exp2((codes.double() - 127).repeat_interleave(32, dim=2)[:, :, :K])
        return phys.numpy(), per_elem

    sfa, ea = factors(M)
    sfb, eb = factors(N)
    assert sfa.size == L * ((M + 127) // 128) * ((K + 127) // 128) * 512
    ce, _, ab = oracle.scaled_gemm(a, b, sfa, sfb, scale_mode=oracle.SCALE_MX32_UE8M0)
    Ah = torch.as_tensor(a).view(torch.float8_e4m3fn).double() * ea
    Bh = torch.as_tensor(b).view(torch.float8_e4m3fn).double() * eb
    ref = torch.bmm(Ah, Bh.transpose(1, 2)).numpy()
    refab = torch.bmm(Ah.abs(), Bh.abs().transpose(1, 2)).numpy()
    assert np.all(np.abs(ce - ref) <= refab * K * 2.0 ** -52)
    # another row order inside the atom (i4 fastest) gives another result
    MB, KB = (M + 127) // 128, (K + 127) // 128
    swapped = sfa.reshape(L, MB, KB, 32, 4, 4).transpose(0, 1, 2, 4, 3, 5).copy().reshape(-1)
    assert not np.array_equal(swapped, sfa)
    ce_s = oracle.scaled_gemm(a, b, swapped, sfb, scale_mode=oracle.SCALE_MX32_UE8M0)[0]
    assert not np.all(np.abs(ce_s - ref) <= refab * K * 2.0 ** -52)


def test_amax_definition():
    p = synth.llm_per_tensor(M=33, N=17, K=256, seed=71)
    ce, co, _ = _run(p)
    assert oracle.amax(co) == float(np.abs(co).max())
    assert oracle.amax(np.zeros((0, 5))) == 0.0
    z = oracle.amax(np.array([-0.0, -0.0]))
    assert z == 0.0 and math.copysign(1.0, z) == 1.0
    assert oracle.amax(np.array([1.0, -math.inf, 3.0])) == math.inf
    assert math.isnan(oracle.amax(np.array([1.0, math.nan, math.inf])))


def test_row_subset_equals_full():
    p = synth.llm_per_tensor(M=50, N=20, K=256, seed=81)
    full = _run(p)
    part = _run(p, rows=(17, 31))
    for x, y in zip(full, part):
        assert np.array_equal(x[:, 17:31], y)


def test_planted_mistakes_are_caught():
    # A plausible slip anywhere (dropped chunk scale, sign flip, transposed
    # operand) must break one of the pins above; check the ones cheap to
    # plant here against the float64 matmul route.
    p = synth.random_codes(16, 8, 64, seed=91)
    a, b = p.a.numpy()[0], p.b.numpy()[0]
    one = np.array([1.0], np.float32)
    ce = oracle.scaled_gemm(a, b, one, one)[0]
    A = torch.as_tensor(a).view(torch.float8_e4m3fn).double()
    B = torch.as_tensor(b).view(torch.float8_e4m3fn).double()
    ref = (A @ B.T).numpy()
    assert np.array_equal(ce, ref)
    assert not np.array_equal(-ce, ref)                      # sign flip
    ce_t = oracle.scaled_gemm(b[:, :], a[:8, :], one, one)[0]
    assert not np.array_equal(ce_t, ref[:8, :8])             # swapped operands
