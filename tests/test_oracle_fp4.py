"""Pins for the oracle's FP4 block-scaled forms (a row the scope table marks next).

cuDNN "GEMM + Amax (SM100)": A and B may be packed FP4 (float4_e2m1fn_x2, two
values per byte, K-major); their scale factors come per sf_vec_size = 32 (UE8M0)
or 16 (float8_e4m3fn) elements along K, in the same 512-byte atoms as the MX
form; C = sum_k A_hat B_hat.  Independent routes:
- the E2M1 value table from the format's definition (bias 1, one mantissa bit);
- torch's own bf16 -> float4_e2m1fn_x2 conversion and its blocked scale
  layout routine, for the packing order and the factor placement;
- torch's float64 matmul on dequantised values (exact: E2M1 values are
  multiples of 1/2 up to 6 and the factors are powers of two or E4M3 values).
"""
import numpy as np
import pytest
import torch

import library_refs
import oracle

E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table():
    got = oracle.decode(oracle.FMT_E2M1, np.arange(16, dtype=np.uint8))
    assert list(got[:8]) == E2M1_VALUES
    assert list(got[8:]) == [-v for v in E2M1_VALUES]
    assert np.signbit(got[8])                                 # code 8 is -0


def test_packing_order_matches_torch():
    to_fp4 = library_refs.get("_bfloat16_to_float4_e2m1fn_x2")
    g = torch.Generator().manual_seed(71)
    vals = torch.tensor(E2M1_VALUES + [-v for v in E2M1_VALUES])
    x = vals[torch.randint(0, 16, (6, 64), generator=g)]
    packed = to_fp4(x.to(torch.bfloat16)).view(torch.uint8).numpy()
    assert packed.shape == (6, 32)
    back = oracle.decode(oracle.FMT_E2M1, oracle.unpack_fp4(packed))
    assert np.array_equal(back, x.double().numpy())


def _factors(to_blocked, g, L, R, K, vec, codes):
    """Per-(row, factor) codes -> (atoms as placed by torch, per-element scale)."""
    nf = (K + vec - 1) // vec
    pick = codes[torch.randint(0, len(codes), (L, R, nf), generator=g)]
    phys = torch.cat([to_blocked(pick[l]) for l in range(L)]).to(torch.uint8)
    if vec == 32:
        per = torch.exp2(pick.double() - 127)
    else:
        per = pick.to(torch.uint8).view(torch.float8_e4m3fn).double()
    return phys.numpy(), per.repeat_interleave(vec, dim=2)[:, :, :K]


@pytest.mark.parametrize("vec,mode", [(32, oracle.SCALE_MX32_UE8M0), (16, oracle.SCALE_NV16_E4M3)])
def test_fp4_gemm_against_dequantised_matmul(vec, mode):
    to_fp4 = library_refs.get("_bfloat16_to_float4_e2m1fn_x2")
    to_blocked = library_refs.get("to_blocked")
    g = torch.Generator().manual_seed(72 + vec)
    L, M, N, K = 2, 136, 72, 320          # ragged rows; K spans 2.5 (sf 32) or 5 (sf 16) atoms
    vals = torch.tensor(E2M1_VALUES + [-v for v in E2M1_VALUES])
    xa = vals[torch.randint(0, 16, (L, M, K), generator=g)]
    xb = vals[torch.randint(0, 16, (L, N, K), generator=g)]
    pa = to_fp4(xa.to(torch.bfloat16)).view(torch.uint8).numpy()
    pb = to_fp4(xb.to(torch.bfloat16)).view(torch.uint8).numpy()
    if vec == 32:
        codes = torch.arange(121, 134)                     # UE8M0 2^-6 .. 2^6
    else:
        codes = torch.arange(0x20, 0x58)                   # positive E4M3 factors 0.125 .. 15
    sfa, ea = _factors(to_blocked, g, L, M, K, vec, codes)
    sfb, eb = _factors(to_blocked, g, L, N, K, vec, codes)
    ce, _, ab = oracle.scaled_gemm(pa, pb, sfa, sfb, a_fmt=oracle.FMT_E2M1, b_fmt=oracle.FMT_E2M1,
                                   scale_mode=mode)
    Ah, Bh = xa.double() * ea, xb.double() * eb
    ref = torch.bmm(Ah, Bh.transpose(1, 2)).numpy()
    refab = torch.bmm(Ah.abs(), Bh.abs().transpose(1, 2)).numpy()
    assert ce.shape == (L, M, N)
    assert np.array_equal(ce, ref)                          # every product and partial sum is exact
    assert np.array_equal(ab, refab)
    # the other row order inside an atom gives another result
    MB, KB = (M + 127) // 128, (K + 4 * vec - 1) // (4 * vec)
    swapped = sfa.reshape(L, MB, KB, 32, 4, 4).transpose(0, 1, 2, 4, 3, 5).copy().reshape(-1)
    ce_s = oracle.scaled_gemm(pa, pb, swapped, sfb, a_fmt=oracle.FMT_E2M1, b_fmt=oracle.FMT_E2M1,
                              scale_mode=mode)[0]
    assert not np.array_equal(ce_s, ref)


def test_fp4_operands_go_in_pairs():
    a = np.zeros((4, 8), np.uint8)
    sf = np.full(512, 127, np.uint8)
    with pytest.raises(ValueError):
        oracle.scaled_gemm(a, np.zeros((4, 16), np.uint8), sf, sf, a_fmt=oracle.FMT_E2M1,
                           b_fmt=oracle.FMT_E4M3, scale_mode=oracle.SCALE_MX32_UE8M0)
