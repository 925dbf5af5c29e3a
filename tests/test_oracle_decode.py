"""Pins for the oracle's FP8 / UE8M0 decode and its saturating encoder.

The decode is checked code by code against torch's own float8 conversions (a
library routine that shares nothing with the oracle's bit-level decode) and
against the facts the pages state (largest finite E4M3 448, 254 finite codes,
canonical NaN byte 0x7F).
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _torch_decode(fmt, codes):
    dt = torch.float8_e5m2 if fmt == oracle.FMT_E5M2 else torch.float8_e4m3fn
    return torch.tensor(codes, dtype=torch.uint8).view(dt).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E5M2])
def test_decode_all_codes_match_torch(fmt):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode(fmt, codes)
    ref = _torch_decode(fmt, list(range(256)))
    for c in range(256):
        if math.isnan(ref[c]):
            assert math.isnan(ours[c]), hex(c)
        else:
            assert ours[c] == ref[c], hex(c)
            assert math.copysign(1.0, ours[c]) == math.copysign(1.0, ref[c]), hex(c)


def test_e4m3_page_facts(facts):
    vals = oracle.decode(oracle.FMT_E4M3, np.arange(256, dtype=np.uint8))
    finite = vals[np.isfinite(vals)]
    assert finite.size == int(facts["e4m3_finite_code_count"])
    assert finite.max() == float(facts["e4m3_max_finite"])
    assert finite.min() == -float(facts["e4m3_max_finite"])
    # no infinities in float8_e4m3fn; the NaN codes are 0x7F and 0xFF
    assert not np.isinf(vals).any()
    assert [c for c in range(256) if math.isnan(vals[c])] == [0x7F, 0xFF]
    assert int(facts["nan_fp8_bits"], 16) == 0x7F


def test_e4m3_closed_forms():
    d = lambda c: float(oracle.decode(oracle.FMT_E4M3, np.uint8(c)))
    assert d(0x01) == 2.0 ** -9          # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert d(0x08) == 2.0 ** -6          # smallest normal
    assert d(0x38) == 1.0                # exponent field 7 = bias
    assert d(0x7E) == 448.0
    assert math.copysign(1.0, d(0x80)) == -1.0 and d(0x80) == 0.0


def test_e5m2_closed_forms():
    d = lambda c: float(oracle.decode(oracle.FMT_E5M2, np.uint8(c)))
    assert d(0x01) == 2.0 ** -16
    assert d(0x04) == 2.0 ** -14
    assert d(0x3C) == 1.0
    assert d(0x7B) == 57344.0
    assert d(0x7C) == math.inf and d(0xFC) == -math.inf
    for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF):
        assert math.isnan(d(c))


def test_ue8m0_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_ue8m0(codes)
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.tensor(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        for c in range(256):
            if math.isnan(ref[c]):
                assert math.isnan(ours[c])
            else:
                assert ours[c] == ref[c], c
    assert ours[127] == 1.0 and ours[0] == 2.0 ** -127 and ours[254] == 2.0 ** 127
    assert math.isnan(ours[255])


def _grid_with_midpoints(fmt):
    vals = oracle.decode(fmt, np.arange(256, dtype=np.uint8))
    pos = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (pos[:-1] + pos[1:]) / 2
    fmax = pos.max()
    extra = np.array([fmax * 1.01, fmax * 2, 1e9, pos[1] / 2, pos[1] / 3, pos[1] * 0.75])
    rng = np.random.default_rng(11)
    rand = rng.uniform(0, fmax * 1.1, 2000).astype(np.float32).astype(np.float64)
    nudge = np.concatenate([np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                            np.nextafter(mids.astype(np.float32), np.float32(0))]).astype(np.float64)
    g = np.concatenate([pos, mids, extra, rand, nudge])
    return np.concatenate([g, -g])


@pytest.mark.parametrize("fmt", [oracle.FMT_E4M3, oracle.FMT_E5M2])
def test_encoder_matches_torch_cast_on_clamped_values(fmt):
    x = _grid_with_midpoints(fmt)
    fmax = 448.0 if fmt == oracle.FMT_E4M3 else 57344.0
    ours = oracle.encode_sat(fmt, x)
    dt = torch.float8_e5m2 if fmt == oracle.FMT_E5M2 else torch.float8_e4m3fn
    # torch rounds float32 -> fp8; feed values that are exact in float32
    x32 = torch.tensor(x, dtype=torch.float64).to(torch.float32)
    exact = x32.to(torch.float64).numpy() == x
    ref = x32.clamp(-fmax, fmax).to(dt).view(torch.uint8).numpy()
    assert exact.sum() > 1000
    assert (ours[exact] == ref[exact]).all(), np.nonzero(ours[exact] != ref[exact])


def test_encoder_nan_and_saturation():
    assert oracle.encode_sat(oracle.FMT_E4M3, [math.nan])[0] == 0x7F
    assert oracle.encode_sat(oracle.FMT_E4M3, [math.inf])[0] == 0x7E
    assert oracle.encode_sat(oracle.FMT_E4M3, [-math.inf])[0] == 0xFE
    assert oracle.encode_sat(oracle.FMT_E5M2, [math.inf])[0] == 0x7B
    # 464 is the midpoint of 448 and the (non-existent) 480: ties to even -> 448
    assert oracle.encode_sat(oracle.FMT_E4M3, [464.0])[0] == 0x7E
    assert oracle.encode_sat(oracle.FMT_E4M3, [-0.0])[0] == 0x80
