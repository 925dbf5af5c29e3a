"""The torch._scaled_mm and batched (BmmFP8FwdOp) calling conventions on the host (CPU only).

``torch_scaled_mm`` only rearranges arguments for ``scaled_mm``: mat2 [K, N]
column-major becomes the [N, K] K-contiguous operand (same storage), the
scales are tensor-wise, bias and scale_result (read for FP8 outputs only) are
passed on, and torch's refusals (E5M2 x E5M2, E4M3 x E4M3 -> E5M2) are
requested from the planner.  ``bmm_fp8`` passes b as a [B, N, K] view
whatever its axis order; the library copies an N-innermost b into K-major
workspace.  The device call is replaced here by a recorder.
"""
import pytest
import torch

import precision_matmul_gb300 as pm


@pytest.fixture
def calls(monkeypatch):
    seen = []

    def fake(a, b, sa, sb, **kw):
        seen.append((a, b, sa, sb, kw))
        return "C", "amax"

    monkeypatch.setattr(pm, "scaled_mm", fake)
    return seen


def _operands(M=32, N=48, K=64, fa=torch.float8_e4m3fn, fb=torch.float8_e4m3fn):
    g = torch.Generator().manual_seed(7)
    a = torch.randn(M, K, generator=g).to(fa)
    w = torch.randn(N, K, generator=g).to(fb)
    s = torch.tensor([0.5])
    return a, w, s, s.clone()


def test_column_major_mat2_becomes_the_k_contiguous_operand(calls):
    a, w, sa, sb = _operands()
    out = torch.empty(32, 48, dtype=torch.bfloat16)
    assert pm.torch_scaled_mm(a, w.t(), sa, sb, out_dtype=torch.bfloat16, use_fast_accum=True, out=out) == "C"
    (a2, b2, sa2, sb2, kw), = calls
    assert a2 is a and b2.shape == (48, 64) and b2.is_contiguous() and b2.data_ptr() == w.data_ptr()
    assert sa2.shape == (1,) and sb2.shape == (1,) and sa2.data_ptr() == sa.data_ptr()
    assert kw == dict(out_dtype=torch.bfloat16, use_fast_accum=True, scale_mode=pm.FP8MM_SCALE_TENSOR, out=out,
                      strict_torch=True, bias=None, scale_result=None)


def test_defaults_follow_torch(calls):
    a, w, sa, sb = _operands()
    pm.torch_scaled_mm(a, w.t(), sa, sb)               # out_dtype defaults to input's FP8 dtype
    assert calls[-1][4]["out_dtype"] == torch.float8_e4m3fn and calls[-1][4]["scale_result"] is None
    pm.torch_scaled_mm(a, w.t(), sa, sb, None, torch.tensor([2.0]), torch.float32)  # positional; scale_result ignored
    kw = calls[-1][4]
    assert kw["use_fast_accum"] is False and kw["out_dtype"] == torch.float32 and kw["scale_result"] is None
    pm.torch_scaled_mm(a, w.t(), sa, sb, None, torch.tensor(2.0), torch.float8_e4m3fn)   # read for FP8 outputs
    assert float(calls[-1][4]["scale_result"]) == 2.0 and calls[-1][4]["scale_result"].shape == (1,)
    bias = torch.zeros(48, dtype=torch.bfloat16)
    pm.torch_scaled_mm(a, w.t(), sa, sb, bias=bias, out_dtype=torch.bfloat16)
    assert calls[-1][4]["bias"] is bias


def test_refusals(calls):
    a, w, sa, sb = _operands()
    with pytest.raises(NotImplementedError):
        pm.torch_scaled_mm(a, w.t(), torch.ones(32, 1), torch.ones(1, 48), out_dtype=torch.bfloat16)
    with pytest.raises(ValueError):                    # row-major [K, N]
        pm.torch_scaled_mm(a, w.t().contiguous(), sa, sb, out_dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pm.torch_scaled_mm(a, w[:, :32].t(), sa, sb, out_dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pm.torch_scaled_mm(a[None], w.t(), sa, sb, out_dtype=torch.bfloat16)
    assert not calls


def test_e5m2_pair_is_sent_with_torchs_refusal(calls):
    a, w, sa, sb = _operands(fa=torch.float8_e5m2, fb=torch.float8_e5m2)
    pm.torch_scaled_mm(a, w.t(), sa, sb, out_dtype=torch.bfloat16)
    assert calls[-1][4]["strict_torch"] is True


def test_bmm_b_in_either_axis_order_is_read_in_place(calls):
    g = torch.Generator().manual_seed(8)
    a = torch.randn(3, 16, 64, generator=g).to(torch.float8_e4m3fn)
    w = torch.randn(3, 24, 64, generator=g).to(torch.float8_e4m3fn)     # [B, N, K]
    sa, sb = torch.tensor(0.5), torch.tensor(2.0)                        # 0-dim, as the page states
    pm.bmm_fp8(a, w, sa, sb, trans_b=True)
    pm.bmm_fp8(a, w.transpose(1, 2), sa, sb)                             # [B, K, N] view of the same storage
    for a2, b2, sa2, sb2, kw in calls:
        assert a2 is a and b2.shape == (3, 24, 64) and b2.is_contiguous() and b2.data_ptr() == w.data_ptr()
        assert sa2.shape == (1,) and sb2.shape == (1,) and float(sa2) == 0.5 and float(sb2) == 2.0
        assert kw["scale_mode"] == pm.FP8MM_SCALE_TENSOR and kw["out_dtype"] == torch.bfloat16
        assert kw["use_fast_accum"] is False


def test_bmm_passes_an_n_innermost_b_as_a_transposed_view(calls):
    g = torch.Generator().manual_seed(9)
    a = torch.randn(3, 16, 64, generator=g).to(torch.float8_e4m3fn)
    bkn = torch.randn(3, 64, 32, generator=g).to(torch.float8_e4m3fn)   # [B, K, N] with N innermost
    s = torch.tensor(1.0)
    pm.bmm_fp8(a, bkn, s, s)
    (a2, b2, _, _, _), = calls
    assert b2.shape == (3, 32, 64) and not b2.is_contiguous() and b2.transpose(1, 2).is_contiguous()
    assert pm.operand_majors(a2, b2) == (0, 1)                          # the library copies it K-major


def test_bmm_refuses_bad_shapes(calls):
    g = torch.Generator().manual_seed(9)
    a = torch.randn(3, 16, 64, generator=g).to(torch.float8_e4m3fn)
    bkn = torch.randn(3, 64, 24, generator=g).to(torch.float8_e4m3fn)
    s = torch.tensor(1.0)
    with pytest.raises(ValueError):
        pm.bmm_fp8(a, bkn.transpose(1, 2).contiguous(), s, s)           # [B, N, K] without trans_b: K mismatch
    with pytest.raises(ValueError):
        pm.bmm_fp8(a[:2], bkn.transpose(1, 2).contiguous(), s, s, trans_b=True)
    with pytest.raises(ValueError):
        pm.bmm_fp8(a[0], bkn[0], s, s)
    assert not calls
