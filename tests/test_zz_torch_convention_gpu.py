"""torch._scaled_mm's calling convention on the GPU: the same kernels as
``scaled_mm``, so the result is bit-identical, and torch's E5M2 x E5M2
refusal comes back from the planner."""
import pytest
import torch

import precision_matmul_gb300 as pm

pytestmark = pytest.mark.gpu


def _operands(fa, fb, M=200, N=264, K=384):
    g = torch.Generator().manual_seed(31)
    a = (torch.randn(M, K, generator=g) * 20).clamp(-448, 448).to(fa).cuda()
    w = (torch.randn(N, K, generator=g) * 20).clamp(-448, 448).to(fb).cuda()
    return a, w, torch.tensor([0.25], device="cuda"), torch.tensor([0.5], device="cuda")


@pytest.mark.parametrize("fast", [True, False])
def test_same_bits_as_scaled_mm(fast):
    a, w, sa, sb = _operands(torch.float8_e4m3fn, torch.float8_e5m2)
    c = pm.torch_scaled_mm(a, w.t(), sa, sb, out_dtype=torch.bfloat16, use_fast_accum=fast)
    ref, _ = pm.scaled_mm(a, w, sa, sb, out_dtype=torch.bfloat16, use_fast_accum=fast)
    torch.cuda.synchronize()
    assert c.shape == (200, 264)
    assert torch.equal(c.view(torch.int16), ref.view(torch.int16))


def test_e5m2_pair_is_refused_like_torch():
    a, w, sa, sb = _operands(torch.float8_e5m2, torch.float8_e5m2)
    with pytest.raises(pm.FP8MMError) as e:
        pm.torch_scaled_mm(a, w.t(), sa, sb, out_dtype=torch.bfloat16)
    assert e.value.status == pm._binding.FP8MM_ERR_REJECTED
    c, _ = pm.scaled_mm(a, w, sa, sb, out_dtype=torch.bfloat16)  # the library's own call computes it
    torch.cuda.synchronize()
    assert c.shape == (200, 264)


def test_bmm_same_bits_as_scaled_mm():
    g = torch.Generator().manual_seed(32)
    a = (torch.randn(2, 136, 256, generator=g) * 20).clamp(-448, 448).to(torch.float8_e4m3fn).cuda()
    w = (torch.randn(2, 200, 256, generator=g) * 20).clamp(-448, 448).to(torch.float8_e4m3fn).cuda()
    sa, sb = torch.tensor(0.5, device="cuda"), torch.tensor(0.125, device="cuda")
    d = pm.bmm_fp8(a, w.transpose(1, 2), sa, sb)                 # b as torch.bmm's [B, K, N] view
    ref, _ = pm.scaled_mm(a, w, sa.reshape(1), sb.reshape(1), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert d.shape == (2, 136, 200)
    assert torch.equal(d.view(torch.int16), ref.view(torch.int16))
