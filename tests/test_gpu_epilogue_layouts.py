"""GPU parity of the epilogue forms and operand layouts beyond the plain NT GEMM.

- FP8 outputs (mmaemu "API reference (v0.1)", mmaemu.scaled_mm: out_dtype
  float8_e4m3fn / float8_e5m2 with scale_result): C = round_sat(scale_result *
  C), amax taken before scale_result.
- Bias (TileOPs "Linear Algebra Operators", GemmFP8FwdOp): d = (a s_a) @
  (b s_b)^T + bias, bias [N] in out_dtype.
- NN / TN / TT layouts (GemmFwdOp's layout table) and BmmFP8FwdOp's b given as
  [B, K, N]: M/N-major operands are copied K-major by the library first.

Every case is compared with the oracle element by element (tests/parity.py);
the layouts are also compared bit for bit with the NT call on the same values.
"""
import pytest
import torch

import precision_matmul_gb300 as pm
from precision_matmul_gb300 import synth

from parity import check, run_gpu, to_device

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _fp8_problem(out, fast=True, M=300, N=272, K=528, seed=60, L=1):
    # alpha = 2^-12 brings |C| to tens or hundreds: some E4M3 outputs saturate at 448
    p = synth.llm_per_tensor(L=L, M=M, N=N, K=K, seed=seed, fast_accum=fast, out_dtype=out)
    p.scale_a.fill_(2.0 ** -6)
    p.scale_b.fill_(2.0 ** -6)
    return p


def _run_check(p, **kw):
    c, amax, plan = run_gpu(p, **kw)
    torch.cuda.synchronize()
    assert pm.fp8mm_device_error(0) == 0
    check(p, c, amax, scale_result=kw.get("scale_result"), bias=kw.get("bias"))
    return c, amax, plan


# ----------------------------------------------------------------- FP8 outputs

@pytest.mark.parametrize("out,sr", [(synth.OUT_E4M3, 1.0), (synth.OUT_E4M3, 3.0), (synth.OUT_E5M2, 64.0),
                                    (synth.OUT_E5M2, 2.0 ** -3)])
@pytest.mark.parametrize("fast", [True, False])
def test_fp8_out_per_tensor(out, sr, fast):
    _run_check(_fp8_problem(out, fast), scale_result=sr)


@pytest.mark.parametrize("knobs", [dict(block_n=32, swap_ab=2), dict(block_n=128, swap_ab=2, splitk=3),
                                   dict(swap_ab=1, splitk=2), dict(block_n=256, cta_pair=1, swap_ab=2),
                                   dict(block_n=224, cta_pair=1, swap_ab=2)])
def test_fp8_out_plan_forms(knobs):
    # narrow, split, swapped and CTA-pair tiles all store one-byte rows
    p = _fp8_problem(synth.OUT_E4M3, fast=True, M=72 if knobs.get("swap_ab") == 1 else 520, N=400, K=768, seed=61)
    _run_check(p, scale_result=0.5, **knobs)


@pytest.mark.parametrize("block_n", [224, 256])
def test_fp8_out_slow_held_tiles(block_n):
    p = _fp8_problem(synth.OUT_E5M2, fast=False, M=300, N=528, K=640, seed=62)
    _run_check(p, scale_result=16.0, block_n=block_n, cta_pair=1 if block_n == 224 else 2, swap_ab=2)


@pytest.mark.parametrize("tile", [(2, 192), (2, 224), (2, 256), (1, 192), (1, 224), (1, 256)])
@pytest.mark.parametrize("form", ["bf16_bias", "f16", "e4m3"])
def test_held_tiles_several_per_cta(tile, form):
    # Held slow tiles with 1- or 2-byte outputs stage a warp's whole block and
    # store its chunks back to back; with more tiles than SMs (or SM pairs) each
    # CTA reuses that staging for its next tile.  Ragged in M, N and K.
    pair, block_n = tile
    if form == "e4m3":
        p = _fp8_problem(synth.OUT_E4M3, fast=False, M=1000, N=2608, K=400, seed=64, L=2)
        kw = dict(scale_result=0.75)
    else:
        out = synth.OUT_BF16 if form == "bf16_bias" else synth.OUT_F16
        p = synth.llm_per_tensor(L=2, M=1000, N=2608, K=400, seed=65, fast_accum=False, out_dtype=out)
        p.scale_a.fill_(0.0625)
        p.scale_b.fill_(0.5)
        kw = dict(bias=_bias(p, 68)) if form == "bf16_bias" else {}
    c, amax, plan = _run_check(p, block_n=block_n, cta_pair=pair, swap_ab=2, **kw)
    info = plan.info()
    assert (info["block_n"], info["cta_pair"], info["splitk"]) == (block_n, 1 if pair == 1 else 0, 1)
    assert info["units"] > (76 if pair == 1 else 152)


def test_fp8_out_blockwise_and_mx():
    p = synth.blockwise(M=272, N=400, K=640, seed=63, out_dtype=synth.OUT_E4M3)
    p.scale_a.mul_(2.0 ** -16)
    _run_check(p, scale_result=2.0)
    q = synth.mx_batched(L=2, M=256, N=384, K=512, seed=64, out_dtype=synth.OUT_E5M2)
    q.scale_a.fill_(127 - 7)
    q.scale_b.fill_(127 - 7)
    _run_check(q, scale_result=1.0)


def test_fp8_out_saturates_inf_and_keeps_nan():
    g = torch.Generator().manual_seed(65)
    M, N, K = 130, 48, 64
    a = synth.cast_fp8(torch.randn(1, M, K, generator=g), synth.E5M2)
    b = synth.cast_fp8(torch.randn(1, N, K, generator=g), synth.E5M2)
    a[0, 3, 5] = 0x7C      # +Inf: saturates to the largest finite FP8 value
    a[0, 11, 1] = 0x7F     # NaN
    one = torch.tensor([1.0], dtype=torch.float32)
    p = synth.Problem("special", 1, M, N, K, a, b, one, one.clone(), synth.E5M2, synth.E5M2, synth.SCALE_TENSOR,
                      synth.OUT_E4M3, True)
    c, amax, _ = _run_check(p, scale_result=1.0)
    assert int(amax.view(torch.int32).item()) == 0x7FFFFFFF


def test_fp8_out_full_4096():
    p = synth.llm_per_tensor(fast_accum=True, out_dtype=synth.OUT_E4M3)
    p.scale_a.fill_(2.0 ** -8)
    p.scale_b.fill_(2.0 ** -7)
    _run_check(p, scale_result=1.0)


# ------------------------------------------------------------------------ bias

def _bias(p, seed, scale=100.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(p.N, generator=g) * scale).to(synth.OUT_TORCH[p.out_dtype])


@pytest.mark.parametrize("out", [synth.OUT_BF16, synth.OUT_F16, synth.OUT_F32])
@pytest.mark.parametrize("fast", [True, False])
def test_bias_per_tensor(out, fast):
    p = synth.llm_per_tensor(M=300, N=264, K=528, seed=66, fast_accum=fast, out_dtype=out)
    p.scale_a.fill_(0.0625)
    p.scale_b.fill_(0.5)
    _run_check(p, bias=_bias(p, 67))


@pytest.mark.parametrize("knobs", [dict(swap_ab=1, splitk=2), dict(block_n=128, swap_ab=2, splitk=3),
                                   dict(block_n=256, swap_ab=2), dict(block_n=224, cta_pair=1, swap_ab=2)])
def test_bias_plan_forms(knobs):
    # swapped tiles add one bias value per lane; split tiles add it once, after the partial sums
    p = synth.llm_per_tensor(M=72 if knobs.get("swap_ab") == 1 else 520, N=400, K=768, seed=68,
                             fast_accum="block_n" not in knobs or knobs["block_n"] == 128)
    if knobs.get("block_n") in (224, 256):
        p.fast_accum = False
    _run_check(p, bias=_bias(p, 69, 1000.0), **knobs)


def test_bias_blockwise_mx_and_batch():
    p = synth.blockwise(M=272, N=392, K=640, seed=70)
    _run_check(p, bias=_bias(p, 71, 1e6))
    q = synth.mx_batched(L=2, M=200, N=136, K=320, seed=72, out_dtype=synth.OUT_F32)
    _run_check(q, bias=_bias(q, 73))
    r = synth.llm_per_tensor(L=3, M=136, N=200, K=256, seed=74, fast_accum=False)
    _run_check(r, bias=_bias(r, 75))


def test_bias_with_empty_k():
    # K = 0: the product is empty, every row is the bias; amax = max |bias|
    bias = torch.tensor([1.5, -3.0, 0.25, 7.0] * 4, dtype=torch.bfloat16, device=DEV)
    a = torch.zeros(5, 0, dtype=torch.uint8, device=DEV)
    b = torch.zeros(16, 0, dtype=torch.uint8, device=DEV)
    s = torch.ones(1, dtype=torch.float32, device=DEV)
    c, amax = pm.scaled_mm(a, b, s, s, out_dtype=torch.bfloat16, a_fmt=0, b_fmt=0, bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(c, bias.expand(5, 16))
    assert float(amax) == 7.0


# --------------------------------------------------------------------- layouts

def _mn_major(t):
    """The same values as a view whose storage is [.., K, rows] (rows innermost)."""
    return t.transpose(-1, -2).contiguous().transpose(-1, -2)


@pytest.mark.parametrize("layout", ["NN", "TN", "TT"])
@pytest.mark.parametrize("fast", [True, False])
def test_layouts_per_tensor(layout, fast):
    p = synth.llm_per_tensor(L=2, M=304, N=272, K=528, seed=76, fast_accum=fast)
    a, b, sa, sb = to_device(p)
    ref, ref_amax, _ = run_gpu(p, tensors=(a, b, sa, sb))
    ref = ref.clone()
    ta = _mn_major(a) if layout[0] == "T" else a
    tb = _mn_major(b) if layout[1] == "N" else b
    assert pm.operand_majors(ta, tb) == (int(layout[0] == "T"), int(layout[1] == "N"))
    c, amax, _ = _run_check_tensors(p, (ta, tb, sa, sb))
    # the K-major copy is exact, so the result is the NT call's, bit for bit
    assert torch.equal(c.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(amax.view(torch.int32), ref_amax.view(torch.int32))


def _run_check_tensors(p, tensors, **kw):
    c, amax, plan = run_gpu(p, tensors=tensors, **kw)
    torch.cuda.synchronize()
    assert pm.fp8mm_device_error(0) == 0
    check(p, c, amax)
    return c, amax, plan


@pytest.mark.parametrize("kind", ["blockwise", "mx", "skinny_swapped"])
def test_layouts_other_forms(kind):
    if kind == "blockwise":
        p = synth.blockwise(M=272, N=400, K=640, seed=77)
    elif kind == "mx":
        p = synth.mx_batched(L=2, M=208, N=144, K=320, seed=78)
    else:
        p = synth.skinny(M=48, N=1536, K=2048, seed=79)
    a, b, sa, sb = to_device(p)
    _run_check_tensors(p, (_mn_major(a), _mn_major(b), sa, sb))


def test_bmm_fp8_b_as_bkn_against_oracle():
    # BmmFP8FwdOp with b in torch.bmm's [B, K, N] order, N innermost: transposed by the library
    p = synth.llm_per_tensor(L=3, M=136, N=208, K=256, seed=80, fast_accum=False)
    a = p.a.to(DEV).view(torch.float8_e4m3fn)
    b_kn = p.b.transpose(1, 2).contiguous().to(DEV).view(torch.float8_e4m3fn)      # [B, K, N] storage
    d = pm.bmm_fp8(a, b_kn, p.scale_a.to(DEV).reshape(()), p.scale_b.to(DEV).reshape(()))
    torch.cuda.synchronize()
    assert d.shape == (3, 136, 208)
    check(p, d, torch.tensor([0.0]), full_amax=False)
