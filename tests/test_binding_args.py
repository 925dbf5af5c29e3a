"""Host-side argument checks of the torch-facing call (CPU only).

The C ABI sees plain pointers, so ``describe`` is what stands between a
caller's tensors and the kernels' reads: operand formats, one device,
contiguity, and scale tensors that hold exactly the elements their form
reads.  Every argument set the GPU tests pass must be accepted (checked here
on CPU copies of the same seeded problems), and each kind of mistake must be
refused before anything reaches the device.
"""
import pytest
import torch

import precision_matmul_gb300 as pm
from precision_matmul_gb300 import synth

from test_gpu_fuzz import _case


def _describe(p, **kw):
    args = dict(out_dtype=synth.OUT_TORCH[p.out_dtype], a_fmt=p.a_fmt, b_fmt=p.b_fmt, scale_mode=p.scale_mode)
    args.update(kw)
    return pm.describe(p.a, p.b, p.scale_a, p.scale_b, **args)


@pytest.mark.parametrize("i", range(96))
def test_every_fuzz_case_is_accepted(i):
    p, _, _ = _case(i)
    L, M, N, K, fa, fb, mode, oc, shape = _describe(p)
    assert (L, M, N, K, fa, fb, mode) == (p.L, p.M, p.N, p.K, p.a_fmt, p.b_fmt, p.scale_mode)
    assert shape == (p.L, p.M, p.N)


@pytest.mark.parametrize("make", [
    lambda: synth.tiny_per_tensor(M=40, N=24, K=96),
    lambda: synth.llm_per_tensor(M=0, N=64, K=64),
    lambda: synth.llm_per_tensor(M=64, N=64, K=0),
    lambda: synth.blockwise(M=130, N=200, K=300, b_block=128),
    lambda: synth.blockwise(M=130, N=200, K=300, b_block=1),
    lambda: synth.blockwise(M=8, N=16, K=0, b_block=128),
    lambda: synth.mx_batched(L=2, M=200, N=136, K=416, fmt=synth.E5M2),
    lambda: synth.mx_batched(L=1, M=0, N=16, K=64),
    lambda: synth.skinny(M=16, N=256, K=512, data="adversarial"),
    lambda: synth.random_codes(16, 8, 64),
    lambda: synth.adversarial_codes(64, 64, 256),
])
def test_workload_generators_are_accepted_and_inferred(make):
    p = make()
    assert _describe(p)[6] == p.scale_mode
    # with the scale form left to inference (for uint8 factors: MX); at K = 0
    # both block forms read no scales and either reading gives C = 0
    inferred = _describe(p, scale_mode=None)[6]
    if p.K > 0 or p.scale_mode in (synth.SCALE_TENSOR, synth.SCALE_MX32_UE8M0):
        assert inferred == p.scale_mode


def test_unbatched_operands():
    p = synth.llm_per_tensor(M=32, N=48, K=128)
    out = pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b, a_fmt=0, b_fmt=0)
    assert out[:4] == (1, 32, 48, 128) and out[8] == (32, 48)
    # float8 dtypes carry their own format
    a8, b8 = p.a[0].view(torch.float8_e4m3fn), p.b[0].view(torch.float8_e5m2)
    assert pm.describe(a8, b8, p.scale_a, p.scale_b)[4:6] == (pm.FP8MM_E4M3, pm.FP8MM_E5M2)


def _raises(exc, p, **kw):
    with pytest.raises(exc):
        _describe(p, **kw)


def test_short_or_long_block_scales_are_refused():
    p = synth.blockwise(M=130, N=200, K=300, b_block=128)
    for sa, sb in ((p.scale_a[:, :-1], p.scale_b), (p.scale_a, p.scale_b[:, :, :-1]),
                   (p.scale_a, torch.ones(1, 200, 3))):
        q = synth.Problem(p.name, p.L, p.M, p.N, p.K, p.a, p.b, sa.contiguous(), sb.contiguous(), p.a_fmt,
                          p.b_fmt, p.scale_mode, p.out_dtype, p.fast_accum)
        _raises(ValueError, q)


def test_scale_form_and_dtype_must_agree():
    p = synth.llm_per_tensor(M=32, N=48, K=128)
    _raises(ValueError, p, scale_mode=pm.FP8MM_SCALE_A1x128_B1x128)   # one element each is too few
    _raises(ValueError, p, scale_mode=7)
    q = synth.Problem(p.name, 1, 32, 48, 128, p.a, p.b, p.scale_a.half(), p.scale_b, 0, 0, synth.SCALE_TENSOR,
                      p.out_dtype, True)
    _raises(TypeError, q)                                              # fp16 scale
    m = synth.mx_batched(L=1, M=64, N=64, K=128)
    mf = synth.Problem(m.name, 1, 64, 64, 128, m.a, m.b, m.scale_a.float(), m.scale_b.float(), m.a_fmt,
                       m.b_fmt, synth.SCALE_MX32_UE8M0, m.out_dtype, True)
    _raises(TypeError, mf)                                             # MX factors as fp32
    _raises(ValueError, m, b_fmt=synth.E5M2)                           # MX needs one format


def test_operand_formats():
    p = synth.llm_per_tensor(M=32, N=48, K=128)
    with pytest.raises(TypeError):
        pm.describe(p.a, p.b, p.scale_a, p.scale_b)                    # uint8 codes without a format
    with pytest.raises(ValueError):
        pm.describe(p.a.view(torch.float8_e4m3fn), p.b, p.scale_a, p.scale_b, a_fmt=pm.FP8MM_E5M2, b_fmt=0)
    with pytest.raises(ValueError):
        pm.describe(p.a, p.b, p.scale_a, p.scale_b, a_fmt=2, b_fmt=0)
    with pytest.raises(TypeError):
        pm.describe(p.a.float(), p.b, p.scale_a, p.scale_b, a_fmt=0, b_fmt=0)


def test_shapes_layout_and_outputs():
    p = synth.llm_per_tensor(M=32, N=48, K=128)
    kw = dict(a_fmt=0, b_fmt=0)
    with pytest.raises(ValueError):
        pm.describe(p.a[0], p.b, p.scale_a, p.scale_b, **kw)                         # 2-D with 3-D
    with pytest.raises(ValueError):
        pm.describe(p.a[0], p.b[0, :, :64], p.scale_a, p.scale_b, **kw)              # K differs
    # a b stored [K, N] (N innermost) is an N-major operand: accepted, copied K-major by the library
    assert pm.describe(p.a[0], p.b[0].t().contiguous().t(), p.scale_a, p.scale_b, **kw)[:4] == (1, 32, 48, 128)
    assert pm.operand_majors(p.a[0].t().contiguous().t(), p.b[0].t().contiguous().t()) == (1, 1)
    with pytest.raises(ValueError):                                                  # N-major with N % 16
        q = synth.llm_per_tensor(M=32, N=40, K=128)
        pm.describe(q.a[0], q.b[0].t().contiguous().t(), q.scale_a, q.scale_b, **kw)
    with pytest.raises(ValueError):                                                  # neither axis contiguous
        pm.describe(p.a[0], torch.empty(48, 256, dtype=torch.uint8)[:, ::2], p.scale_a, p.scale_b, **kw)
    with pytest.raises(ValueError):                                                  # bias of the wrong dtype
        pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b, bias=torch.zeros(48), **kw)
    with pytest.raises(ValueError):                                                  # no bias with FP8 outputs
        pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b, out_dtype=torch.float8_e4m3fn,
                    bias=torch.zeros(48, dtype=torch.float8_e4m3fn), **kw)
    with pytest.raises(ValueError):
        pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b, scale_result=torch.ones(2), **kw)
    with pytest.raises(ValueError):
        pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b.to("meta"), **kw)           # another device
    with pytest.raises(ValueError):
        pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b, out=torch.empty(48, 32, dtype=torch.bfloat16), **kw)
    with pytest.raises(ValueError):
        pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b, out=torch.empty(32, 48), **kw)  # fp32 for bf16
    with pytest.raises(ValueError):
        pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b, amax=torch.empty(1, dtype=torch.float16), **kw)
    with pytest.raises(TypeError):
        pm.describe(p.a[0], p.b[0], p.scale_a, p.scale_b, out_dtype=torch.int8, **kw)


def test_scaled_mm_refuses_host_tensors():
    p = synth.llm_per_tensor(M=32, N=48, K=128)
    with pytest.raises(ValueError):
        pm.scaled_mm(p.a[0], p.b[0], p.scale_a, p.scale_b, a_fmt=0, b_fmt=0)


def test_plan_keys_of_every_length_agree():
    full = (64, 64, 128, 1, 0, 0, 0, 1, 1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0)
    assert pm.normalize_key(full[:13]) == full      # without pair, epilogue warps or strictness
    assert pm.normalize_key(full[:14]) == full
    assert pm.normalize_key(full[:15]) == full
    assert pm.normalize_key(full) == full
    with pytest.raises(ValueError):
        pm.normalize_key(full[:12])
    with pytest.raises(ValueError):
        pm.normalize_key(full + (0,))


def test_plan_for_builds_one_descriptor_per_key(monkeypatch):
    made = []

    class FakePlan:
        def __init__(self, desc):
            made.append(desc)

    monkeypatch.setattr(pm, "Plan", FakePlan)
    monkeypatch.setattr(pm, "_plans", {})
    p1 = pm.plan_for((64, 80, 128, 2, 1, 0, 0, 2, 1, 3, 2, 64, 0, 2))
    p2 = pm.plan_for((64, 80, 128, 2, 1, 0, 0, 2, 1, 3, 2, 64, 0, 2, 0, 0))
    p3 = pm.plan_for((64, 80, 128, 2, 1, 0, 0, 2, 1, 3, 2, 64, 0, 2, 16, 1))
    assert p1 is p2 and p3 is not p1 and len(made) == 2
    d, e = made
    assert (d.M, d.N, d.K, d.L, d.a_fmt, d.b_fmt, d.scale_mode, d.out_dtype, d.fast_accum) == (64, 80, 128, 2, 1, 0, 0, 2, 1)
    assert (d.splitk, d.swap_ab, d.block_n, d.device, d.cta_pair, d.epi_warps, d.stages, d.strict_torch) == \
        (3, 2, 64, 0, 2, 0, 0, 0)
    assert (e.epi_warps, e.strict_torch) == (16, 1)


def test_a_failed_plan_raises_and_is_not_cached(monkeypatch):
    # Without a GPU the library's device query fails: fp8mm_plan returns
    # FP8MM_ERR_CUDA, the binding raises, and nothing is cached for the key,
    # so a later call plans afresh instead of reusing a broken plan.
    from precision_matmul_gb300 import _binding as B
    from precision_matmul_gb300 import build as cuda_build
    if torch.cuda.is_available():
        pytest.skip("needs a host without a GPU")
    cuda_build.build()
    monkeypatch.setattr(pm, "_plans", {})
    key = (64, 64, 128, 1, 0, 0, 0, 1, 1, 0, 0, 0, 0)
    for _ in range(2):
        with pytest.raises(pm.FP8MMError) as e:
            pm.plan_for(key)
        assert e.value.status == B.FP8MM_ERR_CUDA
        assert pm._plans == {}
