"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Sizes here finish in seconds on the oracle yet span several tiles with ragged
edges in M, N and K; the full workload sizes are in test_gpu_full.py.
Bound: |C_gpu - C_exact| <= K 2^-23 sum|a_hat b_hat| + half an ulp of out_dtype
(see tests/parity.py); amax bit-equal to max |C| of the GPU's own C.
"""
import numpy as np
import pytest
import torch

import precision_matmul_gb300 as pm
from precision_matmul_gb300 import synth

from parity import amax_bits_of, check, run_gpu, to_device

pytestmark = pytest.mark.gpu


def _run_check(p, **kw):
    c, amax, plan = run_gpu(p, **kw)
    torch.cuda.synchronize()
    assert pm.fp8mm_device_error(0) == 0
    check(p, c, amax)
    return c, amax, plan


def test_tiny_per_tensor_fp32():
    # 256^3, E4M3, scales 0.5 / 2.0, fast accumulation, fp32 out
    _run_check(synth.tiny_per_tensor())


@pytest.mark.parametrize("out", [synth.OUT_BF16, synth.OUT_F16, synth.OUT_F32])
@pytest.mark.parametrize("fast", [True, False])
def test_per_tensor_ragged(out, fast):
    p = synth.llm_per_tensor(M=300, N=264, K=528, seed=11, fast_accum=fast, out_dtype=out)
    if out == synth.OUT_F16:
        # keep the fp16 range: scales 2^-4 .. 1
        p.scale_a.fill_(0.0625)
        p.scale_b.fill_(0.5)
    _run_check(p)


@pytest.mark.parametrize("block_n", [16, 32, 64, 128, 256])
def test_per_tensor_every_tile_width(block_n):
    p = synth.llm_per_tensor(M=260, N=520, K=384, seed=12, fast_accum=True)
    _run_check(p, block_n=block_n, swap_ab=2)


@pytest.mark.parametrize("fmts", [(0, 1), (1, 0), (1, 1)])
def test_e5m2_operand_pairs(fmts):
    g = torch.Generator().manual_seed(13)
    M, N, K = 200, 136, 256
    a = synth.cast_fp8(torch.randn(1, M, K, generator=g) * 300, fmts[0])
    b = synth.cast_fp8(torch.randn(1, N, K, generator=g) * 300, fmts[1])
    one = torch.tensor([0.25], dtype=torch.float32)
    p = synth.Problem("pairs", 1, M, N, K, a, b, one, one.clone(), fmts[0], fmts[1], synth.SCALE_TENSOR,
                      synth.OUT_F32, True)
    _run_check(p)


@pytest.mark.parametrize("mode", [synth.SCALE_A1x128_B128x128, synth.SCALE_A1x128_B1x128])
def test_blockwise_ragged(mode):
    p = synth.blockwise(M=272, N=392, K=640, seed=14, b_block=128 if mode == synth.SCALE_A1x128_B128x128 else 1)
    _run_check(p)


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
def test_mx_batched(fmt):
    p = synth.mx_batched(L=2, M=256, N=384, K=512, fmt=fmt, seed=15)
    _run_check(p)


def test_mx_ragged():
    p = synth.mx_batched(L=3, M=200, N=136, K=320, seed=16)
    _run_check(p)


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
def test_mx_wide_tiles(fmt):
    # 256-column tiles: two factor atoms per stage, one TMEM accumulator
    p = synth.mx_batched(L=2, M=264, N=520, K=384, fmt=fmt, seed=27)
    c, amax, plan = _run_check(p, block_n=256)
    assert plan.info()["block_n"] == 256


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
def test_mx_224_tiles_every_atom_shift(fmt):
    # 224-column tiles start at 0, 96, 64 and 32 rows into a 128-row factor
    # atom (columns 0, 224, 448, 672); the kernel rebuilds Y's atoms per tile
    p = synth.mx_batched(L=2, M=264, N=904, K=384, fmt=fmt, seed=36)
    c, amax, plan = _run_check(p, block_n=224)
    assert plan.info()["block_n"] == 224


@pytest.mark.parametrize("M", [16, 40, 64, 120])
@pytest.mark.parametrize("data", ["gauss40", "adversarial"])
@pytest.mark.parametrize("fast", [True, False])
def test_skinny_swap_ab_split_k(M, data, fast):
    p = synth.skinny(M=M, N=1536, K=2048, data=data, seed=17, fast_accum=fast)
    c, amax, plan = _run_check(p)
    info = plan.info()
    assert info["swap_ab"] == 1


@pytest.mark.parametrize("fast", [True, False])
def test_skinny_200_rows_unswapped(fast):
    # 129..256 rows run unswapped (pair tiles when fast, 256-column tiles when slow)
    p = synth.skinny(M=200, N=1536, K=2048, data="gauss40", seed=30, fast_accum=fast)
    c, amax, plan = _run_check(p)
    assert plan.info()["swap_ab"] == 0


@pytest.mark.parametrize("splitk", [2, 3, 5])
def test_forced_split_k_non_swapped(splitk):
    p = synth.llm_per_tensor(M=384, N=512, K=1280, seed=18, fast_accum=True)
    c, amax, plan = _run_check(p, splitk=splitk, swap_ab=2)
    assert plan.info()["splitk"] == splitk


def test_blockwise_split_k_swapped():
    p = synth.blockwise(M=48, N=512, K=1536, seed=19)
    c, amax, plan = _run_check(p, splitk=3, swap_ab=1)
    assert plan.info()["swap_ab"] == 1 and plan.info()["splitk"] == 3


def test_smoke_gate_cases():
    _run_check(synth.random_codes(16, 8, 64))
    _run_check(synth.adversarial_codes(64, 64, 256))


def test_special_values_nan_inf():
    # E5M2 Inf and NaN codes: Inf * 0 -> NaN, Inf + finite -> Inf; NaN output canonical, amax NaN
    g = torch.Generator().manual_seed(20)
    M, N, K = 130, 40, 64
    a = synth.cast_fp8(torch.randn(1, M, K, generator=g), synth.E5M2)
    b = synth.cast_fp8(torch.randn(1, N, K, generator=g), synth.E5M2)
    a[0, 3, 5] = 0x7C      # +Inf
    a[0, 7, :] = 0         # zeros ...
    a[0, 7, 9] = 0x7C      # ... and +Inf: NaN where B[n, 9] == 0, else +-Inf
    b[0, 2, 9] = 0
    a[0, 11, 1] = 0x7F     # NaN code
    one = torch.tensor([1.0], dtype=torch.float32)
    for out in (synth.OUT_F32, synth.OUT_BF16):
        p = synth.Problem("special", 1, M, N, K, a, b, one, one.clone(), synth.E5M2, synth.E5M2,
                          synth.SCALE_TENSOR, out, True)
        c, amax, _ = _run_check(p)
        assert int(amax.view(torch.int32).item()) == 0x7FFFFFFF


def test_empty_and_zero_k():
    dev = torch.device("cuda:0")
    for (M, N, K) in [(0, 64, 64), (64, 0, 64), (64, 64, 0)]:
        a = torch.zeros(M, K, dtype=torch.uint8, device=dev)
        b = torch.zeros(N, K, dtype=torch.uint8, device=dev)
        s = torch.ones(1, dtype=torch.float32, device=dev)
        c, amax = pm.scaled_mm(a, b, s, s, out_dtype=torch.bfloat16, a_fmt=0, b_fmt=0)
        torch.cuda.synchronize()
        assert c.shape == (M, N)
        if c.numel():
            assert (c.float() == 0).all()
        assert float(amax) == 0.0


def test_deterministic_repeat():
    p = synth.skinny(M=64, N=1024, K=4096, seed=21)
    t = to_device(p)
    c1, a1, _ = run_gpu(p, tensors=t)
    c1 = c1.clone()
    a1 = a1.clone()
    c2, a2, _ = run_gpu(p, tensors=t)
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
    assert torch.equal(a1.view(torch.int32), a2.view(torch.int32))


def test_out_prior_contents_do_not_matter():
    p = synth.llm_per_tensor(M=128, N=256, K=256, seed=22, fast_accum=True)
    a, b, sa, sb = to_device(p)
    out = torch.full((128, 256), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    amax = torch.full((1,), 12345.0, dtype=torch.float32, device="cuda:0")
    c, am = pm.scaled_mm(a[0], b[0], sa, sb, out=out, amax=amax, use_fast_accum=True, a_fmt=0, b_fmt=0)
    torch.cuda.synchronize()
    assert not torch.isnan(c.float()).any()
    assert int(am.view(torch.int32).item()) == amax_bits_of(c)


def test_launch_count_is_one_kernel():
    p = synth.llm_per_tensor(M=256, N=256, K=256, seed=23)
    _, _, plan = run_gpu(p)
    assert plan.kernel_launches() == 1


@pytest.mark.parametrize("fast,block_n", [(True, 256), (True, 224), (True, 192), (True, 128), (False, 128)])
def test_cta_pair_tiles_ragged(fast, block_n):
    # two-SM MMAs: 256-row tiles split over a CTA pair, ragged in M, N and K
    p = synth.llm_per_tensor(M=520, N=392, K=640, seed=24, fast_accum=fast)
    c, amax, plan = _run_check(p, block_n=block_n, cta_pair=1, swap_ab=2)
    assert plan.info()["cta_pair"] == 1


@pytest.mark.parametrize("epi_warps", [8, 16])
@pytest.mark.parametrize("case", ["tensor_bf16", "tensor_f32", "tensor_f16", "block128", "block1", "block128_f32"])
def test_slow_wide_tiles(case, epi_warps):
    # slow accumulation on 256-column tiles: 128 promoted sums per epilogue thread,
    # ragged in M, N (a last tile 8 columns wide) and K
    if case.startswith("tensor"):
        out = {"bf16": synth.OUT_BF16, "f32": synth.OUT_F32, "f16": synth.OUT_F16}[case.split("_")[1]]
        p = synth.llm_per_tensor(M=300, N=520, K=640, seed=28, fast_accum=False, out_dtype=out)
        if out == synth.OUT_F16:
            p.scale_a.fill_(0.0625)
            p.scale_b.fill_(0.5)
    else:
        p = synth.blockwise(M=300, N=520, K=640, seed=29, b_block=1 if case == "block1" else 128,
                            out_dtype=synth.OUT_F32 if case.endswith("f32") else synth.OUT_BF16)
    c, amax, plan = _run_check(p, block_n=256, swap_ab=2, epi_warps=epi_warps)
    info = plan.info()
    assert info["block_n"] == 256 and info["splitk"] == 1 and info["epi_warps"] == epi_warps


def test_cta_pair_blockwise_and_split_k():
    p = synth.blockwise(M=384, N=264, K=1024, seed=25)
    c, amax, plan = _run_check(p, cta_pair=1, splitk=3, swap_ab=2)
    assert plan.info()["cta_pair"] == 1 and plan.info()["splitk"] == 3


def test_cta_pair_matches_single_cta_within_bound():
    p = synth.llm_per_tensor(M=512, N=512, K=1024, seed=26, fast_accum=True)
    t = to_device(p)
    c1, a1, pl1 = run_gpu(p, tensors=t, cta_pair=1, block_n=256)
    c1 = c1.clone()
    c2, a2, pl2 = run_gpu(p, tensors=t, cta_pair=2, block_n=256)
    torch.cuda.synchronize()
    assert pl1.info()["cta_pair"] == 1 and pl2.info()["cta_pair"] == 0
    check(p, c1, a1)
    check(p, c2, a2)


@pytest.mark.parametrize("shape", [(4096, 4096, 4096, 1, 1), (4096, 4096, 4096, 0, 1), (16, 28672, 8192, 1, 1),
                                   (8192, 7168, 2048, 0, 2), (4096, 4096, 4096, 1, 3)])
def test_plan_preview_matches_device_plan(shape):
    # the host-only preview (used by the CPU planner tests) chooses what the device plan chooses
    M, N, K, fast, mode = shape
    L = 4 if mode == 3 else 1
    d = pm.make_desc(M, N, K, L, out_dtype=0 if mode == 3 else 1, fast_accum=fast, scale_mode=mode)
    props = torch.cuda.get_device_properties(0)
    smem = getattr(props, "shared_memory_per_block_optin", 232448)
    pre = pm._binding.fp8mm_plan_preview(d, props.multi_processor_count, smem)
    got = pm.Plan(d).info()
    keys = ("swap_ab", "block_n", "splitk", "stages", "units", "slow", "smem_bytes", "cta_pair", "epi_warps")
    assert {k: pre[k] for k in keys} == {k: got[k] for k in keys}



@pytest.mark.parametrize("fast", [True, False])
@pytest.mark.parametrize("L,M,N,K", [(2, 256, 384, 512), (3, 200, 264, 400)])
def test_per_tensor_batched(L, M, N, K, fast):
    # a batch of per-tensor GEMMs: the batch stride of the tensor maps and of the scheduler's units
    p = synth.llm_per_tensor(L=L, M=M, N=N, K=K, seed=40 + L, fast_accum=fast)
    _run_check(p)


@pytest.mark.parametrize("mode", [synth.SCALE_A1x128_B128x128, synth.SCALE_A1x128_B1x128])
@pytest.mark.parametrize("L,M,N,K", [(2, 272, 392, 640), (3, 136, 520, 384)])
def test_blockwise_batched(L, M, N, K, mode):
    # per-batch block scales ([L][..][..]) on ragged shapes
    p = synth.blockwise(L=L, M=M, N=N, K=K, seed=42 + L, b_block=128 if mode == synth.SCALE_A1x128_B128x128 else 1)
    _run_check(p)


@pytest.mark.parametrize("knobs", [dict(swap_ab=1, splitk=2), dict(block_n=256, swap_ab=2),
                                   dict(cta_pair=1, swap_ab=2, block_n=128)])
def test_batched_plan_forms(knobs):
    # swapped, 256-column held and CTA-pair tiles over a batch
    p = synth.llm_per_tensor(L=2, M=72 if knobs.get("swap_ab") == 1 else 264, N=392, K=768, seed=44,
                             fast_accum=knobs.get("block_n") != 256)
    _run_check(p, **knobs)


def test_bmm_fp8_against_oracle():
    # TileOPs BmmFP8FwdOp's convention, d[i] = (a[i] @ b[i]) * s_a * s_b, compared with the oracle
    p = synth.llm_per_tensor(L=3, M=136, N=200, K=256, seed=45, fast_accum=False)
    dev = torch.device("cuda:0")
    a = p.a.to(dev).view(torch.float8_e4m3fn)
    w = p.b.to(dev).view(torch.float8_e4m3fn)                    # [B, N, K]
    sa, sb = p.scale_a.to(dev).reshape(()), p.scale_b.to(dev).reshape(())
    d = pm.bmm_fp8(a, w.transpose(1, 2), sa, sb, use_fast_accum=False)   # b given as [B, K, N]
    torch.cuda.synchronize()
    assert d.shape == (3, 136, 200)
    check(p, d, torch.tensor([0.0]), full_amax=False)


def test_torch_scaled_mm_against_oracle():
    p = synth.llm_per_tensor(M=200, N=264, K=384, seed=46, fast_accum=True, out_dtype=synth.OUT_F32)
    dev = torch.device("cuda:0")
    a = p.a[0].to(dev).view(torch.float8_e4m3fn)
    w = p.b[0].to(dev).view(torch.float8_e4m3fn)
    c = pm.torch_scaled_mm(a, w.t(), p.scale_a.to(dev), p.scale_b.to(dev), out_dtype=torch.float32,
                           use_fast_accum=True)
    torch.cuda.synchronize()
    check(p, c, torch.tensor([0.0]), full_amax=False)


@pytest.mark.parametrize("block_n", [192, 224, 256])
@pytest.mark.parametrize("case", ["tensor_bf16", "tensor_f32", "tensor_f16", "block128", "block1"])
def test_slow_pair_held_tiles(case, block_n):
    # slow accumulation on CTA pairs: 256-row tiles whose 96, 112 or 128 promoted sums
    # per epilogue thread stay in registers; ragged in M (a half-empty second CTA), N and K
    if case == "block128" and block_n != 256:
        pytest.skip("128x128 Y scales need 128-aligned halves (planned as 256)")
    if case.startswith("tensor"):
        out = {"bf16": synth.OUT_BF16, "f32": synth.OUT_F32, "f16": synth.OUT_F16}[case.split("_")[1]]
        p = synth.llm_per_tensor(M=300, N=520, K=640, seed=47, fast_accum=False, out_dtype=out)
        if out == synth.OUT_F16:
            p.scale_a.fill_(0.0625)
            p.scale_b.fill_(0.5)
    else:
        p = synth.blockwise(M=300, N=520, K=640, seed=48, b_block=1 if case == "block1" else 128)
    c, amax, plan = _run_check(p, block_n=block_n, cta_pair=1, swap_ab=2)
    info = plan.info()
    assert (info["block_n"], info["cta_pair"], info["splitk"], info["epi_warps"]) == (block_n, 1, 1, 8)


def test_slow_pair_held_batched_multiwave():
    # more pair tiles than SM pairs, over a batch of two
    p = synth.llm_per_tensor(L=2, M=1280, N=2240, K=512, seed=49, fast_accum=False)
    c, amax, plan = _run_check(p, block_n=224, cta_pair=1)
    assert plan.info()["units"] > 76


@pytest.mark.parametrize("block_n", [192, 224])
@pytest.mark.parametrize("case", ["tensor_bf16", "tensor_f32", "block1"])
def test_slow_held_one_cta_192_224(case, block_n):
    # one-CTA held slow tiles of 192 / 224 columns (96 / 112 promoted sums per
    # epilogue thread); ragged in M, N and K
    if case.startswith("tensor"):
        out = synth.OUT_BF16 if case.endswith("bf16") else synth.OUT_F32
        p = synth.llm_per_tensor(M=300, N=520, K=640, seed=50, fast_accum=False, out_dtype=out)
    else:
        p = synth.blockwise(M=300, N=520, K=640, seed=51, b_block=1)
    c, amax, plan = _run_check(p, block_n=block_n, cta_pair=2, swap_ab=2)
    info = plan.info()
    assert (info["block_n"], info["cta_pair"], info["splitk"]) == (block_n, 0, 1)


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
@pytest.mark.parametrize("out", [synth.OUT_F32, synth.OUT_BF16])
def test_mx_pair_tiles(fmt, out):
    # block-scaled MMAs on CTA pairs: 256 x 256 held tiles; each CTA stages its own
    # rows' factor atom and both of the Y tile's; ragged in M (a half-empty second
    # CTA), N (a last tile past N) and K, over a batch of two
    p = synth.mx_batched(L=2, M=392, N=600, K=416, fmt=fmt, seed=52, out_dtype=out)
    c, amax, plan = _run_check(p, block_n=256, cta_pair=1)
    info = plan.info()
    assert (info["block_n"], info["cta_pair"]) == (256, 1)


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
@pytest.mark.parametrize("out", [synth.OUT_F32, synth.OUT_BF16])
def test_mx_one_cta_held_tiles(fmt, out):
    # the one-CTA MX form (128 x 256 held tiles, one accumulator), now planned only
    # with pairs off; ragged in M, N and K over a batch of two, several tiles per CTA
    p = synth.mx_batched(L=2, M=1288, N=2600, K=416, fmt=fmt, seed=54, out_dtype=out)
    c, amax, plan = _run_check(p, block_n=256, cta_pair=2)
    info = plan.info()
    assert (info["block_n"], info["cta_pair"]) == (256, 0) and info["units"] > 152


def test_mx_pair_tiles_multiwave_with_fp8_output():
    p = synth.mx_batched(L=3, M=1024, N=2304, K=512, seed=53, out_dtype=synth.OUT_E4M3)
    p.scale_a.fill_(127 - 8)
    p.scale_b.fill_(127 - 8)
    c, amax, plan = run_gpu(p, block_n=256, cta_pair=1, scale_result=1.0)
    torch.cuda.synchronize()
    assert pm.fp8mm_device_error(0) == 0
    check(p, c, amax, scale_result=1.0)
    assert plan.info()["cta_pair"] == 1 and plan.info()["units"] > 76
