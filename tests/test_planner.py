"""The planner's choices, computed on the host without CUDA (fp8mm_plan_preview).

These pin the tile shapes, CTA pairing, split-K, swap-AB, epilogue warps and
ring depths that the kernels were measured with, for a GB300 (152 SMs,
227 KiB of opt-in shared memory per block), plus the plan-time refusals.
A GPU test checks that the preview agrees with fp8mm_plan on the device.
"""
import pytest

from precision_matmul_gb300 import _binding as B
from precision_matmul_gb300 import build as cuda_build

SMS, SMEM = 152, 232448


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()  # nvcc cross-compiles without a GPU; the planner runs on the host
    return B.load()


def preview(M, N, K, L=1, sms=SMS, smem=SMEM, **kw):
    return B.fp8mm_plan_preview(B.make_desc(M, N, K, L, **kw), sms, smem)


def status(M, N, K, L=1, **kw):
    try:
        preview(M, N, K, L, **kw)
        return B.FP8MM_OK
    except B.FP8MMError as e:
        return e.status


def test_llm_4096_fast_uses_pair_tiles(lib):
    i = preview(4096, 4096, 4096, out_dtype=1, fast_accum=1)
    assert (i["cta_pair"], i["block_n"], i["splitk"], i["swap_ab"]) == (1, 224, 1, 0)
    assert i["units"] == 16 * 19 and i["stages"] == 6 and i["grid"] == SMS


def test_llm_4096_slow_uses_held_256_column_pair_tiles(lib):
    # held pair tiles of 256 x 256 (4 x 224-column waves cost more: their 112-column parts store
    # in 16-column chunks)
    i = preview(4096, 4096, 4096, out_dtype=1, fast_accum=0)
    assert (i["cta_pair"], i["block_n"], i["splitk"], i["epi_warps"], i["slow"]) == (1, 256, 1, 8, 1)
    assert i["stages"] == 5 and i["units"] == 16 * 16
    # pairs off: one-CTA held tiles of 128 x 256
    j = preview(4096, 4096, 4096, out_dtype=1, fast_accum=0, cta_pair=2)
    assert (j["cta_pair"], j["block_n"], j["units"]) == (0, 256, 32 * 16)
    # on request: 256 x 224 pair tiles, 16 x 19 of them
    k = preview(4096, 4096, 4096, out_dtype=1, fast_accum=0, block_n=224, cta_pair=1)
    assert (k["cta_pair"], k["block_n"], k["units"]) == (1, 224, 16 * 19)


@pytest.mark.parametrize("mode,stages", [(B.FP8MM_SCALE_A1x128_B128x128, 3), (B.FP8MM_SCALE_A1x128_B1x128, 2)])
def test_blockwise_shallow_ring(lib, mode, stages):
    i = preview(8192, 7168, 2048, out_dtype=1, scale_mode=mode, fast_accum=1)  # block scales are always slow
    assert (i["block_n"], i["slow"], i["stages"], i["epi_warps"], i["cta_pair"]) == (256, 1, stages, 8, 1)
    assert i["units"] == 32 * 28  # 256 x 256 pair tiles


def test_mx_batched_held_256(lib):
    # 256 x 256 held tiles on CTA pairs, 5 stages of 34 KiB per SM beside the fp32 output staging
    i = preview(4096, 4096, 4096, 4, scale_mode=B.FP8MM_SCALE_MX32_UE8M0, out_dtype=0, fast_accum=1)
    assert (i["block_n"], i["cta_pair"], i["splitk"], i["stages"]) == (256, 1, 1, 5)
    assert i["units"] == 4 * 16 * 16
    # pairs off: 128 x 256 held tiles on one CTA, 3 stages of 50 KiB
    j = preview(4096, 4096, 4096, 4, scale_mode=B.FP8MM_SCALE_MX32_UE8M0, out_dtype=0, fast_accum=1, cta_pair=2)
    assert (j["block_n"], j["cta_pair"], j["stages"], j["units"]) == (256, 0, 3, 4 * 32 * 16)


@pytest.mark.parametrize("M,fast,swap,bn,splitk,pair", [
    (16, 1, 1, 16, 2, 0), (16, 0, 1, 16, 2, 0), (64, 1, 1, 64, 2, 0),
    (256, 1, 0, 192, 1, 1), (256, 0, 0, 192, 1, 1), (1024, 0, 0, 256, 1, 1), (2048, 0, 0, 256, 1, 1),
    (1024, 1, 0, 256, 1, 1), (2048, 1, 0, 256, 1, 1), (8192, 1, 0, 256, 1, 1), (8192, 0, 0, 256, 1, 1),
])
def test_skinny_sweep(lib, M, fast, swap, bn, splitk, pair):
    i = preview(M, 28672, 8192, out_dtype=1, fast_accum=fast)
    assert (i["swap_ab"], i["block_n"], i["splitk"], i["cta_pair"]) == (swap, bn, splitk, pair)


def test_workspace_free_plans_have_no_split(lib):
    i = preview(256, 256, 256, out_dtype=0, fast_accum=1)
    assert i["splitk"] == 1 and i["units"] >= 1


@pytest.mark.parametrize("kw,st", [
    (dict(block_n=256, fast_accum=0, splitk=2), B.FP8MM_ERR_UNSUPPORTED),           # held tiles are never split
    (dict(block_n=192, scale_mode=B.FP8MM_SCALE_MX32_UE8M0), B.FP8MM_ERR_UNSUPPORTED),  # MX widths 128/224/256
    (dict(block_n=224, scale_mode=B.FP8MM_SCALE_MX32_UE8M0), B.FP8MM_OK),
    (dict(cta_pair=1, scale_mode=B.FP8MM_SCALE_MX32_UE8M0, block_n=128), B.FP8MM_ERR_UNSUPPORTED),  # MX pairs: 256
    (dict(cta_pair=1, scale_mode=B.FP8MM_SCALE_MX32_UE8M0, block_n=256), B.FP8MM_OK),
    (dict(cta_pair=1, scale_mode=B.FP8MM_SCALE_MX32_UE8M0, block_n=256, fast_accum=0), B.FP8MM_ERR_UNSUPPORTED),
    (dict(block_n=256, fast_accum=0, epi_warps=16), B.FP8MM_OK),
    (dict(block_n=224, fast_accum=0, cta_pair=1), B.FP8MM_OK),                       # held slow pair tile
    (dict(block_n=224, fast_accum=0, cta_pair=2), B.FP8MM_OK),                      # 224 held on one CTA
    (dict(block_n=192, fast_accum=0, cta_pair=1), B.FP8MM_OK),                       # 192 held on a pair
    (dict(block_n=192, cta_pair=1, scale_mode=B.FP8MM_SCALE_A1x128_B128x128), B.FP8MM_ERR_UNSUPPORTED),
    (dict(block_n=224, cta_pair=1, scale_mode=B.FP8MM_SCALE_A1x128_B128x128), B.FP8MM_ERR_UNSUPPORTED),
    (dict(block_n=224, cta_pair=1, scale_mode=B.FP8MM_SCALE_A1x128_B1x128), B.FP8MM_OK),
    (dict(block_n=256, fast_accum=0, cta_pair=1, epi_warps=16), B.FP8MM_ERR_UNSUPPORTED),
    (dict(block_n=48), B.FP8MM_ERR_UNSUPPORTED),                                    # not instantiated
    (dict(epi_warps=12), B.FP8MM_ERR_INVALID),
    (dict(stages=13), B.FP8MM_ERR_INVALID),
])
def test_plan_time_refusals(lib, kw, st):
    base = dict(out_dtype=0, fast_accum=1)
    base.update(kw)
    assert status(512, 1024, 1024, **base) == st


def test_small_devices_and_shared_memory(lib):
    i = preview(4096, 4096, 4096, sms=8, out_dtype=1, fast_accum=1)
    assert i["grid"] <= 8
    # less shared memory: fewer stages, same tile
    full = preview(4096, 4096, 4096, out_dtype=1, fast_accum=0)
    small = preview(4096, 4096, 4096, smem=160 * 1024, out_dtype=1, fast_accum=0)
    assert small["block_n"] == full["block_n"] and small["stages"] < full["stages"]
    assert status(4096, 4096, 4096, smem=40 * 1024, out_dtype=1, fast_accum=0) == B.FP8MM_ERR_UNSUPPORTED


def test_preview_rejects_bad_device_description(lib):
    d = B.make_desc(64, 64, 64)
    for sms, smem in ((0, SMEM), (1, SMEM), (SMS, 0)):
        with pytest.raises(B.FP8MMError) as e:
            B.fp8mm_plan_preview(d, sms, smem)
        assert e.value.status == B.FP8MM_ERR_INVALID


@pytest.mark.parametrize("fa,fb,mode,st", [
    (1, 1, B.FP8MM_SCALE_TENSOR, B.FP8MM_ERR_REJECTED),          # torch._scaled_mm refuses E5M2 x E5M2
    (1, 1, B.FP8MM_SCALE_A1x128_B128x128, B.FP8MM_ERR_REJECTED),
    (1, 1, B.FP8MM_SCALE_MX32_UE8M0, B.FP8MM_ERR_REJECTED),
    (0, 1, B.FP8MM_SCALE_TENSOR, B.FP8MM_OK),
    (1, 0, B.FP8MM_SCALE_TENSOR, B.FP8MM_OK),
    (0, 0, B.FP8MM_SCALE_TENSOR, B.FP8MM_OK),
])
def test_strict_torch_refuses_what_torch_refuses(lib, fa, fb, mode, st):
    kw = dict(a_fmt=fa, b_fmt=fb, scale_mode=mode, out_dtype=0, fast_accum=1)
    assert status(512, 1024, 1024, strict_torch=1, **kw) == st
    assert status(512, 1024, 1024, **kw) == B.FP8MM_OK                # the library's own default computes all four


def test_strict_torch_flag_values(lib):
    assert status(512, 1024, 1024, out_dtype=0, strict_torch=2) == B.FP8MM_ERR_INVALID
    assert status(512, 1024, 1024, out_dtype=0, strict_torch=-1) == B.FP8MM_ERR_INVALID


def test_every_fuzz_case_finds_an_accepted_plan(lib):
    # the GPU fuzz redraws plan overrides until the library accepts them; on the host
    # planner (152 SMs, 227 KiB of shared memory) each case must get there quickly
    import test_gpu_fuzz as fz
    for i in range(96):
        p, knobs, r = fz._case(i)
        for tries in range(200):
            d = B.make_desc(p.M, p.N, p.K, p.L, a_fmt=p.a_fmt, b_fmt=p.b_fmt, scale_mode=p.scale_mode,
                            out_dtype=p.out_dtype, fast_accum=1 if p.fast_accum else 0, **knobs)
            try:
                B.fp8mm_plan_preview(d, 152, 232448)
                break
            except B.FP8MMError as e:
                assert e.status == B.FP8MM_ERR_UNSUPPORTED
                knobs = fz._draw_knobs(r)
        else:
            raise AssertionError(f"case {i}: no accepted override set")
