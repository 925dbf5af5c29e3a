"""GPU parity of packed FP4 operands (cuDNN "GEMM + Amax (SM100)", Dtypes and
Layouts: float4_e2m1fn_x2 A and B, factors per 16 elements as E4M3 (NVFP4) or
per 32 as UE8M0 (MXFP4), in the 512-byte atom layout), through
tcgen05.mma kind::mxf4nvf4 with 4X / 2X scale vectors.  Every output element is
compared with the oracle, which decodes the packed codes and the factors bit
by bit and sums in float64."""
import numpy as np
import pytest
import torch

import precision_matmul_gb300 as pm
from precision_matmul_gb300 import synth

from parity import check, run_gpu

pytestmark = pytest.mark.gpu


def _run_check(p, rows=None, **kw):
    c, amax, plan = run_gpu(p, **kw)
    torch.cuda.synchronize()
    assert pm.fp8mm_device_error(0) == 0
    check(p, c, amax, rows=rows, scale_result=kw.get("scale_result"), bias=kw.get("bias"))
    return c, amax, plan


@pytest.mark.parametrize("form", ["nv16", "mx32"])
@pytest.mark.parametrize("out", [synth.OUT_F32, synth.OUT_BF16])
def test_fp4_ragged(form, out):
    # ragged rows; K = 320: 5 atoms of 64 (NVFP4) or 2.5 of 128 (MXFP4), a half-filled last stage
    p = synth.fp4_batched(L=2, M=200, N=136, K=320, form=form, seed=92, out_dtype=out)
    c, amax, plan = _run_check(p, block_n=128)
    assert plan.info()["block_n"] == 128


@pytest.mark.parametrize("form", ["nv16", "mx32"])
def test_fp4_split_and_swap(form):
    p = synth.fp4_batched(L=1, M=264, N=392, K=1024, form=form, seed=93, out_dtype=synth.OUT_BF16)
    _run_check(p, splitk=2)
    q = synth.fp4_batched(L=1, M=40, N=640, K=768, form=form, seed=94, out_dtype=synth.OUT_F32)
    _, _, plan = _run_check(q, swap_ab=1)
    assert plan.info()["swap_ab"] == 1


def test_fp4_fp8_output_and_bias():
    p = synth.fp4_batched(L=2, M=136, N=208, K=512, form="nv16", seed=95, out_dtype=synth.OUT_E4M3)
    _run_check(p, scale_result=0.25)
    q = synth.fp4_batched(L=1, M=136, N=208, K=512, form="mx32", seed=96, out_dtype=synth.OUT_BF16)
    g = torch.Generator().manual_seed(97)
    _run_check(q, bias=(torch.randn(208, generator=g) * 50).to(torch.bfloat16))


@pytest.mark.parametrize("form", ["nv16", "mx32"])
def test_fp4_batched_4x4096(form):
    p = synth.fp4_batched(form=form, seed=98 if form == "nv16" else 99)
    rows = sorted({0, 1, 127, 128, 2047, 4095} | {int(x) for x in np.linspace(0, 4095, 6)})
    _run_check(p, rows=rows)


@pytest.mark.parametrize("form", ["nv16", "mx32"])
@pytest.mark.parametrize("out", [synth.OUT_F32, synth.OUT_BF16])
def test_fp4_wide_tiles(form, out):
    # 256-column held tiles: X's factor atoms and both 128-row blocks of Y's per
    # stage; the last tile's second row block lies past N and is clamped
    p = synth.fp4_batched(L=2, M=264, N=520, K=576, form=form, seed=100, out_dtype=out)
    c, amax, plan = _run_check(p, block_n=256)
    assert plan.info()["block_n"] == 256
