"""The FP4 input recipe (precision_matmul_gb300/synth.py) against torch's own
float -> float4_e2m1fn_x2 conversion: rounding, ties, saturation, sign and
the packing order of two elements per byte (CPU only)."""
import numpy as np
import torch

import library_refs
import oracle
from precision_matmul_gb300 import synth


def test_cast_and_pack_match_torch():
    to_fp4 = library_refs.get("_bfloat16_to_float4_e2m1fn_x2")
    g = torch.Generator().manual_seed(90)
    grid = torch.tensor([0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0, 7.0])
    x = torch.cat([grid, -grid, torch.randn(4000, generator=g) * 3]).to(torch.bfloat16).float()
    x = x[: x.numel() // 2 * 2].reshape(1, -1)
    ours = synth.pack_fp4(synth.cast_e2m1(x))
    ref = to_fp4(x.to(torch.bfloat16)).view(torch.uint8)
    assert torch.equal(ours, ref.reshape(ours.shape))


def test_fp4_problem_shapes_and_values():
    for form in ("nv16", "mx32"):
        p = synth.fp4_batched(L=2, M=130, N=72, K=320, form=form, seed=91)
        assert p.a.shape == (2, 130, 160) and p.b.shape == (2, 72, 160)
        vec = 16 if form == "nv16" else 32
        assert p.scale_a.shape == (2, 2, (320 + 4 * vec - 1) // (4 * vec), 32, 4, 4)
        vals = oracle.decode(oracle.FMT_E2M1, oracle.unpack_fp4(p.a.numpy()))
        assert np.abs(vals).max() == 6.0           # each block is scaled to its largest magnitude
