"""Seeded synthetic inputs for the FP8 scaled GEMM workloads.

This module holds the input recipes only -- random draws, clamps and the
float32 -> FP8 cast that torch provides -- and none of the GEMM's arithmetic.
Both the CUDA path's tests and the CPU oracle's tests take their inputs from
here, on the CPU, so that both sides see identical bits.

Every draw comes from ``torch.Generator().manual_seed(seed)`` in the order
A, B, scale_a, scale_b.  The FP8 cast clamps to the format's largest finite
value first and then uses torch's ``.to(float8)`` (torch's cast does not
saturate by itself).

Workload sources: the shapes and value recipes of the mmaemu "Testing mmaemu"
T6 sweep (M in {16, 64, 256, 1024, 2048, 8192}, data sets gauss40 and
adversarial), the smoke-gate cases of mmaemu "Backends" (16x8x64 random codes,
64x64x256 adversarial codes), the TileOPs GemmFP8FwdOp scale forms, and the
cuDNN "GEMM + Amax (SM100)" MX form (sf_vec_size 32, UE8M0 factors, batch L).
"""
from __future__ import annotations

import dataclasses

import torch

E4M3, E5M2, E2M1 = 0, 1, 2
OUT_F32, OUT_BF16, OUT_F16, OUT_E4M3, OUT_E5M2 = 0, 1, 2, 3, 4
SCALE_TENSOR, SCALE_A1x128_B1x128, SCALE_A1x128_B128x128, SCALE_MX32_UE8M0, SCALE_NV16_E4M3 = 0, 1, 2, 3, 4

FMAX = {E4M3: 448.0, E5M2: 57344.0}
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
OUT_TORCH = {OUT_F32: torch.float32, OUT_BF16: torch.bfloat16, OUT_F16: torch.float16,
             OUT_E4M3: torch.float8_e4m3fn, OUT_E5M2: torch.float8_e5m2}
OUT_NAME = {OUT_F32: "f32", OUT_BF16: "bf16", OUT_F16: "f16", OUT_E4M3: "e4m3", OUT_E5M2: "e5m2"}


@dataclasses.dataclass
class Problem:
    """One GEMM call's inputs, on the CPU.

    a: uint8 codes [L][M][K]; b: uint8 codes [L][N][K] (both K-innermost; packed
    FP4 operands hold K/2 bytes per row).
    scale_a / scale_b: float32 (per-tensor: shape [1]; 1x128: [L][rows][ceil(K/128)];
    128x128: [L][ceil(N/128)][ceil(K/128)]) or uint8 UE8M0 atoms for the MX form
    (physical layout [L][ceil(rows/128)][ceil(K/128)][32][4][4]).
    """
    name: str
    L: int
    M: int
    N: int
    K: int
    a: torch.Tensor
    b: torch.Tensor
    scale_a: torch.Tensor
    scale_b: torch.Tensor
    a_fmt: int = E4M3
    b_fmt: int = E4M3
    scale_mode: int = SCALE_TENSOR
    out_dtype: int = OUT_F32
    fast_accum: bool = True

    @property
    def flops(self) -> float:
        return 2.0 * self.L * self.M * self.N * self.K


def cast_fp8(x: torch.Tensor, fmt: int) -> torch.Tensor:
    """Clamp to the format's largest finite value, cast with torch, return the codes."""
    f = FMAX[fmt]
    return x.clamp(-f, f).to(TORCH_FP8[fmt]).view(torch.uint8)


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _log_uniform(g: torch.Generator, shape, lo_exp: float, hi_exp: float) -> torch.Tensor:
    u = torch.rand(shape, generator=g, dtype=torch.float64) * (hi_exp - lo_exp) + lo_exp
    return torch.exp2(u).to(torch.float32)


def _kb(K: int) -> int:
    return (K + 127) // 128


# --------------------------------------------------------------------------
# The five workloads (sizes may be overridden for parity tests).
# --------------------------------------------------------------------------

def tiny_per_tensor(M=256, N=256, K=256, seed=0) -> Problem:
    """N(0,1) codes, E4M3, scale_a 0.5, scale_b 2.0, fast accumulation, fp32 out."""
    g = _gen(seed)
    a = cast_fp8(torch.randn(M, K, generator=g), E4M3)
    b = cast_fp8(torch.randn(N, K, generator=g), E4M3)
    return Problem("tiny_per_tensor", 1, M, N, K, a[None], b[None],
                   torch.tensor([0.5], dtype=torch.float32), torch.tensor([2.0], dtype=torch.float32),
                   E4M3, E4M3, SCALE_TENSOR, OUT_F32, True)


def llm_per_tensor(M=4096, N=4096, K=4096, seed=1, fast_accum=True, out_dtype=OUT_BF16, L=1) -> Problem:
    """N(0,1)*112 codes, E4M3, scales 2^U(-4,4), bf16 out; fast or slow accumulation.
    L > 1 draws a batch of L problems sharing the two per-tensor scales (the
    L = 1 draw is the first slice of the same stream)."""
    g = _gen(seed)
    a = cast_fp8(torch.randn(L, M, K, generator=g) * (448.0 / 4), E4M3)
    b = cast_fp8(torch.randn(L, N, K, generator=g) * (448.0 / 4), E4M3)
    sa = _log_uniform(g, (1,), -4, 4)
    sb = _log_uniform(g, (1,), -4, 4)
    return Problem("llm_per_tensor", L, M, N, K, a, b, sa, sb,
                   E4M3, E4M3, SCALE_TENSOR, out_dtype, fast_accum)


def blockwise(M=8192, N=7168, K=2048, seed=2, b_block=128, out_dtype=OUT_BF16, L=1) -> Problem:
    """U(-448,448) codes; A scales per 1x128, B per 128x128 (or 1x128); 2^U(-8,8); slow.
    L > 1 draws a batch with scales per batch ([L][..][..])."""
    g = _gen(seed)
    a = cast_fp8((torch.rand(L, M, K, generator=g) * 2 - 1) * 448.0, E4M3)
    b = cast_fp8((torch.rand(L, N, K, generator=g) * 2 - 1) * 448.0, E4M3)
    sa = _log_uniform(g, (L, M, _kb(K)), -8, 8)
    if b_block == 128:
        sb = _log_uniform(g, (L, (N + 127) // 128, _kb(K)), -8, 8)
        mode = SCALE_A1x128_B128x128
    else:
        sb = _log_uniform(g, (L, N, _kb(K)), -8, 8)
        mode = SCALE_A1x128_B1x128
    return Problem("blockwise", L, M, N, K, a, b, sa, sb,
                   E4M3, E4M3, mode, out_dtype, False)


def _mx_operand(g: torch.Generator, L: int, R: int, K: int, fmt: int) -> torch.Tensor:
    """Per 32-element block along K: x ~ N(0,1), q = cast(x * fmax / max|x_blk|)."""
    Kp = (K + 31) // 32 * 32
    x = torch.randn(L, R, Kp, generator=g)
    blk = x.view(L, R, Kp // 32, 32)
    mx = blk.abs().amax(dim=-1, keepdim=True).clamp_min(1e-30)
    q = (blk * (FMAX[fmt] / mx)).view(L, R, Kp)[:, :, :K]
    return cast_fp8(q.contiguous(), fmt)


def _mx_factors(g: torch.Generator, L: int, R: int, K: int, lo=-6, hi=6) -> torch.Tensor:
    """UE8M0 codes 127 + U{lo..hi}, physical atom layout [L][R/128][K/128][32][4][4]."""
    shape = (L, (R + 127) // 128, _kb(K), 32, 4, 4)
    return (torch.randint(lo, hi + 1, shape, generator=g) + 127).to(torch.uint8)


# E2M1 (FP4) magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7) and the midpoints between them.
_E2M1_MIDS = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def cast_e2m1(x: torch.Tensor) -> torch.Tensor:
    """float32 -> E2M1 codes (one per element, low four bits): round to nearest,
    ties to the even code, saturate at 6; bit 3 is the sign."""
    mag = x.abs().clamp(max=6.0)
    code = torch.bucketize(mag, _E2M1_MIDS)            # midpoints strictly below mag
    tie = (mag == _E2M1_MIDS[code.clamp(max=6)]) & (code % 2 == 1)
    code = code + tie.to(code.dtype)
    return (code | (torch.signbit(x).to(code.dtype) << 3)).to(torch.uint8)


def pack_fp4(codes: torch.Tensor) -> torch.Tensor:
    """Two E2M1 codes per byte along the last dimension: element 2i in the low
    four bits of byte i, element 2i + 1 in the high four bits."""
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).contiguous()


def fp4_batched(L=4, M=4096, N=4096, K=4096, form="nv16", seed=7, out_dtype=OUT_F32) -> Problem:
    """Block-scaled FP4 batched GEMM (cuDNN "GEMM + Amax (SM100)", float4_e2m1fn_x2
    operands): per block of 16 (NVFP4, positive E4M3 factors 0.25 .. 4) or 32
    (MXFP4, UE8M0 factors 2^-6 .. 2^6) elements along K, x ~ N(0,1),
    q = cast_e2m1(x * 6 / max|x_blk|); a and b packed, [L][rows][K/2]."""
    vec = 16 if form == "nv16" else 32
    g = _gen(seed)

    def operand(R):
        Kp = (K + vec - 1) // vec * vec
        x = torch.randn(L, R, Kp, generator=g)
        blk = x.view(L, R, Kp // vec, vec)
        mx = blk.abs().amax(dim=-1, keepdim=True).clamp_min(1e-30)
        return pack_fp4(cast_e2m1((blk * (6.0 / mx)).view(L, R, Kp)[:, :, :K]))

    def factors(R):
        shape = (L, (R + 127) // 128, (K + 4 * vec - 1) // (4 * vec), 32, 4, 4)
        if vec == 16:
            return torch.randint(0x28, 0x49, shape, generator=g).to(torch.uint8)  # E4M3 0.25 .. 4
        return (torch.randint(-6, 7, shape, generator=g) + 127).to(torch.uint8)

    a, b = operand(M), operand(N)
    sfa, sfb = factors(M), factors(N)
    mode = SCALE_NV16_E4M3 if vec == 16 else SCALE_MX32_UE8M0
    return Problem(f"fp4_{form}", L, M, N, K, a, b, sfa, sfb, E2M1, E2M1, mode, out_dtype, True)


def mx_batched(L=4, M=4096, N=4096, K=4096, fmt=E4M3, seed=3, out_dtype=OUT_F32) -> Problem:
    """MX block-scaled batched GEMM, sf_vec_size 32, UE8M0 factors 2^U{-6..6}, fp32 out."""
    g = _gen(seed)
    a = _mx_operand(g, L, M, K, fmt)
    b = _mx_operand(g, L, N, K, fmt)
    sfa = _mx_factors(g, L, M, K)
    sfb = _mx_factors(g, L, N, K)
    return Problem("mx_batched", L, M, N, K, a, b, sfa, sfb, fmt, fmt, SCALE_MX32_UE8M0,
                   out_dtype, True)


def skinny(M=16, N=28672, K=8192, data="gauss40", seed=4, fast_accum=True,
           out_dtype=OUT_BF16) -> Problem:
    """Skinny per-tensor E4M3 GEMM, bf16 out, scales 1.

    gauss40: N(0,1)*40 cast to E4M3.
    adversarial (a reading of "half of each row +-448, the rest +-2^-9 subnormals
    with alternating signs"): for k < K/2, A = (-1)^k * 448 and
    B = (-1)^(floor(k/2)+n) * 448, so the products cancel in every group of four;
    for k >= K/2, A = B = (-1)^k * 2^-9, so the true result is a small positive
    sum hidden under large partial sums.
    """
    g = _gen(seed)
    if data == "gauss40":
        a = cast_fp8(torch.randn(M, K, generator=g) * 40.0, E4M3)
        b = cast_fp8(torch.randn(N, K, generator=g) * 40.0, E4M3)
    elif data == "adversarial":
        k = torch.arange(K)
        half = K // 2
        big = k < half
        sign_k = 1 - 2 * (k % 2)
        a_row = torch.where(big, sign_k * 448.0, sign_k * 2.0 ** -9).to(torch.float32)
        a = cast_fp8(a_row.expand(M, K).contiguous(), E4M3)
        n = torch.arange(N)[:, None]
        sign_b = 1 - 2 * ((k[None, :] // 2 + n) % 2)
        b_val = torch.where(big[None, :], sign_b * 448.0, (sign_k * 2.0 ** -9)[None, :].expand(N, K))
        b = cast_fp8(b_val.to(torch.float32), E4M3)
    else:
        raise ValueError(data)
    one = torch.tensor([1.0], dtype=torch.float32)
    return Problem(f"skinny_{data}", 1, M, N, K, a[None], b[None], one, one.clone(),
                   E4M3, E4M3, SCALE_TENSOR, out_dtype, fast_accum)


# --------------------------------------------------------------------------
# Smoke-gate style cases (mmaemu "Backends", Gates and the verdict cache).
# --------------------------------------------------------------------------

def random_codes(M=16, N=8, K=64, seed=5, fmt=E4M3) -> Problem:
    """Uniformly random finite codes (NaN codes excluded)."""
    g = _gen(seed)

    def draw(R):
        c = torch.randint(0, 256, (R, K), generator=g, dtype=torch.int64)
        if fmt == E4M3:
            c = torch.where((c & 0x7F) == 0x7F, c & 0xF0, c)
        else:
            c = torch.where((c & 0x7C) == 0x7C, c & 0xB3, c)
        return c.to(torch.uint8)

    one = torch.tensor([1.0], dtype=torch.float32)
    return Problem("random_codes", 1, M, N, K, draw(M)[None], draw(N)[None], one, one.clone(),
                   fmt, fmt, SCALE_TENSOR, OUT_F32, True)


def adversarial_codes(M=64, N=64, K=256, seed=6) -> Problem:
    """E4M3 rows built from the smoke gate's adversarial ingredients.

    Row kinds (by row index mod 6): 0 every finite code in turn; 1 subnormals
    and +-0; 2 +-448 with in-block cancellation (x, -x pairs); 3 one exponent
    per 16-element block, random mantissas and signs; 4 -0 everywhere except a
    single 448; 5 random finite codes with -0 on every other position.
    """
    g = _gen(seed)
    finite = torch.tensor([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=torch.int64)

    def rows(R, offset):
        out = torch.empty(R, K, dtype=torch.int64)
        for r in range(R):
            kind = (r + offset) % 6
            k = torch.arange(K)
            if kind == 0:
                out[r] = finite[(k + 7 * r) % finite.numel()]
            elif kind == 1:
                m = torch.randint(0, 8, (K,), generator=g)
                s = torch.randint(0, 2, (K,), generator=g) << 7
                out[r] = m | s
            elif kind == 2:
                s = ((k // 2 + r) % 2) << 7
                out[r] = torch.where(k % 2 == 0, 0x7E | s, 0x7E | (s ^ 0x80))
            elif kind == 3:
                e = torch.randint(1, 16, (K // 16 + 1,), generator=g).repeat_interleave(16)[:K]
                m = torch.randint(0, 8, (K,), generator=g)
                m = torch.where(e == 15, m.clamp(max=6), m)
                s = torch.randint(0, 2, (K,), generator=g) << 7
                out[r] = s | (e << 3) | m
            elif kind == 4:
                out[r] = torch.full((K,), 0x80)
                out[r, (r * 13) % K] = 0x7E
            else:
                c = finite[torch.randint(0, finite.numel(), (K,), generator=g)]
                out[r] = torch.where(k % 2 == 1, torch.full_like(c, 0x80), c)
        return out.to(torch.uint8)

    one = torch.tensor([1.0], dtype=torch.float32)
    return Problem("adversarial_codes", 1, M, N, K, rows(M, 0)[None], rows(N, 3)[None], one,
                   one.clone(), E4M3, E4M3, SCALE_TENSOR, OUT_F32, True)
