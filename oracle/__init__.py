"""CPU oracle for the FP8 scaled matrix multiply with a fused global amax.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product package
``precision_matmul_gb300`` never imports it, and this package never imports the
product: the two share no code.

The arithmetic lives in ``fp8_oracle.c`` (plain C, float64).  This module only
builds it with gcc and marshals numpy arrays through ctypes.

Definition evaluated (see the C file for the per-step citations)::

    C[l,m,n] = round_out( sum_c S_A(l,m,c) S_B(l,n,c) sum_{k in c} dec(A[l,m,k]) dec(B[l,n,k]) )
    Amax     = max |C|

Sources: mmaemu "API reference (v0.1)" (mmaemu.scaled_mm, including FP8
outputs and scale_result); TileOPs "Linear Algebra Operators" (GemmFP8FwdOp
scale forms and bias); cuDNN "GEMM + Amax (SM100)" (Shapes, Equations, Dtypes,
the physical scale-factor atom layout, FP4 operands).

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py``.  The reading of the MX scale-factor row order inside
one 128-row atom (row = i32 + 32*i4) is pinned against torch's own layout
routine for the same hardware factors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FMT_E4M3, FMT_E5M2, FMT_E2M1 = 0, 1, 2
OUT_F32, OUT_BF16, OUT_F16, OUT_E4M3, OUT_E5M2 = 0, 1, 2, 3, 4
SCALE_TENSOR, SCALE_A1x128_B1x128, SCALE_A1x128_B128x128, SCALE_MX32_UE8M0, SCALE_NV16_E4M3 = 0, 1, 2, 3, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile fp8_oracle.c into oracle/_build/liboracle.so with gcc.

    Plain ISO C with contraction off, so that no multiply-add is fused and the
    float64 evaluation order is exactly the source order on every host.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        d, u8, i64, i32, vp = (ctypes.c_double, ctypes.c_uint8, ctypes.c_int64, ctypes.c_int,
                              ctypes.c_void_p)
        for name in ("oracle_decode_e4m3", "oracle_decode_e5m2", "oracle_decode_e2m1", "oracle_decode_ue8m0"):
            getattr(lib, name).argtypes = [u8]
            getattr(lib, name).restype = d
        lib.oracle_decode.argtypes = [i32, u8]
        lib.oracle_decode.restype = d
        for name in ("oracle_round_f32", "oracle_round_bf16", "oracle_round_f16"):
            getattr(lib, name).argtypes = [d]
            getattr(lib, name).restype = d
        lib.oracle_round_out.argtypes = [i32, d]
        lib.oracle_round_out.restype = d
        lib.oracle_encode_e4m3_sat.argtypes = [d]
        lib.oracle_encode_e4m3_sat.restype = u8
        lib.oracle_encode_e5m2_sat.argtypes = [d]
        lib.oracle_encode_e5m2_sat.restype = u8
        lib.oracle_scaled_gemm.argtypes = [i64, i64, i64, i64,
                                           vp, i64, i64, i64, i32,
                                           vp, i64, i64, i64, i32,
                                           i32, vp, vp, i32,
                                           d, vp, vp, vp, vp, i64, i64, i32]
        lib.oracle_scaled_gemm.restype = i32
        lib.oracle_amax.argtypes = [vp, i64]
        lib.oracle_amax.restype = d
        _lib = lib
        return lib


def decode(fmt: int, codes) -> np.ndarray:
    """float64 values of FP8 codes (E4M3 or E5M2) or of FP4 codes (E2M1, one
    per byte in the low four bits), decoded bit by bit."""
    lib = _load()
    fn = {FMT_E5M2: lib.oracle_decode_e5m2, FMT_E2M1: lib.oracle_decode_e2m1}.get(fmt, lib.oracle_decode_e4m3)
    codes = np.asarray(codes, dtype=np.uint8)
    return np.array([fn(int(c)) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)


def decode_ue8m0(codes) -> np.ndarray:
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_decode_ue8m0(int(c)) for c in codes.ravel()],
                    dtype=np.float64).reshape(codes.shape)


def encode_sat(fmt: int, values) -> np.ndarray:
    """FP8 codes of float64 values: round to nearest even, saturate, NaN -> 0x7F."""
    lib = _load()
    fn = lib.oracle_encode_e5m2_sat if fmt == FMT_E5M2 else lib.oracle_encode_e4m3_sat
    values = np.asarray(values, dtype=np.float64)
    return np.array([fn(float(v)) for v in values.ravel()], dtype=np.uint8).reshape(values.shape)


def round_out(out_dtype: int, values) -> np.ndarray:
    """Round float64 values once, to nearest even, onto fp32/bf16/fp16 (Inf
    past the largest finite value) or onto E4M3/E5M2 (saturating)."""
    lib = _load()
    values = np.asarray(values, dtype=np.float64)
    return np.array([lib.oracle_round_out(out_dtype, float(v)) for v in values.ravel()],
                    dtype=np.float64).reshape(values.shape)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    """One E2M1 code per byte from packed FP4 operands (float4_e2m1fn_x2: two
    values per byte along the contiguous dimension).  Reading: element 2i sits
    in the low four bits of byte i and element 2i + 1 in the high four bits."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = packed & 0x0F
    out[..., 1::2] = packed >> 4
    return out


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def scaled_gemm(A: np.ndarray, B: np.ndarray, scale_a: np.ndarray, scale_b: np.ndarray, *,
                a_fmt: int = FMT_E4M3, b_fmt: int = FMT_E4M3, scale_mode: int = SCALE_TENSOR,
                out_dtype: int = OUT_F32, scale_result: float | None = None,
                bias: np.ndarray | None = None,
                rows: tuple[int, int] | None = None, nthreads: int | None = None):
    """Evaluate the definition on uint8 code arrays.

    A is [L][M][K] (or [M][K]) and B is [L][N][K] (or [N][K]) uint8 arrays of any
    element strides (numpy views such as ``x.T`` are honoured, which is how the
    layout-equivalence pin feeds NN/TN/TT operands).  Scales: float32 arrays for
    the per-tensor and block modes, uint8 UE8M0 atoms for the MX mode.

    FP4 operands (``a_fmt = b_fmt = FMT_E2M1``) are given packed, [L][M][K/2]
    and [L][N][K/2] bytes (``unpack_fp4``); they go with the block-scaled forms
    SCALE_MX32_UE8M0 (UE8M0 per 32 along K) or SCALE_NV16_E4M3 (E4M3 factor
    codes per 16 along K), both in the atom layout.

    Returns ``(C_exact, C_out, absum)``, float64 arrays of shape [L][rows][N]
    (batch dim dropped when the inputs had none): the unrounded value, the value
    rounded once to ``out_dtype``, and sum_k |a_hat b_hat| for the error bound.
    For the FP8 outputs (OUT_E4M3, OUT_E5M2) ``C_out`` is the FP8 value of
    ``scale_result * C_exact`` (scale_result, an fp32 number, defaults to 1);
    for the others scale_result is ignored.  ``bias`` ([N] values of the
    output type, as float64) is added to every row before the rounding and is
    included in ``C_exact`` (not defined for FP8 outputs).
    """
    lib = _load()
    squeeze = A.ndim == 2
    if squeeze:
        A = A[None]
        B = B[None]
    assert A.dtype == np.uint8 and B.dtype == np.uint8
    if (a_fmt == FMT_E2M1) != (b_fmt == FMT_E2M1):
        raise ValueError("FP4 operands go in pairs (A and B of the same dtype)")
    if a_fmt == FMT_E2M1:
        A, B = unpack_fp4(A), unpack_fp4(B)
    L, M, K = A.shape
    Lb, N, Kb = B.shape
    if Lb != L or Kb != K:
        raise ValueError("A and B disagree on L or K")
    m0, m1 = rows if rows is not None else (0, M)
    sa = np.ascontiguousarray(scale_a)
    sb = np.ascontiguousarray(scale_b)
    if scale_mode in (SCALE_MX32_UE8M0, SCALE_NV16_E4M3):
        assert sa.dtype == np.uint8 and sb.dtype == np.uint8
    else:
        assert sa.dtype == np.float32 and sb.dtype == np.float32
    shape = (L, m1 - m0, N)
    C_exact = np.empty(shape, np.float64)
    C_out = np.empty(shape, np.float64)
    absum = np.empty(shape, np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    sr = 1.0 if scale_result is None else float(np.float32(scale_result))
    bias_arr = None
    if bias is not None:
        bias_arr = np.ascontiguousarray(bias, dtype=np.float64).reshape(-1)
        if bias_arr.size != N:
            raise ValueError("bias must hold N values")
    rc = lib.oracle_scaled_gemm(L, M, N, K,
                                _ptr(A), A.strides[0], A.strides[1], A.strides[2], a_fmt,
                                _ptr(B), B.strides[0], B.strides[1], B.strides[2], b_fmt,
                                scale_mode, _ptr(sa), _ptr(sb), out_dtype, sr, _ptr(bias_arr),
                                _ptr(C_exact), _ptr(C_out), _ptr(absum), m0, m1, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_scaled_gemm rejected its arguments")
    if squeeze:
        return C_exact[0], C_out[0], absum[0]
    return C_exact, C_out, absum


def amax(C: np.ndarray) -> float:
    """max |C| with |-0| = +0, NaN if any element is NaN, +0 for an empty C."""
    lib = _load()
    C = np.ascontiguousarray(C, dtype=np.float64)
    return lib.oracle_amax(_ptr(C), C.size)


def amax_before_quantization(C_exact: np.ndarray) -> float:
    """Amax for an FP8 output: max |C| of the result before scale_result and
    the FP8 rounding, as an fp32 number (reading: the amax that sets the next
    quantisation scale is taken on the unquantised result)."""
    return float(round_out(OUT_F32, [amax(C_exact)])[0])
