"""ctypes binding of the C ABI in include/fp8mm.h (argument marshalling only).

Every name here mirrors the C entry point of the same name.  All arithmetic
runs in the CUDA library; if the library has not been built this module
raises instead of computing anything on the host.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfp8mm.so")

FP8MM_E4M3, FP8MM_E5M2, FP8MM_E2M1 = 0, 1, 2
FP8MM_OUT_F32, FP8MM_OUT_BF16, FP8MM_OUT_F16, FP8MM_OUT_E4M3, FP8MM_OUT_E5M2 = 0, 1, 2, 3, 4
(FP8MM_SCALE_TENSOR, FP8MM_SCALE_A1x128_B1x128, FP8MM_SCALE_A1x128_B128x128,
 FP8MM_SCALE_MX32_UE8M0, FP8MM_SCALE_NV16_E4M3) = 0, 1, 2, 3, 4
STATUS = {0: "FP8MM_OK", 1: "FP8MM_ERR_INVALID", 2: "FP8MM_ERR_ALIGNMENT", 3: "FP8MM_ERR_UNSUPPORTED",
          4: "FP8MM_ERR_REJECTED", 5: "FP8MM_ERR_WORKSPACE", 6: "FP8MM_ERR_CUDA", 7: "FP8MM_ERR_DEVICE"}
FP8MM_OK, FP8MM_ERR_INVALID, FP8MM_ERR_ALIGNMENT, FP8MM_ERR_UNSUPPORTED = 0, 1, 2, 3
FP8MM_ERR_REJECTED, FP8MM_ERR_WORKSPACE, FP8MM_ERR_CUDA, FP8MM_ERR_DEVICE = 4, 5, 6, 7

# Every symbol include/fp8mm.h declares.
EXPORTS = ("fp8mm_plan", "fp8mm_workspace_size", "fp8mm_run", "fp8mm_plan_roofline",
           "fp8mm_plan_get_info", "fp8mm_destroy", "fp8mm_status_string", "fp8mm_device_error",
           "fp8mm_plan_kernel_launches", "fp8mm_gemm", "fp8mm_run_static_workspace", "fp8mm_plan_preview",
           "fp8mm_run_ex", "fp8mm_test_withhold_loads")
FP8MM_STATIC_WORKSPACE_BYTES = 16 * 1024 * 1024


class fp8mm_desc(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("L", ctypes.c_int64),
                ("a_fmt", ctypes.c_int32), ("b_fmt", ctypes.c_int32), ("scale_mode", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("fast_accum", ctypes.c_int32), ("splitk", ctypes.c_int32),
                ("swap_ab", ctypes.c_int32), ("block_n", ctypes.c_int32), ("device", ctypes.c_int32),
                ("cta_pair", ctypes.c_int32), ("epi_warps", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("strict_torch", ctypes.c_int32), ("bias", ctypes.c_int32), ("a_major", ctypes.c_int32),
                ("b_major", ctypes.c_int32)]


class fp8mm_plan_info(ctypes.Structure):
    _fields_ = [("swap_ab", ctypes.c_int32), ("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("splitk", ctypes.c_int32), ("stages", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("units", ctypes.c_int64), ("slow", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("cta_pair", ctypes.c_int32), ("epi_warps", ctypes.c_int32)]


class FP8MMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({fp8mm_status_string(status)})")


_lib = None


def load():
    """Load the in-tree CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"the CUDA library {LIB_PATH} is missing: run "
                           "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, szp = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)
    lib.fp8mm_plan.argtypes = [ctypes.POINTER(fp8mm_desc), ctypes.POINTER(vp)]
    lib.fp8mm_plan.restype = i32
    lib.fp8mm_workspace_size.argtypes = [vp, szp]
    lib.fp8mm_workspace_size.restype = i32
    lib.fp8mm_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.fp8mm_run.restype = i32
    lib.fp8mm_plan_roofline.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    lib.fp8mm_plan_roofline.restype = i32
    lib.fp8mm_plan_get_info.argtypes = [vp, ctypes.POINTER(fp8mm_plan_info)]
    lib.fp8mm_plan_get_info.restype = i32
    lib.fp8mm_destroy.argtypes = [vp]
    lib.fp8mm_destroy.restype = None
    lib.fp8mm_status_string.argtypes = [i32]
    lib.fp8mm_status_string.restype = ctypes.c_char_p
    lib.fp8mm_device_error.argtypes = [i32, ctypes.POINTER(ctypes.c_uint32), i32]
    lib.fp8mm_device_error.restype = i32
    lib.fp8mm_plan_kernel_launches.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.fp8mm_plan_kernel_launches.restype = i32
    lib.fp8mm_gemm.argtypes = [ctypes.POINTER(fp8mm_desc), vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.fp8mm_gemm.restype = i32
    lib.fp8mm_run_static_workspace.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.fp8mm_run_static_workspace.restype = i32
    lib.fp8mm_plan_preview.argtypes = [ctypes.POINTER(fp8mm_desc), i32, i32, ctypes.POINTER(fp8mm_plan_info)]
    lib.fp8mm_plan_preview.restype = i32
    lib.fp8mm_run_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.fp8mm_test_withhold_loads.argtypes = [i32]
    lib.fp8mm_test_withhold_loads.restype = i32
    lib.fp8mm_run_ex.restype = i32
    _lib = lib
    return lib


def fp8mm_status_string(status: int) -> str:
    return load().fp8mm_status_string(int(status)).decode()


def _check(st: int, where: str):
    if st != FP8MM_OK:
        raise FP8MMError(st, where)


def make_desc(M, N, K, L=1, *, a_fmt=FP8MM_E4M3, b_fmt=FP8MM_E4M3, scale_mode=FP8MM_SCALE_TENSOR,
              out_dtype=FP8MM_OUT_BF16, fast_accum=1, splitk=0, swap_ab=0, block_n=0, device=0,
              cta_pair=0, epi_warps=0, stages=0, strict_torch=0, bias=0, a_major=0, b_major=0) -> fp8mm_desc:
    d = fp8mm_desc()
    d.M, d.N, d.K, d.L = int(M), int(N), int(K), int(L)
    d.a_fmt, d.b_fmt, d.scale_mode, d.out_dtype = int(a_fmt), int(b_fmt), int(scale_mode), int(out_dtype)
    d.fast_accum, d.splitk, d.swap_ab, d.block_n, d.device = (int(fast_accum), int(splitk), int(swap_ab),
                                                              int(block_n), int(device))
    d.cta_pair = int(cta_pair)
    d.epi_warps = int(epi_warps)
    d.stages = int(stages)
    d.strict_torch = int(strict_torch)
    d.bias, d.a_major, d.b_major = int(bias), int(a_major), int(b_major)
    return d


class Plan:
    """Owns one fp8mm_plan_t handle."""

    def __init__(self, desc: fp8mm_desc):
        self.desc = desc
        self._h = ctypes.c_void_p()
        _check(load().fp8mm_plan(ctypes.byref(desc), ctypes.byref(self._h)), "fp8mm_plan")

    @property
    def handle(self):
        return self._h

    def workspace_size(self) -> int:
        n = ctypes.c_size_t()
        _check(load().fp8mm_workspace_size(self._h, ctypes.byref(n)), "fp8mm_workspace_size")
        return int(n.value)

    def roofline(self) -> tuple[float, float]:
        f, b = ctypes.c_double(), ctypes.c_double()
        _check(load().fp8mm_plan_roofline(self._h, ctypes.byref(f), ctypes.byref(b)), "fp8mm_plan_roofline")
        return f.value, b.value

    def info(self) -> dict:
        i = fp8mm_plan_info()
        _check(load().fp8mm_plan_get_info(self._h, ctypes.byref(i)), "fp8mm_plan_get_info")
        return {k: getattr(i, k) for k, _ in fp8mm_plan_info._fields_}

    def kernel_launches(self) -> int:
        n = ctypes.c_int32()
        _check(load().fp8mm_plan_kernel_launches(self._h, ctypes.byref(n)), "fp8mm_plan_kernel_launches")
        return int(n.value)

    def run(self, a_ptr, b_ptr, sa_ptr, sb_ptr, c_ptr, amax_ptr, ws_ptr, ws_bytes, stream) -> None:
        st = load().fp8mm_run(self._h, a_ptr, b_ptr, sa_ptr, sb_ptr, c_ptr, amax_ptr, ws_ptr,
                              ctypes.c_size_t(int(ws_bytes)), stream)
        _check(st, "fp8mm_run")

    def run_ex(self, a_ptr, b_ptr, sa_ptr, sb_ptr, sr_ptr, bias_ptr, c_ptr, amax_ptr, ws_ptr, ws_bytes,
               stream) -> None:
        st = load().fp8mm_run_ex(self._h, a_ptr, b_ptr, sa_ptr, sb_ptr, sr_ptr, bias_ptr, c_ptr, amax_ptr, ws_ptr,
                                 ctypes.c_size_t(int(ws_bytes)), stream)
        _check(st, "fp8mm_run_ex")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.fp8mm_destroy(h)
            self._h = ctypes.c_void_p()


def fp8mm_plan(desc: fp8mm_desc) -> Plan:
    return Plan(desc)


def fp8mm_run(plan: Plan, a_ptr, b_ptr, sa_ptr, sb_ptr, c_ptr, amax_ptr, ws_ptr=None, ws_bytes=0,
              stream=None) -> None:
    plan.run(a_ptr, b_ptr, sa_ptr, sb_ptr, c_ptr, amax_ptr, ws_ptr, ws_bytes, stream)


def fp8mm_run_ex(plan: Plan, a_ptr, b_ptr, sa_ptr, sb_ptr, sr_ptr, bias_ptr, c_ptr, amax_ptr, ws_ptr=None,
                 ws_bytes=0, stream=None) -> None:
    plan.run_ex(a_ptr, b_ptr, sa_ptr, sb_ptr, sr_ptr, bias_ptr, c_ptr, amax_ptr, ws_ptr, ws_bytes, stream)


def fp8mm_device_error(device: int = 0, clear: bool = True) -> int:
    code = ctypes.c_uint32()
    _check(load().fp8mm_device_error(int(device), ctypes.byref(code), int(bool(clear))), "fp8mm_device_error")
    return int(code.value)


def fp8mm_test_withhold_loads(enable: bool) -> None:
    """Test support: GEMM kernels launched while enabled issue no operand loads,
    so their MMA issuer's wait runs out and the kernel aborts (see the header)."""
    _check(load().fp8mm_test_withhold_loads(1 if enable else 0), "fp8mm_test_withhold_loads")


def fp8mm_gemm(desc: fp8mm_desc, a_ptr, b_ptr, sa_ptr, sb_ptr, c_ptr, amax_ptr, ws_ptr=None, ws_bytes=0,
               stream=None) -> None:
    st = load().fp8mm_gemm(ctypes.byref(desc), a_ptr, b_ptr, sa_ptr, sb_ptr, c_ptr, amax_ptr, ws_ptr,
                           ctypes.c_size_t(int(ws_bytes)), stream)
    _check(st, "fp8mm_gemm")


def fp8mm_run_static_workspace(plan: Plan, a_ptr, b_ptr, sa_ptr, sb_ptr, c_ptr, amax_ptr, stream=None) -> None:
    """fp8mm_run without a caller workspace: split-K scratch comes from the
    library's fixed device array (FP8MM_STATIC_WORKSPACE_BYTES), so this call
    allocates nothing; see include/fp8mm.h for the sharing rules."""
    st = load().fp8mm_run_static_workspace(plan.handle, a_ptr, b_ptr, sa_ptr, sb_ptr, c_ptr, amax_ptr, stream)
    _check(st, "fp8mm_run_static_workspace")


def fp8mm_plan_preview(desc: fp8mm_desc, sms: int, max_smem_bytes: int) -> dict:
    """The planner's choices for a device with `sms` SMs and `max_smem_bytes`
    of opt-in shared memory per block, computed on the host without CUDA."""
    i = fp8mm_plan_info()
    _check(load().fp8mm_plan_preview(ctypes.byref(desc), int(sms), int(max_smem_bytes), ctypes.byref(i)),
           "fp8mm_plan_preview")
    return {k: getattr(i, k) for k, _ in fp8mm_plan_info._fields_}

