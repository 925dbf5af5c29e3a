"""CPU checks of the C ABI: the library builds and loads, exports every symbol
include/fp8mm.h declares, and rejects invalid descriptions before touching
CUDA (so these run on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

from precision_matmul_gb300 import _binding as B
from precision_matmul_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return B.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fp8mm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8mm_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_structs_match_the_header_layout(tmp_path):
    # compile the header with gcc and compare every field offset with ctypes
    import subprocess
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "fp8mm.h"', 'int main(void) {']
    for cname, cls in (("fp8mm_desc", B.fp8mm_desc), ("fp8mm_plan_info", B.fp8mm_plan_info)):
        lines.append(f'printf("%zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("%zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = []
    for cls in (B.fp8mm_desc, B.fp8mm_plan_info):
        want.append(ctypes.sizeof(cls))
        want += [getattr(cls, f).offset for f, _ in cls._fields_]
    assert got == want


def test_plain_c_caller_links_and_plans(lib, tmp_path):
    # a C program against the header alone: link with the library, plan the
    # 4096^3 slow GEMM for a 152-SM device on the host, print the choices
    import subprocess
    src = tmp_path / "caller.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "fp8mm.h"
int main(void) {
  fp8mm_desc d;
  memset(&d, 0, sizeof d);
  d.M = d.N = d.K = 4096; d.L = 1;
  d.out_dtype = FP8MM_OUT_BF16; d.fast_accum = 0;
  fp8mm_plan_info i;
  fp8mm_status st = fp8mm_plan_preview(&d, 152, 232448, &i);
  printf("%s %d %d %d %d\n", fp8mm_status_string(st), i.block_n, i.cta_pair, i.splitk, i.slow);
  d.K = 24;  /* K rows must be 16-byte multiples */
  printf("%s\n", fp8mm_status_string(fp8mm_plan_preview(&d, 152, 232448, &i)));
  return st == FP8MM_OK ? 0 : 1;
}
""")
    exe = tmp_path / "caller"
    libdir = os.path.dirname(cuda_build.LIB)
    subprocess.run(["gcc", "-I" + os.path.join(ROOT, "include"), str(src), "-L" + libdir, "-lfp8mm",
                    "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[0].split()[1:] == ["256", "1", "1", "1"]  # held 256 x 256 pair tiles
    assert "ALIGN" in out[1].upper()


def test_status_strings(lib):
    for code in range(8):
        assert B.fp8mm_status_string(code)
    assert B.fp8mm_status_string(99) == "unknown status"


def _plan_status(**kw):
    d = B.make_desc(**kw)
    h = ctypes.c_void_p()
    st = B.load().fp8mm_plan(ctypes.byref(d), ctypes.byref(h))
    if h.value:
        B.load().fp8mm_destroy(h)
    return st


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1, N=16, K=16), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=16, a_fmt=3), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=64, a_fmt=2, scale_mode=3), B.FP8MM_ERR_UNSUPPORTED),          # FP4 x FP8
    (dict(M=16, N=16, K=64, a_fmt=2, b_fmt=2, scale_mode=0), B.FP8MM_ERR_UNSUPPORTED),  # FP4 needs factors
    (dict(M=16, N=16, K=32, a_fmt=2, b_fmt=2, scale_mode=4), B.FP8MM_ERR_ALIGNMENT),    # K % 64
    (dict(M=16, N=16, K=64, a_fmt=2, b_fmt=2, scale_mode=4, fast_accum=0), B.FP8MM_ERR_UNSUPPORTED),
    (dict(M=16, N=16, K=64, a_fmt=2, b_fmt=2, scale_mode=4, block_n=224), B.FP8MM_ERR_UNSUPPORTED),
    (dict(M=16, N=16, K=64, a_fmt=2, b_fmt=2, scale_mode=4), B.FP8MM_OK),
    (dict(M=16, N=16, K=64, a_fmt=2, b_fmt=2, scale_mode=3), B.FP8MM_OK),
    (dict(M=16, N=16, K=16, out_dtype=5), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=16, bias=2), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=16, a_major=2), B.FP8MM_ERR_INVALID),
    (dict(M=8, N=16, K=16, a_major=1), B.FP8MM_ERR_ALIGNMENT),   # [K][M] rows of 8 bytes
    (dict(M=16, N=24, K=16, b_major=1), B.FP8MM_ERR_ALIGNMENT),  # [K][N] rows of 24 bytes
    (dict(M=16, N=8, K=16, out_dtype=3), B.FP8MM_ERR_ALIGNMENT),  # FP8 C rows of 8 bytes
    (dict(M=16, N=16, K=16, out_dtype=3, bias=1), B.FP8MM_ERR_UNSUPPORTED),  # no bias for FP8 outputs
    (dict(M=16, N=16, K=16, out_dtype=4, strict_torch=1), B.FP8MM_ERR_REJECTED),  # E4M3 x E4M3 -> E5M2
    (dict(M=16, N=16, K=16, out_dtype=4), B.FP8MM_OK),
    (dict(M=16, N=16, K=16, out_dtype=3, a_major=1, b_major=1, bias=0), B.FP8MM_OK),
    (dict(M=16, N=16, K=16, scale_mode=5), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=16, scale_mode=4), B.FP8MM_ERR_UNSUPPORTED),   # per-16 factors with FP8 operands
    (dict(M=16, N=16, K=16, fast_accum=2), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=16, block_n=40), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=16, epi_warps=12), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=16, swap_ab=3), B.FP8MM_ERR_INVALID),
    (dict(M=16, N=16, K=24), B.FP8MM_ERR_ALIGNMENT),          # K rows not 16-byte multiples
    (dict(M=16, N=12, K=16), B.FP8MM_ERR_ALIGNMENT),          # bf16 C rows of 24 bytes
    (dict(M=16, N=4, K=16, out_dtype=0), B.FP8MM_OK),         # fp32 rows of 16 bytes pass validation
    (dict(M=16, N=16, K=16, scale_mode=3, a_fmt=0, b_fmt=1), B.FP8MM_ERR_UNSUPPORTED),
    (dict(M=2 ** 31, N=16, K=16), B.FP8MM_ERR_UNSUPPORTED),
])
def test_plan_validation_before_cuda(lib, kw, status):
    st = _plan_status(**kw)
    if status == B.FP8MM_OK:
        # valid descriptions reach the device query, which fails without a GPU
        assert st in (B.FP8MM_OK, B.FP8MM_ERR_CUDA)
    else:
        assert st == status


def test_stage_count_range(lib):
    for bad in (1, 13, -1):
        d = B.make_desc(16, 16, 16, stages=bad)
        h = ctypes.c_void_p()
        assert B.load().fp8mm_plan(ctypes.byref(d), ctypes.byref(h)) == B.FP8MM_ERR_INVALID


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert B.load().fp8mm_plan(None, ctypes.byref(h)) == B.FP8MM_ERR_INVALID
    assert B.load().fp8mm_run(None, None, None, None, None, None, None, None, 0, None) == B.FP8MM_ERR_INVALID
    n = ctypes.c_size_t()
    assert B.load().fp8mm_workspace_size(None, ctypes.byref(n)) == B.FP8MM_ERR_INVALID


def test_product_path_has_no_oracle_dependency():
    # the package must never import the oracle (it is test infrastructure)
    pkg = os.path.join(ROOT, "precision_matmul_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fp8_oracle" not in text, f
