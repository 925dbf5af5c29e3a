// fp8mm_inst_fast128.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn128_fast_f8_cg1_ew8() { return &fp8mm_kernel<128, false, false, 1, 8>; }
KernelFn kernel_bn192_fast_f8_cg1_ew8() { return &fp8mm_kernel<192, false, false, 1, 8>; }

}  // namespace fp8mm
