// fp8mm_inst_slow_held.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn224_slow_f8_cg1_ew8() { return &fp8mm_kernel<224, true, false, 1, 8>; }
KernelFn kernel_bn192_slow_f8_cg1_ew8() { return &fp8mm_kernel<192, true, false, 1, 8>; }

}  // namespace fp8mm
