// fp8mm_inst_slow_pair.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn256_slow_f8_cg2_ew8() { return &fp8mm_kernel<256, true, false, 2, 8>; }
KernelFn kernel_bn224_slow_f8_cg2_ew8() { return &fp8mm_kernel<224, true, false, 2, 8>; }
KernelFn kernel_bn192_slow_f8_cg2_ew8() { return &fp8mm_kernel<192, true, false, 2, 8>; }

}  // namespace fp8mm
