// fp8mm_inst_fast256.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn224_fast_f8_cg1_ew8() { return &fp8mm_kernel<224, false, false, 1, 8>; }
KernelFn kernel_bn256_fast_f8_cg1_ew8() { return &fp8mm_kernel<256, false, false, 1, 8>; }

}  // namespace fp8mm
