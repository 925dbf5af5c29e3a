// fp8mm_inst_mx.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn128_fast_mx_cg1_ew8() { return &fp8mm_kernel<128, false, true, 1, 8>; }
KernelFn kernel_bn224_fast_mx_cg1_ew8() { return &fp8mm_kernel<224, false, true, 1, 8>; }

}  // namespace fp8mm
