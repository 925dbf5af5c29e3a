// fp8mm_inst_pair.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn256_fast_f8_cg2_ew8() { return &fp8mm_kernel<256, false, false, 2, 8>; }
KernelFn kernel_bn224_fast_f8_cg2_ew8() { return &fp8mm_kernel<224, false, false, 2, 8>; }
KernelFn kernel_bn192_fast_f8_cg2_ew8() { return &fp8mm_kernel<192, false, false, 2, 8>; }
KernelFn kernel_bn128_fast_f8_cg2_ew8() { return &fp8mm_kernel<128, false, false, 2, 8>; }
KernelFn kernel_bn128_slow_f8_cg2_ew8() { return &fp8mm_kernel<128, true, false, 2, 8>; }

}  // namespace fp8mm
