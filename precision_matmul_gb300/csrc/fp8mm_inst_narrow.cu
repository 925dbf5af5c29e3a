// fp8mm_inst_narrow.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn16_fast_f8_cg1_ew8() { return &fp8mm_kernel<16, false, false, 1, 8>; }
KernelFn kernel_bn32_fast_f8_cg1_ew8() { return &fp8mm_kernel<32, false, false, 1, 8>; }
KernelFn kernel_bn64_fast_f8_cg1_ew8() { return &fp8mm_kernel<64, false, false, 1, 8>; }
KernelFn kernel_bn16_slow_f8_cg1_ew8() { return &fp8mm_kernel<16, true, false, 1, 8>; }
KernelFn kernel_bn32_slow_f8_cg1_ew8() { return &fp8mm_kernel<32, true, false, 1, 8>; }
KernelFn kernel_bn64_slow_f8_cg1_ew8() { return &fp8mm_kernel<64, true, false, 1, 8>; }

}  // namespace fp8mm
