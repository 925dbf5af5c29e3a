// fp8mm_inst_f4.cu -- explicit instantiations (FP4, and the MX CTA-pair tile) of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn128_fast_f4_cg1_ew8() { return &fp8mm_kernel<128, false, true, 1, 8, true>; }
KernelFn kernel_bn256_fast_f4_cg1_ew8() { return &fp8mm_kernel<256, false, true, 1, 8, true>; }
KernelFn kernel_bn256_fast_mx_cg2_ew8() { return &fp8mm_kernel<256, false, true, 2, 8>; }

}  // namespace fp8mm
