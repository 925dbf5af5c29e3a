// fp8mm_inst_f4.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn128_fast_f4_cg1_ew8() { return &fp8mm_kernel<128, false, true, 1, 8, true>; }
KernelFn kernel_bn256_fast_f4_cg1_ew8() { return &fp8mm_kernel<256, false, true, 1, 8, true>; }

}  // namespace fp8mm
