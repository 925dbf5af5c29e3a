// fp8mm_inst_mx_wide.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn256_fast_mx_cg1_ew8() { return &fp8mm_kernel<256, false, true, 1, 8>; }
KernelFn kernel_bn128_slow_mx_cg1_ew8() { return &fp8mm_kernel<128, true, true, 1, 8>; }

}  // namespace fp8mm
