// fp8mm_inst_slow_wide.cu -- explicit instantiation of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn256_slow_f8_cg1_ew8() { return &fp8mm_kernel<256, true, false, 1, 8>; }
KernelFn kernel_bn256_slow_f8_cg1_ew16() { return &fp8mm_kernel<256, true, false, 1, 16>; }

}  // namespace fp8mm
