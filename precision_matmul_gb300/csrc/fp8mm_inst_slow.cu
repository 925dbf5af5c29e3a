// fp8mm_inst_slow.cu -- explicit instantiations of the GEMM kernel (compiled in parallel).
#include "fp8mm_kernels.h"

namespace fp8mm {

KernelFn kernel_bn128_slow_f8_cg1_ew8() { return &fp8mm_kernel<128, true, false, 1, 8>; }
KernelFn kernel_bn128_slow_f8_cg1_ew16() { return &fp8mm_kernel<128, true, false, 1, 16>; }

}  // namespace fp8mm
