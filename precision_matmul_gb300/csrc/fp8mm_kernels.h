// fp8mm_kernels.h -- the kernel instantiations this library ships and the
// table that selects one by tile width, accumulation mode, scale form, CTA
// pairing and epilogue warp count.
#pragma once
#include <cuda_runtime.h>

#include "fp8mm_kernel.cuh"

namespace fp8mm {

// Helper kernels (fp8mm_aux.cu): MN-major operand [L][K][R] -> K-major [L][R][K]
// scratch; C rows filled with the bias when K = 0.
cudaError_t launch_transpose_to_kmajor(const void* in, void* out, int L, int K, int R, int sms, cudaStream_t stream);
cudaError_t launch_bias_rows(const void* bias, void* c, long long rows, int N, int es, int bf16, unsigned* amax_bits,
                             int sms, cudaStream_t stream);

KernelFn kernel_bn16_fast_f8_cg1_ew8();
KernelFn kernel_bn32_fast_f8_cg1_ew8();
KernelFn kernel_bn64_fast_f8_cg1_ew8();
KernelFn kernel_bn16_slow_f8_cg1_ew8();
KernelFn kernel_bn32_slow_f8_cg1_ew8();
KernelFn kernel_bn64_slow_f8_cg1_ew8();
KernelFn kernel_bn128_fast_f8_cg1_ew8();
KernelFn kernel_bn192_fast_f8_cg1_ew8();
KernelFn kernel_bn224_fast_f8_cg1_ew8();
KernelFn kernel_bn256_fast_f8_cg1_ew8();
KernelFn kernel_bn256_fast_f8_cg2_ew8();
KernelFn kernel_bn224_fast_f8_cg2_ew8();
KernelFn kernel_bn192_fast_f8_cg2_ew8();
KernelFn kernel_bn128_fast_f8_cg2_ew8();
KernelFn kernel_bn128_slow_f8_cg2_ew8();
KernelFn kernel_bn128_slow_f8_cg1_ew8();
KernelFn kernel_bn128_slow_f8_cg1_ew16();
KernelFn kernel_bn256_slow_f8_cg1_ew8();
KernelFn kernel_bn256_slow_f8_cg1_ew16();
KernelFn kernel_bn256_slow_f8_cg2_ew8();
KernelFn kernel_bn224_slow_f8_cg1_ew8();
KernelFn kernel_bn192_slow_f8_cg1_ew8();
KernelFn kernel_bn224_slow_f8_cg2_ew8();
KernelFn kernel_bn192_slow_f8_cg2_ew8();
KernelFn kernel_bn128_fast_mx_cg1_ew8();
KernelFn kernel_bn224_fast_mx_cg1_ew8();
KernelFn kernel_bn256_fast_mx_cg1_ew8();
KernelFn kernel_bn256_fast_mx_cg2_ew8();
KernelFn kernel_bn128_slow_mx_cg1_ew8();
KernelFn kernel_bn128_fast_f4_cg1_ew8();
KernelFn kernel_bn256_fast_f4_cg1_ew8();

struct KernelEntry {
  int bn, slow, mx, cg, ew, f4;
  KernelFn (*get)();
};

inline const KernelEntry* kernel_table(int* n) {
  static const KernelEntry table[] = {
      {16, 0, 0, 1, 8, 0, &kernel_bn16_fast_f8_cg1_ew8},
      {32, 0, 0, 1, 8, 0, &kernel_bn32_fast_f8_cg1_ew8},
      {64, 0, 0, 1, 8, 0, &kernel_bn64_fast_f8_cg1_ew8},
      {16, 1, 0, 1, 8, 0, &kernel_bn16_slow_f8_cg1_ew8},
      {32, 1, 0, 1, 8, 0, &kernel_bn32_slow_f8_cg1_ew8},
      {64, 1, 0, 1, 8, 0, &kernel_bn64_slow_f8_cg1_ew8},
      {128, 0, 0, 1, 8, 0, &kernel_bn128_fast_f8_cg1_ew8},
      {192, 0, 0, 1, 8, 0, &kernel_bn192_fast_f8_cg1_ew8},
      {224, 0, 0, 1, 8, 0, &kernel_bn224_fast_f8_cg1_ew8},
      {256, 0, 0, 1, 8, 0, &kernel_bn256_fast_f8_cg1_ew8},
      {256, 0, 0, 2, 8, 0, &kernel_bn256_fast_f8_cg2_ew8},
      {224, 0, 0, 2, 8, 0, &kernel_bn224_fast_f8_cg2_ew8},
      {192, 0, 0, 2, 8, 0, &kernel_bn192_fast_f8_cg2_ew8},
      {128, 0, 0, 2, 8, 0, &kernel_bn128_fast_f8_cg2_ew8},
      {128, 1, 0, 2, 8, 0, &kernel_bn128_slow_f8_cg2_ew8},
      {128, 1, 0, 1, 8, 0, &kernel_bn128_slow_f8_cg1_ew8},
      {128, 1, 0, 1, 16, 0, &kernel_bn128_slow_f8_cg1_ew16},
      {256, 1, 0, 1, 8, 0, &kernel_bn256_slow_f8_cg1_ew8},
      {256, 1, 0, 1, 16, 0, &kernel_bn256_slow_f8_cg1_ew16},
      {256, 1, 0, 2, 8, 0, &kernel_bn256_slow_f8_cg2_ew8},
      {224, 1, 0, 1, 8, 0, &kernel_bn224_slow_f8_cg1_ew8},
      {192, 1, 0, 1, 8, 0, &kernel_bn192_slow_f8_cg1_ew8},
      {224, 1, 0, 2, 8, 0, &kernel_bn224_slow_f8_cg2_ew8},
      {192, 1, 0, 2, 8, 0, &kernel_bn192_slow_f8_cg2_ew8},
      {128, 0, 1, 1, 8, 0, &kernel_bn128_fast_mx_cg1_ew8},
      {224, 0, 1, 1, 8, 0, &kernel_bn224_fast_mx_cg1_ew8},
      {256, 0, 1, 1, 8, 0, &kernel_bn256_fast_mx_cg1_ew8},
      {256, 0, 1, 2, 8, 0, &kernel_bn256_fast_mx_cg2_ew8},
      {128, 1, 1, 1, 8, 0, &kernel_bn128_slow_mx_cg1_ew8},
      {128, 0, 1, 1, 8, 1, &kernel_bn128_fast_f4_cg1_ew8},
      {256, 0, 1, 1, 8, 1, &kernel_bn256_fast_f4_cg1_ew8},
  };
  *n = (int)(sizeof(table) / sizeof(table[0]));
  return table;
}

inline KernelFn select_kernel(int bn, bool slow, bool mx, int cg, int ew, bool f4 = false) {
  int n = 0;
  const KernelEntry* t = kernel_table(&n);
  for (int i = 0; i < n; ++i)
    if (t[i].bn == bn && t[i].slow == (int)slow && t[i].mx == (int)mx && t[i].cg == cg && t[i].ew == ew &&
        t[i].f4 == (int)f4)
      return t[i].get();
  return nullptr;
}

}  // namespace fp8mm
