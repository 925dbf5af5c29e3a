// fp8mm_aux.cu -- the two helper kernels of the GEMM's call path:
//
//  * transpose_to_kmajor: an MN-major operand (stored [L][K][R], R contiguous:
//    the a of a TN/TT product or the b of an NN/TN one, TileOPs "Linear
//    Algebra Operators", GemmFwdOp layout table; BmmFP8FwdOp's b given as
//    [B, K, N]) is copied into K-major scratch [L][R][K] before the GEMM
//    reads it.  The tensor-core MMA reads 8-bit operands K-major here, so the
//    page's own remedy applies: one extra read and write of the operand.
//  * bias_rows: with K = 0 the product is empty and every row of C is the
//    bias (column n holds bias[n]); amax is max |bias| over the stored values.
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8mm_kernels.h"

namespace fp8mm {
namespace {

constexpr int kTile = 128;  // bytes per tile edge

// One 128 x 128-byte tile per iteration (grid-stride over tiles).  Phase 1:
// each warp reads whole input rows as 4-byte words (coalesced) into a padded
// shared tile of words [k][r/4].  Phase 2: each thread takes a 4 x 4 byte
// block (4 rows k, 4 columns r), transposes it in registers with byte
// permutes, and writes 4 output words (4 rows r, bytes k .. k+3).  A warp's
// lanes cover 8 consecutive words of 4 output rows, so its shared-memory reads
// hit 32 distinct banks and its global stores fill whole 32-byte sectors.
__global__ void __launch_bounds__(256) transpose_to_kmajor(const uint8_t* __restrict__ in, uint8_t* __restrict__ out,
                                                           int L, int K, int R) {
  __shared__ uint32_t tile[kTile][kTile / 4 + 1];
  const int tiles_k = (K + kTile - 1) / kTile;
  const int tiles_r = (R + kTile - 1) / kTile;
  const long long per_l = (long long)tiles_k * tiles_r;
  const long long ntiles = (long long)L * per_l;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int l = (int)(t / per_l);
    const long long rem = t - (long long)l * per_l;
    const int k0 = (int)(rem / tiles_r) * kTile;
    const int r0 = (int)(rem % tiles_r) * kTile;
    const uint8_t* src = in + (size_t)l * K * R;
    uint8_t* dst = out + (size_t)l * R * K;
    uint32_t v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int k = k0 + warp + 8 * i;
      const int r = r0 + 4 * lane;
      v[i] = (k < K && r < R) ? __ldg(reinterpret_cast<const uint32_t*>(src + (size_t)k * R + r)) : 0u;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) tile[warp + 8 * i][lane] = v[i];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int task = warp * 4 + i;                       // 32 tasks of 32 blocks each
      const int j = (task & 3) * 8 + (lane & 7);           // output word: bytes k0 + 4j .. +3
      const int rb = (task >> 2) * 4 + (lane >> 3);        // output rows r0 + 4rb .. +3
      const uint32_t w0 = tile[4 * j][rb], w1 = tile[4 * j + 1][rb];
      const uint32_t w2 = tile[4 * j + 2][rb], w3 = tile[4 * j + 3][rb];
      const uint32_t lo01 = __byte_perm(w0, w1, 0x5140), lo23 = __byte_perm(w2, w3, 0x5140);
      const uint32_t hi01 = __byte_perm(w0, w1, 0x7362), hi23 = __byte_perm(w2, w3, 0x7362);
      const uint32_t o[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                             __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
      const int k = k0 + 4 * j;
      const int r = r0 + 4 * rb;
      if (k < K) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (r + q < R) *reinterpret_cast<uint32_t*>(dst + (size_t)(r + q) * K + k) = o[q];
      }
    }
    __syncthreads();
  }
}

// C[l][m][n] = bias[n] (NaN canonical), amax = max |stored value|.
__global__ void __launch_bounds__(256) bias_rows(const void* __restrict__ bias, void* __restrict__ c, long long rows,
                                                 int N, int es, int bf16, unsigned* amax_bits) {
  const long long total = rows * N;
  uint32_t mx = 0u;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(i % N);
    float f;
    if (es == 4) {
      uint32_t b = __ldg(static_cast<const uint32_t*>(bias) + n);
      if ((b & 0x7FFFFFFFu) > 0x7F800000u) b = 0x7FFFFFFFu;
      static_cast<uint32_t*>(c)[i] = b;
      f = __uint_as_float(b);
    } else {
      unsigned short h = __ldg(static_cast<const unsigned short*>(bias) + n);
      const bool nan = bf16 ? ((h & 0x7FFFu) > 0x7F80u) : ((h & 0x7FFFu) > 0x7C00u);
      if (nan) h = 0x7FFF;
      static_cast<unsigned short*>(c)[i] = h;
      f = bf16 ? __uint_as_float((uint32_t)h << 16) : __half2float(__ushort_as_half(h));
    }
    const uint32_t a = __float_as_uint(fabsf(f));
    mx = max(mx, (a > 0x7F800000u) ? 0x7FFFFFFFu : a);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if ((threadIdx.x & 31) == 0 && mx != 0u) atomicMax(amax_bits, mx);
}

}  // namespace

cudaError_t launch_transpose_to_kmajor(const void* in, void* out, int L, int K, int R, int sms, cudaStream_t stream) {
  const long long ntiles = (long long)L * ((K + kTile - 1) / kTile) * ((R + kTile - 1) / kTile);
  if (ntiles == 0) return cudaSuccess;
  const int grid = (int)(ntiles < (long long)sms * 8 ? ntiles : (long long)sms * 8);
  transpose_to_kmajor<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(in), static_cast<uint8_t*>(out), L, K, R);
  return cudaGetLastError();
}

cudaError_t launch_bias_rows(const void* bias, void* c, long long rows, int N, int es, int bf16, unsigned* amax_bits,
                             int sms, cudaStream_t stream) {
  const long long total = rows * N;
  if (total == 0) return cudaSuccess;
  const long long blocks = (total + 255) / 256;
  const int grid = (int)(blocks < (long long)sms * 8 ? blocks : (long long)sms * 8);
  bias_rows<<<grid, 256, 0, stream>>>(bias, c, rows, N, es, bf16, amax_bits);
  return cudaGetLastError();
}

}  // namespace fp8mm
