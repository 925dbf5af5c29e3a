// fp8mm_kernel.cuh -- persistent, warp-specialised FP8 scaled GEMM + amax for
// sm_103a.
//
// What one launch computes (mmaemu "API reference (v0.1)", mmaemu.scaled_mm;
// TileOPs "Linear Algebra Operators", GemmFP8FwdOp; cuDNN "GEMM + Amax
// (SM100)", Equations):
//
//   C[l,m,n] = out( sum_c S_A(l,m,c) S_B(l,n,c) sum_{k in chunk c} A[l,m,k] B[l,n,k] ),
//   amax     = max |C|.
//
// The kernel works in the frame of the tensor-core instruction: X is the
// operand on the MMA's M side (tiles of 128 rows, one TMEM lane per row) and
// Y the operand on its N side (tiles of BN rows).  Normally X = A and Y = B;
// for skinny M the roles swap (X = B, Y = A) and the epilogue stores the
// tile transposed, so that the long dimension fills the 128-row side.
//
// Roles ((EW + 2) warps, or EW + 4 for held tiles; one CTA per SM, or a
// cluster of two CTAs per 256-row tile; persistent over work units):
//   warps 0..EW-1  epilogue (EW = 8 or 16): TMEM -> registers; for slow
//              accumulation and block scales, one promotion per 128-K chunk
//              (acc += s_x s_y chunk in fp32); split-K fix-up; scale, cast,
//              NaN canonicalisation, amax, shared-memory staging, TMA stores.
//   warp EW    TMA producer: A/B tiles (128 B of K per row, 128-byte swizzle)
//              and, for the MX form, the 512-byte scale-factor atoms (for
//              224-column tiles gathered by the whole warp to start at the
//              tile), into a ring of `stages` shared-memory slots guarded by
//              mbarriers.
//   warp EW+1  MMA issuer: tcgen05.mma kind::f8f6f4 (cta_group::1, or
//              cta_group::2 over a CTA pair) or kind::mxf8f6f4 with block
//              scaling, into up to four TMEM accumulators; also owns the TMEM
//              allocation.
//   warps EW+2, EW+3  (held tiles only) idle: they complete the last
//              warpgroup, which hands registers to the epilogue (setmaxnreg).
//
// Every wait on an mbarrier is bounded in time: when a limit is hit the
// kernel records an error code in a device word, the other roles leave their
// loops, in-flight copies and MMAs are drained, TMEM is freed and the kernel
// returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fp8mm {

constexpr int kBlockM = 128;      // MMA M: TMEM lanes per tile
constexpr int kBlockK = 128;      // K per pipeline stage: one 128-byte swizzle row per operand row
constexpr int kUmmaK = 32;        // K per tcgen05.mma for 8-bit operands
// Bound on one wait: 2^31 SM clock cycles, about one second at GB300 clocks.
constexpr uint64_t kWaitLimitCycles = 1ull << 31;

// Block geometry shared by the kernel and the host planner: EW epilogue
// warps, the producer and the MMA issuer, and (for held tiles) two idle warps
// that complete the last warpgroup of the register split below.
__host__ __device__ constexpr int kernel_threads(int ew, bool held) { return (ew + (held ? 4 : 2)) * 32; }
// Held tiles split the register file by warpgroup (setmaxnreg): the
// producer/MMA warpgroup drops to kRegRoles so that the epilogue warps,
// which keep a whole tile row range in registers, rise to epi_regs(ew).
// Launch cap: 12 warps -> 3 per SM sub-partition -> 168; 20 warps -> 5 -> 96.
constexpr int kRegRoles = 64;
__host__ __device__ constexpr int launch_regs(int ew) { return ew == 8 ? 168 : 96; }
__host__ __device__ constexpr int epi_regs(int ew) { return ew == 8 ? 216 : 104; }
// Each sub-partition holds EW/4 epilogue warps and one warp of the last group.
static_assert(2 * epi_regs(8) + kRegRoles <= 512 && 4 * epi_regs(16) + kRegRoles <= 512,
              "register split per SM sub-partition");
static_assert((8 * epi_regs(8) + 4 * kRegRoles) <= 12 * launch_regs(8) &&
                  (16 * epi_regs(16) + 4 * kRegRoles) <= 20 * launch_regs(16),
              "register split within the launch's allocation");
// Slow accumulation on 192-, 224- and 256-column tiles: each epilogue warp
// keeps 96, 112 or 128 (8 warps) or 64 (16 warps, 256 columns) promoted fp32
// sums per row in registers.
__host__ __device__ constexpr bool wide_slow(int bn, bool slow) { return slow && bn > 128; }
// Tiles whose epilogue holds the whole tile in registers before storing it:
// slow 256-column tiles (the promoted sums) and MX 256-column tiles, whose
// single TMEM accumulator is copied out and released at once so that the
// next tile's MMAs overlap the stores.  Such tiles are never split or swapped.
__host__ __device__ constexpr bool held_tile(int bn, bool slow, bool mx) {
  return wide_slow(bn, slow) || (mx && !slow && bn == 256);
}
// Per-warp output staging: two buffers of 32 rows x 64 B (8 epilogue warps)
// or 32 rows x 32 B (16 epilogue warps, or held tiles, whose registers leave
// less room).  (Rows of 16 B measured far slower: the stores then write half
// sectors.)
// Output staging per epilogue warp.  Held tiles with 1- or 2-byte outputs
// stage the warp's whole 32 x hmax block (all its chunks at once, stored
// without waiting between them); the others alternate two chunk buffers
// (held fp32 tiles: two of 32 rows x 16 columns).
__host__ __device__ constexpr int stage_out_bytes(int ew, bool held, int es = 4, int hmax = 0) {
  return held ? (es <= 2 ? 32 * hmax * es : 4096) : (ew == 8 ? 4096 : 2048);
}
// Columns [0, half0_cols) belong to epilogue warps 0-3, the rest to warps 4-7
// (slow 224- and 256-column tiles split evenly: every warp promotes as many
// columns as its neighbour).
__host__ __device__ constexpr int half0_cols(int bn, bool slow = false) {
  return (bn <= 64 || wide_slow(bn, slow)) ? bn / 2 : ((bn / 2 + 31) / 32) * 32;
}
// Widest column range of one epilogue warp.
__host__ __device__ constexpr int part_max_cols(int bn, int ew, bool slow = false) {
  return ew == 8 ? half0_cols(bn, slow) : bn / 4;
}
// Columns of one output chunk (one TMA store of 32 tile rows).  Held tiles
// with 1- or 2-byte outputs take the widest of 64, 32 and 16 columns that
// divides both warps' parts (256-, 192- and 224-column slow tiles); fp32
// outputs 16 (64-byte rows: 16 chunks of 8 waited on the TMA twice as often,
// measured 3-4% slower for MX and FP4 batches).
__host__ __device__ constexpr int chunk_cols(int bn, int es, int ew, bool held, bool slow = false) {
  return held ? (es == 4 ? 16
                         : (part_max_cols(bn, ew, slow) % 64 == 0 && (bn - part_max_cols(bn, ew, slow)) % 64 == 0)
                               ? 64
                               : (part_max_cols(bn, ew, slow) % 32 == 0 && (bn - part_max_cols(bn, ew, slow)) % 32 == 0)
                                     ? 32
                                     : 16)
         : es == 1 ? (32 < part_max_cols(bn, ew) ? 32 : part_max_cols(bn, ew))
                   : (((ew == 8 ? 64 : 32) / es) < part_max_cols(bn, ew) ? ((ew == 8 ? 64 : 32) / es)
                                                                          : part_max_cols(bn, ew));
}
// MX: shared-memory bytes per stage for the factor atoms: X's atom and up to
// three of Y's (a 256-column tile copies whole atoms; a 224-column one has two
// atoms gathered to start at the tile's first row).
constexpr uint32_t kSfStageBytes = 2048;

// Abort codes (OR-ed into the device word).
constexpr unsigned kErrProducer = 1u, kErrMmaFull = 2u, kErrMmaAcc = 4u, kErrEpiAcc = 8u,
                   kErrEpiSync = 16u, kErrDrain = 32u, kErrPlan = 64u;

enum ScaleKind : int { kScaleNone = 0, kScaleRow = 1, kScaleBlock128 = 2 };

struct KParams {
  int R, Q, K, L;         // rows of X (MMA M side), rows of Y (MMA N side), K, batches
  int num_kb;             // ceil(K / 128)
  int kb_per_split;
  int splits;
  int tiles_r, tiles_q;
  int group;              // tile rows per raster group
  long long units;        // L * tiles_r * tiles_q * splits
  int swap;               // 1: C[m][n] is tile(q = m, r = n)
  int withhold_loads;     // abort-path test: the producer issues nothing, so the MMA issuer's wait runs out
  int out_dtype;          // 0 f32, 1 bf16, 2 f16, 3 E4M3, 4 E5M2
  int out_es;             // bytes per output element
  const float* scale_result;  // FP8 outputs: multiplies the result before the FP8 rounding (device), or null
  const void* bias;       // [N] of out_dtype added to every row before the rounding, or null
  int stages;
  int num_acc;            // TMEM accumulators (1, 2 or 4)
  uint32_t tmem_cols;
  uint32_t idesc;         // instruction descriptor without the scale-factor ids
  const float* sa_tensor; // per-tensor scales (device), or null
  const float* sb_tensor;
  const float* x_scale;   // block scales of X and Y (fp32), or null
  int x_kind;
  const float* y_scale;
  int y_kind;
  int scale_kb;           // block scales: ceil(K / 128), the row stride of the scale arrays; factor
                          // atoms: their count along K (ceil(K / 128) for FP8, ceil(K / (4 vec)) for FP4)
  const uint8_t* sfx;     // MX scale-factor atoms of X and Y
  const uint8_t* sfy;
  int f4_vec16;           // FP4 operands: 1 E4M3 factors per 16 elements (4X), 0 UE8M0 per 32 (2X)
  int sfx_mb, sfy_mb;     // ceil(R / 128), ceil(Q / 128)
  float* ws_partials;     // split-K partial tiles [tile][split][col][row]
  unsigned* ws_counters;  // split-K arrivals per tile
  unsigned* amax_bits;    // fp32 amax as its bit pattern (non-negative floats order as uints)
  unsigned* abort_word;   // device word recording aborted waits (read by fp8mm_device_error)
  uint32_t off_x, off_y, off_sf, off_out, off_ys, off_bias, off_bar;  // shared-memory layout
  uint32_t x_stage_bytes, y_stage_bytes, sf_stage_bytes;
  uint32_t out_swz_mask;  // 16-byte-chunk XOR mask of the output staging swizzle
  uint32_t out_rowbytes;  // bytes per staging row
};


struct Unit {
  int l, tr, tq, s, kb0, kb1;
};

__device__ __forceinline__ Unit decode_unit(long long u, const KParams& p) {
  Unit t;
  t.s = (int)(u % p.splits);
  const long long tile = u / p.splits;
  const long long per_l = (long long)p.tiles_r * p.tiles_q;
  t.l = (int)(tile / per_l);
  const long long t2 = tile - (long long)t.l * per_l;
  const long long gspan = (long long)p.group * p.tiles_q;
  const int grp = (int)(t2 / gspan);
  const int first = grp * p.group;
  const int gsize = min(p.group, p.tiles_r - first);
  const int within = (int)(t2 - (long long)grp * gspan);
  t.tr = first + within % gsize;
  t.tq = within / gsize;
  t.kb0 = t.s * p.kb_per_split;
  t.kb1 = min(t.kb0 + p.kb_per_split, p.num_kb);
  return t;
}

// Bounded wait on an mbarrier phase.  Returns false if another role aborted or
// the limit was hit (which sets the abort flag and the device error word).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         unsigned* abort_word, unsigned code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::clock_cycles();
  uint32_t spins = 0;
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((++spins & 15u) == 0) {
      if (*abort_flag) return false;
      if (ptx::clock_cycles() - t0 > kWaitLimitCycles) {
        *abort_flag = 1u;
        atomicOr(abort_word, code);
        return false;
      }
    }
  }
}

// Bounded wait used while tearing down: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned* abort_word) {
  const uint64_t t0 = ptx::clock_cycles();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::clock_cycles() - t0 > kWaitLimitCycles) {
      atomicOr(abort_word, kErrDrain);
      return;
    }
  }
}

template <int N>
__device__ __forceinline__ void tmem_load(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 64) {
    ptx::tmem_ld_32x32b_x32(taddr, reinterpret_cast<uint32_t(&)[32]>(r[0]));
    ptx::tmem_ld_32x32b_x32(taddr + 32, reinterpret_cast<uint32_t(&)[32]>(r[32]));
    ptx::tmem_ld_wait_x32(reinterpret_cast<uint32_t(&)[32]>(r[0]));
    ptx::tmem_ld_wait_x32(reinterpret_cast<uint32_t(&)[32]>(r[32]));
  } else if constexpr (N == 32) {
    ptx::tmem_ld_32x32b_x32(taddr, r);
    ptx::tmem_ld_wait_x32(r);
  } else if constexpr (N == 16) {
    ptx::tmem_ld_32x32b_x16(taddr, r);
    ptx::tmem_ld_wait_x16(r);
  } else {
    static_assert(N == 8, "tcgen05.ld width");
    ptx::tmem_ld_32x32b_x8(taddr, r);
    ptx::tmem_ld_wait_x8(r);
  }
}

__device__ __forceinline__ uint32_t swz(uint32_t off, uint32_t mask) {
  return off ^ (((off >> 7) & mask) << 4);
}


// max that returns NaN if either input is NaN
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two fp32 values to two FP8 codes (lo in the low byte): round to nearest
// even, saturate to the largest finite value (Inf included), NaN stays NaN.
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi, bool e5m2) {
  uint16_t r;
  if (e5m2)
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}
// Bias value of output column n (bias has out_dtype: fp32, bf16 or fp16).
__device__ __forceinline__ float bias_at(const KParams& p, int n) {
  if (p.out_es == 4) return __ldg(static_cast<const float*>(p.bias) + n);
  const unsigned short h = __ldg(static_cast<const unsigned short*>(p.bias) + n);
  return p.out_dtype == 1 ? __uint_as_float((uint32_t)h << 16) : __half2float(__ushort_as_half(h));
}

// Scales CW values of this thread's tile row by alpha (and adds the bias of
// each value's output column), casts them to out_dtype (round to nearest
// even; NaN becomes the canonical pattern; FP8 outputs are multiplied by
// scale_result first and saturate), folds the largest |value| into the
// running amax (inside C only; for bf16/fp16/fp32 the largest stored value:
// rounding is monotone, so it is the rounded largest value; for FP8 outputs
// the fp32 value before scale_result and the rounding), stages the warp's
// 32 x CW block in one of its two shared-memory buffers and stores it with one
// TMA copy at (cx, cy, cl).  xr is the thread's X row (the output column when
// the operands are swapped).  v holds at least CW values (the chunk is its
// first CW); NOSWAP drops the transposed staging of swapped operands.
// With a bias, bias_cols points at the chunk's CW bias values staged in
// shared memory (unswapped tiles; 0 past the last column) and bias_lane holds
// the thread's own column's value (swapped tiles).  STREAM: the caller has
// made the buffer free and commits the bulk group after its last chunk (a
// held tile's chunks go out back to back).
template <int CW, int ES, int NV, bool NOSWAP = false, bool STREAM = false>
__device__ __forceinline__ void store_chunk(const KParams& p, const CUtensorMap* tm_c, float (&v)[NV], float alpha,
                                            float sr, const float* bias_cols, float bias_lane, bool row_ok, int q0,
                                            int lane, uint8_t* stg_gen, uint32_t stg_s, int cx, int cy, int cl,
                                            bool in_bounds, float& amax_f, uint32_t& amax_nan) {
  if (ES != 1 && p.bias != nullptr) {
    // d = (a s_a) @ (b s_b)^T + bias: one fp32 fma, then the one rounding to out_dtype
    if (NOSWAP || !p.swap) {
#pragma unroll
      for (int i = 0; i < CW; ++i) v[i] = fmaf(v[i], alpha, bias_cols[i]);
    } else {
#pragma unroll
      for (int i = 0; i < CW; ++i) v[i] = fmaf(v[i], alpha, bias_lane);
    }
  } else {
#pragma unroll
    for (int i = 0; i < CW; ++i) v[i] *= alpha;
  }
  // largest |value| of the chunk inside C (NaN-propagating)
  float m = 0.0f;
  if (row_ok && q0 + CW <= p.Q) {
#pragma unroll
    for (int i = 0; i < CW; ++i) m = max_nan(m, fabsf(v[i]));
  } else if (row_ok) {
#pragma unroll
    for (int i = 0; i < CW; ++i) m = max_nan(m, (q0 + i < p.Q) ? fabsf(v[i]) : 0.0f);
  }
  const bool has_nan = m != m;
  if constexpr (!STREAM) {
    if (lane == 0) ptx::bulk_wait_read_one();  // this buffer's previous store has read it
    __syncwarp();
  }
  if constexpr (ES == 1) {
    // FP8 output: amax of the fp32 values before scale_result (it sets the
    // next quantisation scale), then one saturating rounding of v * sr.
    if (!has_nan) amax_f = fmaxf(amax_f, m);
    const bool e5 = p.out_dtype == 4;
    uint32_t w[(CW + 3) / 4];
#pragma unroll
    for (int i = 0; i < CW / 4; ++i)
      w[i] = cvt_fp8x2(v[4 * i] * sr, v[4 * i + 1] * sr, e5) | (cvt_fp8x2(v[4 * i + 2] * sr, v[4 * i + 3] * sr, e5) << 16);
    if (NOSWAP || !p.swap) {
#pragma unroll
      for (int c = 0; c < CW / 16; ++c) {
        const uint32_t off = swz((uint32_t)lane * p.out_rowbytes + c * 16u, p.out_swz_mask);
        *reinterpret_cast<uint4*>(stg_gen + off) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      }
    } else if constexpr (!NOSWAP) {
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        const uint32_t off = swz((uint32_t)i * p.out_rowbytes + lane, p.out_swz_mask);
        stg_gen[off] = (uint8_t)(w[i / 4] >> (8 * (i % 4)));
      }
    }
  } else if constexpr (ES == 4) {
    uint32_t w[CW];
#pragma unroll
    for (int i = 0; i < CW; ++i) {
      const uint32_t bits = __float_as_uint(v[i]);
      w[i] = ((bits & 0x7FFFFFFFu) > 0x7F800000u) ? 0x7FFFFFFFu : bits;
    }
    if (!has_nan) amax_f = fmaxf(amax_f, m);
    if (NOSWAP || !p.swap) {
#pragma unroll
      for (int c = 0; c < CW / 4; ++c) {
        const uint32_t off = swz((uint32_t)lane * p.out_rowbytes + c * 16u, p.out_swz_mask);
        *reinterpret_cast<uint4*>(stg_gen + off) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      }
    } else if constexpr (!NOSWAP) {
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        const uint32_t off = swz((uint32_t)i * p.out_rowbytes + lane * 4u, p.out_swz_mask);
        *reinterpret_cast<uint32_t*>(stg_gen + off) = w[i];
      }
    }
  } else {
    uint32_t w[CW / 2];
    const bool bf = p.out_dtype == 1;
#pragma unroll
    for (int i = 0; i < CW / 2; ++i) w[i] = bf ? cvt_bf16x2(v[2 * i], v[2 * i + 1]) : cvt_f16x2(v[2 * i], v[2 * i + 1]);
    if (has_nan) {
#pragma unroll
      for (int i = 0; i < CW / 2; ++i) {
        if (v[2 * i] != v[2 * i]) w[i] = (w[i] & 0xFFFF0000u) | 0x7FFFu;
        if (v[2 * i + 1] != v[2 * i + 1]) w[i] = (w[i] & 0x0000FFFFu) | 0x7FFF0000u;
      }
    } else {
      // the stored magnitude of the largest value, widened back to fp32
      const float mr = bf ? __uint_as_float(cvt_bf16x2(m, 0.0f) << 16)
                          : __half2float(__ushort_as_half((unsigned short)(cvt_f16x2(m, 0.0f) & 0xFFFFu)));
      amax_f = fmaxf(amax_f, mr);
    }
    if (NOSWAP || !p.swap) {
#pragma unroll
      for (int c = 0; c < CW / 8; ++c) {
        const uint32_t off = swz((uint32_t)lane * p.out_rowbytes + c * 16u, p.out_swz_mask);
        *reinterpret_cast<uint4*>(stg_gen + off) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
      }
    } else if constexpr (!NOSWAP) {
#pragma unroll
      for (int i = 0; i < CW; ++i) {
        const uint32_t off = swz((uint32_t)i * p.out_rowbytes + lane * 2u, p.out_swz_mask);
        *reinterpret_cast<uint16_t*>(stg_gen + off) = (uint16_t)((i & 1) ? (w[i / 2] >> 16) : (w[i / 2] & 0xFFFFu));
      }
    }
  }
  if (has_nan) amax_nan = 1u;
  ptx::fence_proxy_async_smem();
  __syncwarp();
  // A box that starts inside C is clipped by the TMA unit; one that starts
  // past its end holds nothing to store and is skipped (no group is committed).
  if (lane == 0) {
    if (in_bounds) ptx::tma_store_3d(tm_c, stg_s, cx, cy, cl);
    if constexpr (!STREAM) ptx::bulk_commit();
  }
}

// Epilogue warps 0..EW-1.  Warp w reads TMEM lanes 32*(w%4) .. +31 (the tile
// rows it may access) and the columns of part w/4 (two parts for 8 warps,
// four for 16).  Per work unit: (slow) promote
// each 128-K chunk into fp32 registers; (split-K) publish the partial tile and
// let the last arrival finish it; then scale, cast, amax and store.
template <int BN, bool SLOW, int CG, int EW, int CW, int ES, bool HOLD>
__device__ __forceinline__ void epilogue(const KParams& p, const CUtensorMap* tm_c, uint8_t* sgen, uint32_t sbase,
                                         uint32_t tmem_base, uint32_t bar_tfull, uint32_t bar_tempty, uint32_t bar_epi,
                                         volatile uint32_t* misc, volatile uint32_t* abort_flag, uint32_t rank,
                                         long long u_first, long long u_step, int warp, int lane) {
  constexpr int HMAX = part_max_cols(BN, EW, SLOW);  // widest column range of a warp
  constexpr bool WIDE = wide_slow(BN, SLOW);  // slow 224/256-column tile: HMAX promoted sums per thread
  // columns per tcgen05.ld while promoting (held tiles: 16, measured faster than 8 or 32)
  constexpr int LDW = HMAX < 32 ? HMAX : (HOLD ? 16 : 32);
  static_assert(!WIDE || HOLD, "slow 256-column tiles hold their sums");
  static_assert(EW == 8 || EW == 16, "8 or 16 epilogue warps");
  static_assert(EW == 8 || BN % 128 == 0, "16 epilogue warps split 128-multiple tiles in four");
  static_assert(!SLOW || HMAX * (EW / 4) == BN, "slow accumulation splits the tile evenly");
  static_assert(HMAX % CW == 0 && (BN - HMAX) % CW == 0, "chunks tile each part");
  constexpr int kStageOut = stage_out_bytes(EW, HOLD, ES, HMAX);
  // Held tiles with 1- or 2-byte outputs stage all of a warp's chunks at once
  // and store them back to back: with two alternating buffers each chunk
  // waited for the TMA unit to read the one before last, and on GB300 a held
  // 128 x 256 tile's stores took about 19,000 cycles, during which the MMA
  // could run only two chunks ahead.
  constexpr bool kWhole = HOLD && ES <= 2;
  constexpr int kChunkBytes = 32 * CW * ES;
  static_assert(!kWhole || kStageOut == (HMAX / CW) * kChunkBytes, "a whole block of chunks");
  const int qd = warp & 3;
  const int h = warp >> 2;
  const int row = qd * 32 + lane;
  const int col0 = (EW == 8) ? (h ? HMAX : 0) : h * HMAX;
  const int ncols = (EW == 8) ? (h ? BN - HMAX : HMAX) : HMAX;
  const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
  uint32_t abuf = 0, aphase = 0, epi_phase = 0;
  float amax_f = 0.0f;
  uint32_t amax_nan = 0u;
  bool ok = true;
  const float alpha = p.sa_tensor ? (__ldg(p.sa_tensor) * __ldg(p.sb_tensor)) : 1.0f;
  const float sr = (ES == 1 && p.scale_result) ? __ldg(p.scale_result) : 1.0f;
  float* ys_w = reinterpret_cast<float*>(sgen + p.off_ys) + warp * HMAX;
  float* bias_w = reinterpret_cast<float*>(sgen + p.off_bias) + warp * HMAX;  // this warp's columns' bias
  uint8_t* stg = sgen + p.off_out + warp * kStageOut;
  const uint32_t stg_s = sbase + p.off_out + warp * kStageOut;
  uint32_t stg_sel = 0;
  // Slow accumulation: fp32 running sums of the promoted chunks -- in pairs
  // for the packed (two-lane) fp32 instructions on 256-column tiles, single
  // on the narrower ones (which measured faster with scalar code).
  static_assert(HMAX % 2 == 0, "column ranges pair up");
  float acc1[(SLOW && !WIDE) ? HMAX : 1];
  float2 acc2[HOLD ? HMAX / 2 : 1];
  auto acc = [&](int i) -> float& {
    if constexpr (HOLD)
      return (i & 1) ? acc2[i >> 1].y : acc2[i >> 1].x;
    else
      return acc1[i];
  };
  (void)acc;
  (void)ys_w;
  // The pair leader's accumulator-empty barrier collects both CTAs' warps.
  const uint32_t tempty_target = (CG == 2) ? ptx::mapa_shared(bar_tempty, 0u) : bar_tempty;
  // Every TMEM read before a release went through tmem_load, whose
  // tcgen05.wait::ld has the values in registers, so nothing the next MMA
  // writes can reach them.  One CTA keeps the tcgen05 fence before the arrive
  // (it costs nothing there); on a CTA pair it measured ~70 cycles per chunk
  // of the hand-off on GB300, and is left out.
  auto release_acc = [&]() {
    if constexpr (CG == 1) ptx::tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
      if constexpr (CG == 2)
        ptx::mbar_arrive_cluster(tempty_target + 8u * abuf);
      else
        ptx::mbar_arrive(bar_tempty + 8u * abuf);
    }
    if (++abuf == (uint32_t)p.num_acc) {
      abuf = 0;
      aphase ^= 1u;
    }
  };

  for (long long u = u_first; ok && u < p.units; u += u_step) {
    const Unit t = decode_unit(u, p);
    const int xbase = t.tr * kBlockM * CG + (int)rank * kBlockM;  // first X row of this CTA's half
    const int xr = xbase + row;                                   // row of X this thread owns
    const bool row_ok = xr < p.R;
    if constexpr (SLOW && !WIDE) {
      // One hand-off per 128-K chunk: acc += s_x(row, c) * s_y(col, c) * chunk.
      for (int g = 0; g < t.kb1 - t.kb0; ++g) {
        float xs = 1.0f, yb = 1.0f;
        if (p.x_kind != kScaleNone) {
          const int c = t.kb0 + g;
          if (row_ok) {
            xs = (p.x_kind == kScaleRow)
                     ? __ldg(p.x_scale + ((size_t)t.l * p.R + xr) * p.scale_kb + c)
                     : __ldg(p.x_scale + ((size_t)t.l * ((p.R + 127) / 128) + xr / 128) * p.scale_kb + c);
          }
          if (p.y_kind == kScaleBlock128) {
            // a warp's columns lie in one 128-column block: one scale per warp and chunk
            const int yq = t.tq * BN + col0;
            yb = (yq < p.Q) ? __ldg(p.y_scale + ((size_t)t.l * ((p.Q + 127) / 128) + yq / 128) * p.scale_kb + c)
                            : 0.0f;
          } else {
            __syncwarp();
            for (int j = lane; j < ncols; j += 32) {
              const int yq = t.tq * BN + col0 + j;
              ys_w[j] = (yq < p.Q) ? __ldg(p.y_scale + ((size_t)t.l * p.Q + yq) * p.scale_kb + c) : 0.0f;
            }
            __syncwarp();
          }
        }
        if (!wait_bar(bar_tfull + 8u * abuf, aphase, abort_flag, p.abort_word, kErrEpiAcc)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after_sync();
        const uint32_t taddr = tmem_base + lane_off + abuf * BN + col0;
        const float f = xs * yb;
#pragma unroll
        for (int pc = 0; pc < HMAX / LDW; ++pc) {
          uint32_t r[LDW];
          tmem_load<LDW>(taddr + pc * LDW, r);
          // One fp32 instruction per element (the promotion is issue-bound).
#pragma unroll
          for (int i = 0; i < LDW; ++i) {
            const int j = pc * LDW + i;
            const float v = __uint_as_float(r[i]);
            if (p.x_kind == kScaleNone)
              acc1[j] = (g == 0) ? v : acc1[j] + v;
            else if (p.y_kind == kScaleBlock128)
              acc1[j] = (g == 0) ? f * v : fmaf(f, v, acc1[j]);
            else
              acc1[j] = (g == 0) ? (xs * ys_w[j]) * v : fmaf(xs * ys_w[j], v, acc1[j]);
          }
        }
        release_acc();
      }
      if (!ok) break;
    } else if constexpr (WIDE) {
      // One hand-off per 128-K chunk: acc += s_x(row, c) * s_y(col, c) * chunk.
      // The sums start at -0, which leaves the first product (even a zero)
      // unchanged, so every chunk takes the same single instruction per element.
#pragma unroll
      for (int j = 0; j < HMAX / 2; ++j) acc2[j] = make_float2(-0.0f, -0.0f);
      // Block scales of chunk g + 1 are loaded while chunk g is promoted.
      constexpr int YSR = (HMAX + 31) / 32;  // per-column Y scales held per lane
      auto load_scales = [&](int g, float& xs, float& yb, float (&ysr)[YSR]) {
        xs = 1.0f;
        yb = 1.0f;
        if (p.x_kind == kScaleNone) return;
        const int c = t.kb0 + g;
        if (row_ok) {
          xs = (p.x_kind == kScaleRow)
                   ? __ldg(p.x_scale + ((size_t)t.l * p.R + xr) * p.scale_kb + c)
                   : __ldg(p.x_scale + ((size_t)t.l * ((p.R + 127) / 128) + xr / 128) * p.scale_kb + c);
        }
        if (p.y_kind == kScaleBlock128) {
          // a warp's columns lie in one 128-column block: one scale per warp and chunk
          const int yq = t.tq * BN + col0;
          yb = (yq < p.Q) ? __ldg(p.y_scale + ((size_t)t.l * ((p.Q + 127) / 128) + yq / 128) * p.scale_kb + c)
                          : 0.0f;
        } else {
#pragma unroll
          for (int i = 0; i < YSR; ++i) {
            const int j = lane + 32 * i;
            const int yq = t.tq * BN + col0 + j;
            ysr[i] = (j < ncols && yq < p.Q) ? __ldg(p.y_scale + ((size_t)t.l * p.Q + yq) * p.scale_kb + c) : 0.0f;
          }
        }
      };
      auto stage_ys = [&](const float (&ysr)[YSR]) {
        if (p.x_kind == kScaleNone || p.y_kind == kScaleBlock128) return;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < YSR; ++i)
          if (lane + 32 * i < HMAX) ys_w[lane + 32 * i] = ysr[i];
        __syncwarp();
      };
      float xs, yb, ysr[YSR];
      load_scales(0, xs, yb, ysr);
      stage_ys(ysr);
      const int nchunks = t.kb1 - t.kb0;
      for (int g = 0; g < nchunks; ++g) {
        float xs_n = 1.0f, yb_n = 1.0f, ysr_n[YSR];
        if (g + 1 < nchunks) load_scales(g + 1, xs_n, yb_n, ysr_n);
        if (!wait_bar(bar_tfull + 8u * abuf, aphase, abort_flag, p.abort_word, kErrEpiAcc)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after_sync();
        const uint32_t taddr = tmem_base + lane_off + abuf * BN + col0;
        // One packed fp32 instruction per two elements.  Per-tensor scales
        // (f = 1: fma(1, v, acc) rounds v + acc once, like an add) and 128x128
        // blocks of Y take one factor per warp; per-column Y scales one per
        // column.  Each form is its own straight-line loop: the promotion runs
        // once per chunk and must stay small in the instruction cache.
        if (p.x_kind == kScaleNone || p.y_kind == kScaleBlock128) {
          const float f = xs * yb;
          const float2 f2 = make_float2(f, f);
#pragma unroll
          for (int pc = 0; pc < HMAX / LDW; ++pc) {
            uint32_t r[LDW];
            tmem_load<LDW>(taddr + pc * LDW, r);
#pragma unroll
            for (int i = 0; i < LDW; i += 2) {
              const int j = (pc * LDW + i) / 2;
              acc2[j] = __ffma2_rn(f2, make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), acc2[j]);
            }
          }
        } else {
          const float2 xs2 = make_float2(xs, xs);
#pragma unroll
          for (int pc = 0; pc < HMAX / LDW; ++pc) {
            uint32_t r[LDW];
            tmem_load<LDW>(taddr + pc * LDW, r);
#pragma unroll
            for (int i = 0; i < LDW; i += 2) {
              const int j = (pc * LDW + i) / 2;
              const float2 s2 = __fmul2_rn(xs2, reinterpret_cast<const float2*>(ys_w)[j]);
              acc2[j] = __ffma2_rn(s2, make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), acc2[j]);
            }
          }
        }
        release_acc();
        if (g + 1 < nchunks) {
          xs = xs_n;
          yb = yb_n;
          stage_ys(ysr_n);
        }
      }
      if (!ok) break;
    } else {
      if (!wait_bar(bar_tfull + 8u * abuf, aphase, abort_flag, p.abort_word, kErrEpiAcc)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      if constexpr (HOLD) {
        // Copy the whole accumulator out and hand TMEM back to the MMA issuer
        // before storing anything.
        const uint32_t taddr = tmem_base + lane_off + abuf * BN + col0;
#pragma unroll
        for (int pc = 0; pc < HMAX / 16; ++pc) {
          uint32_t r[16];
          tmem_load<16>(taddr + pc * 16, r);
#pragma unroll
          for (int i = 0; i < 16; i += 2)
            acc2[(pc * 16 + i) / 2] = make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
        }
        release_acc();
      }
    }
    // Fast accumulation reads the finished tile from TMEM chunk by chunk.
    const uint32_t taddr = tmem_base + lane_off + abuf * BN + col0;
    // Slow accumulation: the chunk being stored is always acc[0 .. CW); after
    // each chunk the sums rotate left by CW, so one copy of the loop body
    // serves every chunk and a full pass restores the original order.
    auto rotate_acc = [&](const float(&v)[CW]) {  // v: the chunk just read from acc[0 .. CW)
      if constexpr (SLOW) {
#pragma unroll
        for (int i = 0; i < HMAX - CW; ++i) acc(i) = acc(i + CW);
#pragma unroll
        for (int i = 0; i < CW; ++i) acc(HMAX - CW + i) = v[i];
      }
    };
    auto get_chunk = [&](int ci, float(&v)[CW]) {
      if constexpr (SLOW) {
        (void)ci;
#pragma unroll
        for (int i = 0; i < CW; ++i) v[i] = acc(i);
      } else {
        uint32_t r[CW];
        tmem_load<CW>(taddr + ci * CW, r);
#pragma unroll
        for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]);
      }
    };
    const int nch = ncols / CW;

    // ---------------------------------------------------- split-K fix-up
    bool finish = true;
    float* tile_ws = nullptr;
    if (!HOLD && p.splits > 1) {  // (held tiles are never split)
      const long long tile = (((long long)t.l * p.tiles_r + t.tr) * p.tiles_q + t.tq) * CG + rank;
      tile_ws = p.ws_partials + (size_t)tile * p.splits * (kBlockM * BN);
      float* slot = tile_ws + (size_t)t.s * (kBlockM * BN);
      // One copy of each loop body: a compact epilogue runs from the
      // instruction cache from the first tile on.
#pragma unroll 1
      for (int ci = 0; ci < nch; ++ci) {
        float v[CW];
        get_chunk(ci, v);
        rotate_acc(v);
#pragma unroll
        for (int i = 0; i < CW; ++i) __stcg(slot + (size_t)(col0 + ci * CW + i) * kBlockM + row, v[i]);
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_epi);
      if (!wait_bar(bar_epi, epi_phase, abort_flag, p.abort_word, kErrEpiSync)) {
        ok = false;
        break;
      }
      epi_phase ^= 1u;
      if (warp == 0 && lane == 0) {
        __threadfence();
        misc[2] = atomicAdd(p.ws_counters + tile, 1u);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_epi);
      if (!wait_bar(bar_epi, epi_phase, abort_flag, p.abort_word, kErrEpiSync)) {
        ok = false;
        break;
      }
      epi_phase ^= 1u;
      finish = misc[2] == (uint32_t)(p.splits - 1);  // the last arrival finishes the tile
      if (finish) __threadfence();
    }

    // ---------------------------------------------------- scale, cast, store
    if (finish) {
      const int r0 = xbase + qd * 32;  // X row of the warp's first lane
      // The bias of the warp's columns, staged once per tile (unswapped), or
      // of the thread's own output column (swapped).
      float bias_lane = 0.0f;
      if (ES != 1 && p.bias != nullptr) {
        if (!p.swap) {
          const int qb = t.tq * BN + col0;
          for (int j = lane; j < ncols; j += 32) bias_w[j] = (qb + j < p.Q) ? bias_at(p, qb + j) : 0.0f;
          __syncwarp();
        } else if (row_ok) {
          bias_lane = bias_at(p, xr);
        }
      }
      if constexpr (kWhole) {
        // the previous tile's stores have read the staging block
        if (lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
      }
      auto finish_chunk = [&](int ci) {
        if constexpr (kWhole) {
          // The held sums are stored in place: the chunk is acc[0 .. CW),
          // then the others move down by CW.  Chunk ci has its own slot.
          const int q0 = t.tq * BN + col0 + ci * CW;
          float v[CW];
#pragma unroll
          for (int i = 0; i < CW; ++i) v[i] = acc(i);
          store_chunk<CW, ES, CW, true, true>(p, tm_c, v, alpha, sr, bias_w + ci * CW, bias_lane, row_ok, q0, lane,
                                                stg + ci * kChunkBytes, stg_s + ci * kChunkBytes, q0, r0, t.l,
                                                q0 < p.Q && r0 < p.R, amax_f, amax_nan);
#pragma unroll
          for (int i = 0; i < (HMAX - CW) / 2; ++i) acc2[i] = acc2[i + CW / 2];
        } else if constexpr (HOLD) {
          // The held sums are stored in place: the chunk is acc[0 .. CW),
          // then the others move down by CW.
          const int q0 = t.tq * BN + col0 + ci * CW;
          float v[CW];
#pragma unroll
          for (int i = 0; i < CW; ++i) v[i] = acc(i);
          store_chunk<CW, ES, CW, true>(p, tm_c, v, alpha, sr, bias_w + ci * CW, bias_lane, row_ok, q0, lane,
                                          stg + stg_sel * (kStageOut / 2),
                                          stg_s + stg_sel * (kStageOut / 2), q0, r0, t.l, q0 < p.Q && r0 < p.R,
                                          amax_f, amax_nan);
          stg_sel ^= 1u;
#pragma unroll
          for (int i = 0; i < (HMAX - CW) / 2; ++i) acc2[i] = acc2[i + CW / 2];
        } else {
          float v[CW];
          get_chunk(ci, v);
          rotate_acc(v);
          if (p.splits > 1) {
            // Partials are added in split order 0..S-1 whichever CTA arrived
            // last.  Each split's chunk is loaded as one batch of independent
            // loads before it is added, so the loads overlap.
            const float* base = tile_ws + (size_t)(col0 + ci * CW) * kBlockM + row;
            float sum[CW];
#pragma unroll
            for (int i = 0; i < CW; ++i) sum[i] = (t.s == 0) ? v[i] : __ldcg(base + (size_t)i * kBlockM);
            for (int ss = 1; ss < p.splits; ++ss) {
              float part[CW];
              if (ss == t.s) {
#pragma unroll
                for (int i = 0; i < CW; ++i) part[i] = v[i];
              } else {
                const float* src = base + (size_t)ss * (kBlockM * BN);
#pragma unroll
                for (int i = 0; i < CW; ++i) part[i] = __ldcg(src + (size_t)i * kBlockM);
              }
#pragma unroll
              for (int i = 0; i < CW; ++i) sum[i] += part[i];
            }
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] = sum[i];
          }
          const int q0 = t.tq * BN + col0 + ci * CW;  // Y row of the chunk's first column
          store_chunk<CW, ES>(p, tm_c, v, alpha, sr, bias_w + ci * CW, bias_lane, row_ok, q0, lane,
                              stg + stg_sel * (kStageOut / 2),
                              stg_s + stg_sel * (kStageOut / 2), p.swap ? r0 : q0, p.swap ? q0 : r0, t.l,
                              q0 < p.Q && r0 < p.R, amax_f, amax_nan);
          stg_sel ^= 1u;
        }
      };
#pragma unroll 1
      for (int ci = 0; ci < nch; ++ci) finish_chunk(ci);
      if constexpr (kWhole) {
        if (lane == 0) ptx::bulk_commit();
      }
    }
    if constexpr (!SLOW && !HOLD) release_acc();
  }
  if (lane == 0) ptx::bulk_wait_all();
  uint32_t amax_local = amax_nan ? 0x7FFFFFFFu : __float_as_uint(amax_f);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax_local = max(amax_local, __shfl_xor_sync(0xFFFFFFFFu, amax_local, o));
  if (lane == 0 && amax_local != 0u) atomicMax(p.amax_bits, amax_local);
}

// F4: packed FP4 (E2M1) operands with block scaling (kind::mxf4nvf4): a stage
// row of 128 bytes holds 256 elements, four MMAs of K = 64; each stage brings
// the 4 (E4M3 per 16) or 2 (UE8M0 per 32) factor atoms of X and of Y that
// cover its 256 elements.
template <int BN, bool SLOW, bool MX, int CG, int EW, bool F4 = false>
__global__ void __launch_bounds__(kernel_threads(EW, held_tile(BN, SLOW, MX)), 1)
    fp8mm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
                 const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_sfx,
                 const __grid_constant__ CUtensorMap tm_sfy, const KParams p) {
  static_assert(!F4 || (MX && (BN == 128 || BN == 256) && !SLOW && CG == 1),
                "FP4: 128- or 256-column block-scaled tiles, fast");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
  static_assert(!MX || BN == 128 || BN == 256 || (BN % 32 == 0 && BN < 256),
                "MX tiles start on a 32-row boundary of a factor atom");
  static_assert(!SLOW || BN <= 128 || ((BN == 256 || BN == 224 || BN == 192) && !MX && EW == 8) ||
                    (BN == 256 && CG == 1 && !MX),
                "slow accumulation keeps its promoted sums in registers: 192-, 224- or 256-column tiles");
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair per MMA");
  static_assert(!MX || CG == 1 || (BN == 256 && !SLOW && !F4), "block-scaled CTA pairs: fast FP8 256-column tiles");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sraw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (sraw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - sraw);

  constexpr int kProdWarp = EW;
  // MX tiles not aligned to 128 rows (224 columns): the producer warp gathers
  // Y's factor bytes into atoms that start at the tile's first row, with
  // 4-byte asynchronous copies whose completion the stage's full barrier
  // tracks (one arrival per lane besides the producer's).
  constexpr bool GATHER = MX && (BN % 128) != 0;
  constexpr int kMmaWarp = EW + 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  if constexpr (held_tile(BN, SLOW, MX)) {
    // Held tiles are planned without split-K or swapped operands, and 192-
    // or 224-column tiles (whose halves straddle 128-column blocks) without
    // 128x128 Y scales.
    if (p.splits != 1 || p.swap || (BN % 128 != 0 && p.y_kind == kScaleBlock128)) {
      if (threadIdx.x == 0) atomicOr(p.abort_word, kErrPlan);
      return;
    }
  }
  // FP8 outputs store rows of at least 16 bytes starting on 16-byte columns
  // (a TMA store's rule): unswapped tiles need chunks of 16 columns or more.
  if (p.out_es == 1 && !p.swap && chunk_cols(BN, 1, EW, held_tile(BN, SLOW, MX), SLOW) < 16) {
    if (threadIdx.x == 0) atomicOr(p.abort_word, kErrPlan);
    return;
  }
  // CG == 2: a cluster of two CTAs computes 256-row tiles with two-SM MMAs
  // issued by the leader (rank 0); each CTA stages its own 128 rows of X and
  // half of the Y tile, and holds its 128 rows of the accumulator in TMEM.
  const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0u;
  const long long u_first = blockIdx.x / CG;
  const long long u_step = gridDim.x / CG;

  const uint32_t bar_full = sbase + p.off_bar;
  const uint32_t bar_empty = bar_full + 8u * S;
  const uint32_t bar_tfull = bar_empty + 8u * S;
  const uint32_t bar_tempty = bar_tfull + 32u;  // up to four accumulators
  const uint32_t bar_epi = bar_tempty + 32u;
  const uint32_t bar_done = bar_epi + 8u;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(sgen + p.off_bar + 16u * S + 80u);
  // misc[0] TMEM base address, misc[1] abort flag, misc[2] split-K ticket

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(bar_full + 8u * s, GATHER ? 33 : 1);
      ptx::mbar_init(bar_empty + 8u * s, 1);
    }
    for (int b = 0; b < 4; ++b) {
      ptx::mbar_init(bar_tfull + 8u * b, 1);
      ptx::mbar_init(bar_tempty + 8u * b, EW * CG);  // the pair's epilogue warps arrive on the leader
    }
    ptx::mbar_init(bar_epi, EW);
    ptx::mbar_init(bar_done, 1);
    misc[1] = 0u;
    misc[2] = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    if constexpr (CG == 2) {
      ptx::tmem_alloc_pair(ptx::smem_u32(const_cast<uint32_t*>(misc)), p.tmem_cols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(misc)), p.tmem_cols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before_sync();
  if constexpr (CG == 2)
    ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other
  else
    __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = misc[0];
  volatile uint32_t* abort_flag = misc + 1;

  constexpr bool REGSPLIT = held_tile(BN, SLOW, MX);
  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if constexpr (REGSPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegRoles));
    if (GATHER || lane == 0) {
      if (lane == 0) {
        ptx::prefetch_tensormap(&tm_x);
        ptx::prefetch_tensormap(&tm_y);
        ptx::prefetch_tensormap(&tm_c);
      }
      uint32_t stage = 0, phase = 0;
      long long narm = 0;
      bool ok = !p.withhold_loads;
      // With a CTA pair both CTAs' copies complete on the leader's full barrier,
      // which the leader arms with the bytes of both.
      for (long long u = u_first; ok && u < p.units; u += u_step) {
        const Unit t = decode_unit(u, p);
        const int xrow0 = t.tr * kBlockM * CG + (int)rank * kBlockM;
        const int yrow0 = t.tq * BN + (int)rank * (BN / CG);
        // MX: Y's tile may start inside a 128-row atom; copy every atom it touches.
        const int y_atom0 = (t.tq * BN) / 128;
        const int y_atoms = (MX && !GATHER) ? ((t.tq * BN) % 128 + BN + 127) / 128 : 0;
        const uint32_t tx0 = CG * (p.x_stage_bytes + p.y_stage_bytes + ((MX && !F4) ? 512u * (1 + y_atoms) : 0u));
        const int apk = p.f4_vec16 ? 4 : 2;  // FP4: factor atoms per stage and operand
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          // FP4: the atoms that exist for this stage's 256 elements of K
          const int f4_na = F4 ? min(apk, p.scale_kb - kb * apk) : 0;
          const uint32_t tx = tx0 + (F4 ? 512u * (uint32_t)f4_na * (1 + BN / 128) : 0u);
          {
            bool w = wait_bar(bar_empty + 8u * stage, phase ^ 1u, abort_flag, p.abort_word, kErrProducer);
            if constexpr (GATHER) w = __all_sync(0xFFFFFFFFu, w);  // the lanes leave together
            if (!w) {
              ok = false;
              break;
            }
          }
          const uint32_t fb = bar_full + 8u * stage;
          if (!GATHER || lane == 0) {
          if constexpr (CG == 2) {
            const uint32_t fb_leader = ptx::mapa_shared(fb, 0u);
            if (leader) ptx::mbar_arrive_expect_tx(fb, tx);
            ptx::tma_load_3d_pair(sbase + p.off_x + stage * p.x_stage_bytes, &tm_x, fb_leader, kb * kBlockK, xrow0,
                                  t.l);
            ptx::tma_load_3d_pair(sbase + p.off_y + stage * p.y_stage_bytes, &tm_y, fb_leader, kb * kBlockK, yrow0,
                                  t.l);
          } else {
            ptx::mbar_arrive_expect_tx(fb, tx);
            ptx::tma_load_3d(sbase + p.off_x + stage * p.x_stage_bytes, &tm_x, fb, kb * kBlockK, xrow0, t.l);
            ptx::tma_load_3d(sbase + p.off_y + stage * p.y_stage_bytes, &tm_y, fb, kb * kBlockK, yrow0, t.l);
          }
          if constexpr (F4) {
            // X atoms in slots 0 .. apk-1, then the atoms of each 128-row block
            // of the Y tile (apk slots each).  A row block's atoms lie
            // contiguous along K: one copy per operand and row block.  Blocks
            // past the last one are clamped to it; their rows are never stored.
            const uint32_t sf = sbase + p.off_sf + stage * p.sf_stage_bytes;
            const size_t a0 = (size_t)kb * apk;
            ptx::bulk_load(sf, p.sfx + (((size_t)t.l * p.sfx_mb + t.tr) * p.scale_kb + a0) * 512u,
                           512u * (uint32_t)f4_na, fb);
#pragma unroll
            for (int j = 0; j < BN / 128; ++j) {
              const int mb = min(t.tq * (BN / 128) + j, p.sfy_mb - 1);
              ptx::bulk_load(sf + 512u * apk * (1 + j), p.sfy + (((size_t)t.l * p.sfy_mb + mb) * p.scale_kb + a0) * 512u,
                             512u * (uint32_t)f4_na, fb);
            }
          } else if constexpr (MX && CG == 2) {
            // CTA pair: each CTA stages the factor atom of its own 128 rows of
            // X and every atom of the Y tile (the pair MMA reads all of Y's
            // factors from each CTA's TMEM).  The copies go through TMA
            // tensor maps over the atoms, so that they complete on the
            // leader's full barrier like the operand tiles.
            const uint32_t sf = sbase + p.off_sf + stage * p.sf_stage_bytes;
            const uint32_t fb_leader = ptx::mapa_shared(fb, 0u);
            const int xmb = min(t.tr * 2 + (int)rank, p.sfx_mb - 1);
            ptx::tma_load_3d_pair(sf, &tm_sfx, fb_leader, 0, 0,
                                  (int)(((size_t)t.l * p.sfx_mb + xmb) * p.scale_kb + kb));
            for (int i = 0; i < y_atoms; ++i) {
              const int mb = min(y_atom0 + i, p.sfy_mb - 1);
              ptx::tma_load_3d_pair(sf + 512u * (1 + i), &tm_sfy, fb_leader, 0, 0,
                                    (int)(((size_t)t.l * p.sfy_mb + mb) * p.scale_kb + kb));
            }
          } else if constexpr (MX) {
            const uint32_t sf = sbase + p.off_sf + stage * p.sf_stage_bytes;
            const uint8_t* gx =
                p.sfx + (((size_t)t.l * p.sfx_mb + t.tr) * p.scale_kb + kb) * 512u;
            ptx::bulk_load(sf, gx, 512u, fb);
            for (int i = 0; i < y_atoms; ++i) {
              // atoms past the last row block are clamped to it; their rows are never stored
              const int mb = min(y_atom0 + i, p.sfy_mb - 1);
              const uint8_t* gy = p.sfy + (((size_t)t.l * p.sfy_mb + mb) * p.scale_kb + kb) * 512u;
              ptx::bulk_load(sf + 512u * (1 + i), gy, 512u, fb);
            }
          }
          }  // (lane 0)
          if constexpr (GATHER) {
            // Gathered atom v, line `lane`, word c: the factors of tile row
            // 128 v + 32 c + lane, which sit in word (row % 128) / 32 of line
            // row % 32 (= lane: tiles start on a 32-row boundary) of the row's
            // atom.  Atoms past the last row block are clamped to it.
            const uint32_t sf = sbase + p.off_sf + stage * p.sf_stage_bytes;
#pragma unroll
            for (int v = 0; v < (BN + 127) / 128; ++v) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int row = t.tq * BN + 128 * v + 32 * c + lane;
                const int mb = min(row / 128, p.sfy_mb - 1);
                const uint8_t* src = p.sfy + (((size_t)t.l * p.sfy_mb + mb) * p.scale_kb + kb) * 512u +
                                     (uint32_t)lane * 16u + (uint32_t)((row % 128) / 32) * 4u;
                ptx::cp_async_4(sf + 512u * (1 + v) + (uint32_t)lane * 16u + (uint32_t)c * 4u, src);
              }
            }
            ptx::cp_async_mbar_arrive_noinc(fb);
          }
          ++narm;
          if (++stage == (uint32_t)S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Wait until every copy this thread started has landed (all of them
      // were consumed already unless another role aborted).
      // (stage, phase) is the next slot: slots below it were last armed in
      // this pass of the ring, the others in the previous pass.  With a CTA
      // pair the leader's barriers also track the peer's copies.
      if (leader && lane == 0) {
        for (int s = 0; s < S; ++s) {
          if (narm > s) drain_wait(bar_full + 8u * s, ((uint32_t)s < stage) ? phase : (phase ^ 1u), p.abort_word);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if constexpr (REGSPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegRoles));
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
      bool ok = true;
      for (long long u = u_first; ok && u < p.units; u += u_step) {
        const Unit t = decode_unit(u, p);
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          const bool gstart = SLOW || kb == t.kb0;
          const bool gend = SLOW || kb == t.kb1 - 1;
          if (gstart) {
            if (!wait_bar(bar_tempty + 8u * abuf, aphase ^ 1u, abort_flag, p.abort_word, kErrMmaAcc)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after_sync();
          }
          if (!wait_bar(bar_full + 8u * stage, phase, abort_flag, p.abort_word, kErrMmaFull)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after_sync();
          const uint32_t d = tmem_base + abuf * BN;
          const uint64_t adesc = ptx::desc_sw128_kmajor(sbase + p.off_x + stage * p.x_stage_bytes);
          const uint64_t bdesc = ptx::desc_sw128_kmajor(sbase + p.off_y + stage * p.y_stage_bytes);
          if constexpr (F4) {
            // TMEM slot of 4 apk (1 + BN/128) columns per stage: X's atoms (4
            // columns each), then for each K atom the Y tile's row blocks side
            // by side, so that one MMA reads its BN rows' factors from adjacent
            // columns (row r of the tile in column r / 32).
            constexpr int NYB = BN / 128;
            const int apk = p.f4_vec16 ? 4 : 2;
            const int na = min(apk, p.scale_kb - kb * apk);
            const uint32_t sf_smem = sbase + p.off_sf + stage * p.sf_stage_bytes;
            const uint32_t sf_x = tmem_base + (uint32_t)(p.num_acc * BN) + stage * (uint32_t)(4 * apk * (1 + NYB));
            const uint32_t sf_y = sf_x + 4u * (uint32_t)apk;
            for (int i = 0; i < na; ++i) {
              ptx::tmem_cp_32x128b_warpx4(sf_x + 4u * i, ptx::desc_sf_atom(sf_smem + 512u * i));
#pragma unroll
              for (int j = 0; j < NYB; ++j)
                ptx::tmem_cp_32x128b_warpx4(sf_y + 4u * (uint32_t)(NYB * i + j),
                                            ptx::desc_sf_atom(sf_smem + 512u * (uint32_t)(apk * (1 + j) + i)));
            }
#pragma unroll
            for (int k = 0; k < kBlockK / 32; ++k) {
              // an MMA of K = 64 elements (32 bytes); none past the end of K
              if (kb * 256 + 64 * k >= p.K) break;
              const uint32_t acc = (!gstart || k > 0) ? 1u : 0u;
              if (p.f4_vec16) {
                ptx::mma_mxf4nvf4_4x(d, adesc + 2u * k, bdesc + 2u * k, p.idesc, sf_x + 4u * k,
                                     sf_y + 4u * (uint32_t)(NYB * k), acc);
              } else {
                // the atom holds 4 factors per row: MMA k reads bytes 2 (k % 2) .. +1 of atom k / 2
                const uint32_t id = (uint32_t)(k & 1) * 2u;
                ptx::mma_mxf4nvf4_2x(d, adesc + 2u * k, bdesc + 2u * k, p.idesc | (id << 29) | (id << 4),
                                     sf_x + 4u * (k >> 1), sf_y + 4u * (uint32_t)(NYB * (k >> 1)), acc);
              }
            }
          } else if constexpr (MX) {
            const uint32_t sf_smem = sbase + p.off_sf + stage * p.sf_stage_bytes;
            const uint32_t sf_x = tmem_base + (uint32_t)(p.num_acc * BN) + stage * 16u;
            // TMEM slot of 16 columns per stage: X's atom in columns 0-3, Y's
            // atoms from column 4.  Row r of an atom sits in lane r % 32 of
            // column r / 32, so a Y tile starting at row o of its first atom
            // reads its factors from column 4 + o / 32 on; gathered atoms
            // (224-column tiles) start at the tile's first row: column 4.
            const int y_atoms = GATHER ? (BN + 127) / 128 : ((t.tq * BN) % 128 + BN + 127) / 128;
            const uint32_t sf_y = sf_x + 4u + (GATHER ? 0u : (uint32_t)(((t.tq * BN) % 128) / 32));
            if constexpr (CG == 2) {
              // each CTA copies its own staged atoms into its own TMEM
              ptx::tmem_cp_32x128b_warpx4_pair(sf_x, ptx::desc_sf_atom(sf_smem));
              for (int i = 0; i < y_atoms; ++i)
                ptx::tmem_cp_32x128b_warpx4_pair(sf_x + 4u + 4u * i, ptx::desc_sf_atom(sf_smem + 512u * (1 + i)));
            } else {
              ptx::tmem_cp_32x128b_warpx4(sf_x, ptx::desc_sf_atom(sf_smem));
              for (int i = 0; i < y_atoms; ++i)
                ptx::tmem_cp_32x128b_warpx4(sf_x + 4u + 4u * i, ptx::desc_sf_atom(sf_smem + 512u * (1 + i)));
            }
#pragma unroll
            for (int k = 0; k < kBlockK / kUmmaK; ++k) {
              // scale-factor ids pick byte k of each 32-bit TMEM word: the K block of 32
              const uint32_t idesc = p.idesc | ((uint32_t)k << 29) | ((uint32_t)k << 4);
              if constexpr (CG == 2)
                ptx::mma_mxf8f6f4_pair(d, adesc + 2u * k, bdesc + 2u * k, idesc, sf_x, sf_y,
                                       (!gstart || k > 0) ? 1u : 0u);
              else
                ptx::mma_mxf8f6f4(d, adesc + 2u * k, bdesc + 2u * k, idesc, sf_x, sf_y,
                                  (!gstart || k > 0) ? 1u : 0u);
            }
          } else if constexpr (CG == 2) {
#pragma unroll
            for (int k = 0; k < kBlockK / kUmmaK; ++k)
              ptx::mma_f8f6f4_pair(d, adesc + 2u * k, bdesc + 2u * k, p.idesc, (!gstart || k > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int k = 0; k < kBlockK / kUmmaK; ++k)
              ptx::mma_f8f6f4(d, adesc + 2u * k, bdesc + 2u * k, p.idesc, (!gstart || k > 0) ? 1u : 0u);
          }
          if constexpr (CG == 2)
            ptx::tc_commit_pair(bar_empty + 8u * stage, (uint16_t)0x3);
          else
            ptx::tc_commit(bar_empty + 8u * stage);
          if (gend) {
            if constexpr (CG == 2)
              ptx::tc_commit_pair(bar_tfull + 8u * abuf, (uint16_t)0x3);
            else
              ptx::tc_commit(bar_tfull + 8u * abuf);
            if (++abuf == (uint32_t)p.num_acc) {
              abuf = 0;
              aphase ^= 1u;
            }
          }
          if (++stage == (uint32_t)S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every MMA issued above has completed before TMEM is freed.
      if constexpr (CG == 2)
        ptx::tc_commit_pair(bar_done, (uint16_t)0x1);
      else
        ptx::tc_commit(bar_done);
      drain_wait(bar_done, 0, p.abort_word);
    }
  } else if (warp < EW) {
    // ------------------------------------------------------------ epilogue
    if constexpr (REGSPLIT) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(epi_regs(EW)));
    if (p.out_es == 4)
      epilogue<BN, SLOW, CG, EW, chunk_cols(BN, 4, EW, held_tile(BN, SLOW, MX), SLOW), 4, held_tile(BN, SLOW, MX)>(p, &tm_c, sgen, sbase, tmem_base, bar_tfull, bar_tempty,
                                                            bar_epi, misc, abort_flag, rank, u_first, u_step, warp,
                                                            lane);
    else if (p.out_es == 1)
      epilogue<BN, SLOW, CG, EW, chunk_cols(BN, 1, EW, held_tile(BN, SLOW, MX), SLOW), 1, held_tile(BN, SLOW, MX)>(p, &tm_c, sgen, sbase, tmem_base, bar_tfull, bar_tempty,
                                                            bar_epi, misc, abort_flag, rank, u_first, u_step, warp,
                                                            lane);
    else
      epilogue<BN, SLOW, CG, EW, chunk_cols(BN, 2, EW, held_tile(BN, SLOW, MX), SLOW), 2, held_tile(BN, SLOW, MX)>(p, &tm_c, sgen, sbase, tmem_base, bar_tfull, bar_tempty,
                                                            bar_epi, misc, abort_flag, rank, u_first, u_step, warp,
                                                            lane);
  } else {
    // the idle warps of the last warpgroup give their registers up too
    if constexpr (REGSPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegRoles));
  }

  ptx::tc_fence_before_sync();
  if constexpr (CG == 2) {
    // Neither CTA leaves (or frees TMEM) while the pair's MMAs or copies may
    // still touch its shared memory or TMEM.
    ptx::cluster_sync();
    if (warp == kMmaWarp) {
      ptx::tc_fence_after_sync();
      ptx::tmem_dealloc_pair(tmem_base, p.tmem_cols);
    }
  } else {
    __syncthreads();
    if (warp == kMmaWarp) {
      ptx::tc_fence_after_sync();
      ptx::tmem_dealloc(tmem_base, p.tmem_cols);
    }
  }
}

}  // namespace fp8mm

namespace fp8mm {
using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                          const KParams);
}  // namespace fp8mm
