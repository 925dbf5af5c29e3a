// fp8mm_host.cu -- the C ABI declared in include/fp8mm.h: validation, the
// plan (tile shape, swap-AB, split-K, pipeline depth), TMA descriptor
// encoding and the launch of the persistent kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>

#include "fp8mm.h"
#include "fp8mm_kernels.h"

using namespace fp8mm;

// Device word recording aborted waits; kernels receive its address.
__device__ unsigned g_fp8mm_abort_word = 0u;

struct fp8mm_plan_s {
  fp8mm_desc d;
  int sms = 0;
  int max_smem = 0;
  int swap = 0, bn = 0, splits = 1, kb_per_split = 0, num_kb = 0, stages = 0, num_acc = 2;
  int group = 1, slow = 0, mx = 0, out_es = 4, cg = 1, ew = 8;
  int f4 = 0, vec16 = 0;  // packed FP4 operands; their factors per 16 (E4M3) rather than per 32 (UE8M0)
  int64_t R = 0, Q = 0;
  int tiles_r = 0, tiles_q = 0;
  long long units = 0;
  int grid = 0;
  uint32_t tmem_cols = 0;
  int x_kind = kScaleNone, y_kind = kScaleNone;
  uint32_t off_x = 0, off_y = 0, off_sf = 0, off_out = 0, off_ys = 0, off_bias = 0, off_bar = 0;
  uint32_t x_stage_bytes = 0, y_stage_bytes = 0, sf_stage_bytes = 0;
  size_t smem_bytes = 0;
  size_t ws_partials_bytes = 0, ws_counters_off = 0, ws_counters_bytes = 0, ws_bytes = 0;
  // K-major copies of M/N-major operands (offsets into the workspace), and
  // where the split-K part of the workspace starts
  size_t ws_ta_off = 0, ws_tb_off = 0, ws_split_off = 0;
};

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int out_size(int out_dtype) {
  return out_dtype == FP8MM_OUT_F32 ? 4 : (out_dtype == FP8MM_OUT_E4M3 || out_dtype == FP8MM_OUT_E5M2) ? 1 : 2;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Device address of the abort word, looked up once per device (the current
// device must be `device`).
unsigned* abort_word_address(int device) {
  static std::mutex mu;
  static unsigned* addr[64] = {};
  if (device < 0 || device >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fp8mm_abort_word) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[device] = static_cast<unsigned*>(p);
  }
  return addr[device];
}

// Per-device, per-kernel opt-in to the device's full dynamic shared memory.
cudaError_t ensure_smem_attr(KernelFn fn, int device, size_t bytes) {
  static std::mutex mu;
  static const void* done[64][32] = {};
  std::lock_guard<std::mutex> lk(mu);
  if (device >= 0 && device < 64) {
    for (int i = 0; i < 32; ++i) {
      if (done[device][i] == (const void*)fn) return cudaSuccess;
    }
  }
  cudaError_t e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (device >= 0 && device < 64) {
    for (int i = 0; i < 32; ++i) {
      if (done[device][i] == nullptr) {
        done[device][i] = (const void*)fn;
        break;
      }
    }
  }
  return cudaSuccess;
}

// Shared-memory layout for a given stage count; returns total bytes.
size_t layout(fp8mm_plan_s* P, int stages) {
  const uint32_t x_bytes = kBlockM * kBlockK;
  const uint32_t y_bytes = (uint32_t)(P->bn / P->cg) * kBlockK;
  // FP4: the 4 (per 16) or 2 (per 32) factor atoms of X and of Y per stage
  const uint32_t sf_bytes = P->f4 ? (1u + (uint32_t)P->bn / 128u) * (P->vec16 ? 4u : 2u) * 512u
                                  : (P->mx ? kSfStageBytes : 0u);
  uint32_t off = 0;
  P->x_stage_bytes = x_bytes;
  P->y_stage_bytes = y_bytes;
  P->sf_stage_bytes = sf_bytes;
  P->off_x = off;
  off += x_bytes * stages;
  P->off_y = off;
  off += y_bytes * stages;
  off = (off + 1023u) & ~1023u;
  P->off_sf = off;
  off += sf_bytes * stages;
  off = (off + 1023u) & ~1023u;
  P->off_out = off;
  off += (uint32_t)(P->ew * stage_out_bytes(P->ew, held_tile(P->bn, P->slow != 0, P->mx != 0), P->out_es,
                                             part_max_cols(P->bn, P->ew, P->slow != 0)));
  P->off_ys = off;
  // per-column Y scales of the current chunk, one row per epilogue warp
  if (P->x_kind != kScaleNone && P->y_kind == kScaleRow) off += (uint32_t)(P->ew * part_max_cols(P->bn, P->ew, P->slow != 0) * 4);
  off = (off + 127u) & ~127u;
  P->off_bias = off;
  // the bias of each epilogue warp's columns (fp32), staged once per tile
  if (P->d.bias) off += (uint32_t)(P->ew * part_max_cols(P->bn, P->ew, P->slow != 0) * 4);
  off = (off + 127u) & ~127u;
  P->off_bar = off;
  off += 16u * stages + 80u + 16u;  // full/empty per stage, 4+4 accumulator barriers, epilogue, drain, misc
  off = (off + 127u) & ~127u;
  return (size_t)off + 1024;  // slack for aligning the dynamic base to 1024
}

// Relative mainloop throughput of a single-CTA tile width (measured on
// GB300 with long K: narrower tiles move more bytes per MMA cycle).
double width_efficiency(int bn, bool mx) {
  switch (bn) {
    case 256: return mx ? 0.85 : 1.0;  // the MX form keeps one accumulator at 256 columns
    case 224: return mx ? 0.80 : 0.97;  // MX: factors gathered per stage, fp32 stores beside the mainloop
    case 192: return 0.93;
    default: return 0.6;
  }
}

}  // namespace

namespace {
std::atomic<int> g_withhold_loads{0};  // fp8mm_test_withhold_loads
}  // namespace

extern "C" {

fp8mm_status fp8mm_test_withhold_loads(int enable) {
  g_withhold_loads.store(enable ? 1 : 0);
  return FP8MM_OK;
}

const char* fp8mm_status_string(fp8mm_status s) {
  switch (s) {
    case FP8MM_OK: return "ok";
    case FP8MM_ERR_INVALID: return "invalid argument";
    case FP8MM_ERR_ALIGNMENT: return "misaligned pointer or row (16-byte rule)";
    case FP8MM_ERR_UNSUPPORTED: return "unsupported configuration";
    case FP8MM_ERR_REJECTED: return "rejected combination";
    case FP8MM_ERR_WORKSPACE: return "workspace missing or too small";
    case FP8MM_ERR_CUDA: return "CUDA error";
    case FP8MM_ERR_DEVICE: return "device-side abort";
  }
  return "unknown status";
}

// The planner.  With device_checks it reads the SM count and shared-memory
// limit of desc->device and checks what only the device can answer (the
// held kernels' register count, resident CTA-pair clusters); without, it
// plans for the given `sms` and `max_smem` alone (fp8mm_plan_preview).
static fp8mm_status plan_impl(const fp8mm_desc* desc, int sms, int max_smem, bool device_checks,
                              fp8mm_plan_t** out) {
  if (!desc || !out) return FP8MM_ERR_INVALID;
  *out = nullptr;
  const fp8mm_desc d = *desc;
  if (d.M < 0 || d.N < 0 || d.K < 0 || d.L < 0) return FP8MM_ERR_INVALID;
  if (d.a_fmt < 0 || d.a_fmt > 2 || d.b_fmt < 0 || d.b_fmt > 2) return FP8MM_ERR_INVALID;
  if (d.out_dtype < 0 || d.out_dtype > 4) return FP8MM_ERR_INVALID;
  if (d.bias < 0 || d.bias > 1 || d.a_major < 0 || d.a_major > 1 || d.b_major < 0 || d.b_major > 1)
    return FP8MM_ERR_INVALID;
  if (d.scale_mode < 0 || d.scale_mode > 4) return FP8MM_ERR_INVALID;
  if (d.fast_accum < 0 || d.fast_accum > 1) return FP8MM_ERR_INVALID;
  if (d.splitk < 0 || d.swap_ab < 0 || d.swap_ab > 2 || d.device < 0) return FP8MM_ERR_INVALID;
  if (d.cta_pair < 0 || d.cta_pair > 2) return FP8MM_ERR_INVALID;
  if (d.epi_warps != 0 && d.epi_warps != 8 && d.epi_warps != 16) return FP8MM_ERR_INVALID;
  if (d.stages < 0 || d.stages == 1 || d.stages > 12) return FP8MM_ERR_INVALID;
  if (d.strict_torch < 0 || d.strict_torch > 1) return FP8MM_ERR_INVALID;
  if (d.block_n != 0 && !(d.block_n >= 16 && d.block_n <= 256 && d.block_n % 16 == 0)) return FP8MM_ERR_INVALID;
  const int64_t lim = (int64_t)1 << 31;
  if (d.M >= lim || d.N >= lim || d.K >= lim || d.L >= 65536) return FP8MM_ERR_UNSUPPORTED;
  // Packed FP4 operands (cuDNN "GEMM + Amax (SM100)", Dtypes): A and B both
  // E2M1, with UE8M0 factors per 32 or E4M3 factors per 16 elements of K,
  // K-major, fast accumulation; K a multiple of 64 (one MMA's K, and a whole
  // number of E4M3-factor atoms).
  const bool f4 = d.a_fmt == FP8MM_E2M1 || d.b_fmt == FP8MM_E2M1;
  if (f4) {
    if (d.a_fmt != d.b_fmt) return FP8MM_ERR_UNSUPPORTED;
    if (d.scale_mode != FP8MM_SCALE_MX32_UE8M0 && d.scale_mode != FP8MM_SCALE_NV16_E4M3) return FP8MM_ERR_UNSUPPORTED;
    if (!d.fast_accum || d.a_major || d.b_major || d.cta_pair == 1 || d.strict_torch) return FP8MM_ERR_UNSUPPORTED;
    if (d.block_n != 0 && d.block_n != 128 && d.block_n != 256) return FP8MM_ERR_UNSUPPORTED;
    if (d.K % 64 != 0) return FP8MM_ERR_ALIGNMENT;
  } else if (d.scale_mode == FP8MM_SCALE_NV16_E4M3) {
    return FP8MM_ERR_UNSUPPORTED;  // factors per 16 elements go with FP4 operands only
  }
  if (d.K % 16 != 0) return FP8MM_ERR_ALIGNMENT;
  if ((d.N * out_size(d.out_dtype)) % 16 != 0) return FP8MM_ERR_ALIGNMENT;
  // M/N-major operands: their rows ([K][M] or [K][N] bytes) must be 16-byte multiples
  if ((d.a_major && d.M % 16 != 0) || (d.b_major && d.N % 16 != 0)) return FP8MM_ERR_ALIGNMENT;
  const bool fp8_out = d.out_dtype == FP8MM_OUT_E4M3 || d.out_dtype == FP8MM_OUT_E5M2;
  // the pages define a bias for bf16 / fp16 (and here fp32) outputs only
  if (d.bias && fp8_out) return FP8MM_ERR_UNSUPPORTED;
  const bool mx = d.scale_mode == FP8MM_SCALE_MX32_UE8M0 || d.scale_mode == FP8MM_SCALE_NV16_E4M3;
  if (mx && d.a_fmt != d.b_fmt) return FP8MM_ERR_UNSUPPORTED;
  // torch._scaled_mm refuses E5M2 x E5M2; the library computes it unless the
  // caller asks for torch's refusals.
  if (d.strict_torch && d.a_fmt == FP8MM_E5M2 && d.b_fmt == FP8MM_E5M2) return FP8MM_ERR_REJECTED;
  // ... and E4M3 x E4M3 -> E5M2 (mmaemu "Testing mmaemu", expected error classes)
  if (d.strict_torch && d.a_fmt == FP8MM_E4M3 && d.b_fmt == FP8MM_E4M3 && d.out_dtype == FP8MM_OUT_E5M2)
    return FP8MM_ERR_REJECTED;

  fp8mm_plan_s* P = new (std::nothrow) fp8mm_plan_s();
  if (!P) return FP8MM_ERR_INVALID;
  struct Guard {
    fp8mm_plan_s*& p;
    ~Guard() { delete p; }
  } guard{P};
  P->d = d;
  if (!device_checks) {
    P->sms = sms;
    P->max_smem = max_smem;
  } else if (cudaDeviceGetAttribute(&P->sms, cudaDevAttrMultiProcessorCount, d.device) != cudaSuccess ||
             cudaDeviceGetAttribute(&P->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, d.device) !=
                 cudaSuccess) {
    cudaGetLastError();
    return FP8MM_ERR_CUDA;
  }
  P->mx = mx ? 1 : 0;
  P->f4 = f4 ? 1 : 0;
  P->vec16 = d.scale_mode == FP8MM_SCALE_NV16_E4M3 ? 1 : 0;
  P->out_es = out_size(d.out_dtype);
  const bool blockwise = d.scale_mode == FP8MM_SCALE_A1x128_B1x128 || d.scale_mode == FP8MM_SCALE_A1x128_B128x128;
  P->slow = (blockwise || !d.fast_accum) ? 1 : 0;

  // Swap-AB for skinny M: the long N side then fills the 128-lane MMA M side.
  // (From 129 to 256 rows unswapped 256-row pair tiles, or slow 256-column
  // tiles, measured 13-17% faster on GB300 than swapped ones.)
  bool swap;
  if (d.swap_ab == 1)
    swap = true;
  else if (d.swap_ab == 2)
    swap = false;
  else
    swap = !mx && d.M <= 128 && d.N > d.M;
  P->swap = swap ? 1 : 0;
  P->R = swap ? d.N : d.M;
  P->Q = swap ? d.M : d.N;
  if (blockwise) {
    if (!swap) {
      P->x_kind = kScaleRow;
      P->y_kind = d.scale_mode == FP8MM_SCALE_A1x128_B1x128 ? kScaleRow : kScaleBlock128;
    } else {
      P->x_kind = d.scale_mode == FP8MM_SCALE_A1x128_B1x128 ? kScaleRow : kScaleBlock128;
      P->y_kind = kScaleRow;
    }
  }
  // a stage holds 128 bytes of K per row: 128 FP8 or 256 FP4 elements
  P->num_kb = (int)cdiv(d.K, f4 ? 2 * kBlockK : kBlockK);
  const int64_t L = std::max<int64_t>(1, d.L);
  const int64_t tiles_r1 = std::max<int64_t>(1, cdiv(P->R, kBlockM));

  // Tile width on the MMA's N side.  Wide problems pick the width whose
  // whole waves over the SMs cost least; narrow ones the smallest
  // power-of-two width that covers Q.
  int bn = d.block_n;
  // Two-SM pair tiles (256 rows, cta_group::2): each SM stages half as many
  // Y bytes per MMA, which measured 4-15% faster than single-CTA tiles on
  // GB300 for fast unswapped GEMMs with at least one wave of pairs.
  const int64_t pair_rows = std::max<int64_t>(1, cdiv(P->R, 2 * kBlockM));
  // MX (FP8 operands) pairs: 256-column tiles only, each CTA staging its own
  // rows' factor atom and all of the Y tile's.  Once held tiles stored wider
  // chunks (a whole block per warp for 1- and 2-byte outputs, 16 columns for
  // fp32) they measured faster than one-CTA held tiles on GB300: 4 x 4096^3
  // bf16 out 212 against 224 us, fp32 out 224 against 233 us.
  const bool mx_pairable = mx && !f4 && !P->slow;
  const bool auto_mx_pair = d.cta_pair == 0 && mx_pairable && !swap && d.splitk <= 1 &&
                            (d.block_n == 0 || d.block_n == 256) &&
                            pair_rows * cdiv(P->Q, 256) * L >= (int64_t)(P->sms / 2);
  const bool auto_pair = d.cta_pair == 0 && !mx && !P->slow && !swap && P->Q > 128 &&
                         (d.block_n == 0 || ((d.block_n == 224 || d.block_n == 192) && !mx) || d.block_n == 256) &&
                         pair_rows * cdiv(P->Q, 256) * L >= (int64_t)(P->sms / 2);
  // Slow accumulation on CTA pairs: 256-row held tiles of 192, 224 or 256
  // columns.  Each 128-K chunk is handed from the pair's MMA to both CTAs'
  // epilogues and back; with relaxed cluster-scope arrivals for the hand-back
  // a pair's wave measured about 4% shorter than a one-CTA wave of the same
  // width on GB300 (4096^3: 80.6 vs 82.6 us; 2048x28672x8192: 396 vs 411 us;
  // 8192x7168x2048 with 128x128 scales: 167 vs 179 us), each SM staging a
  // third fewer operand bytes.  A 224-column tile's halves (112 columns per
  // epilogue warp) straddle 128-column scale blocks, so 128x128 Y scales
  // take 256.
  constexpr double kSlowPairWave = 0.96;
  bool slow_pair = false;
  const bool y_block128 = blockwise && P->y_kind == kScaleBlock128;
  if (bn == 0 && auto_mx_pair) bn = 256;
  if (bn == 0 && auto_pair) {
    // the width whose whole waves over the SM pairs cost least
    double best = 1e300;
    for (int c : {256, 224, 192}) {
      if (mx && c != 256) continue;
      const int64_t tiles = pair_rows * cdiv(P->Q, c) * L;
      const double cost = (double)cdiv(tiles, P->sms / 2) * c / width_efficiency(c, false);
      if (cost < best * 0.999) {
        best = cost;
        bn = c;
      }
    }
  }
  if (bn == 0) {
    const int64_t q16 = std::max<int64_t>(16, cdiv(P->Q, 16) * 16);
    int pw = 16;
    while (pw < q16 && pw < 256) pw *= 2;
    if (mx && pw < 128) pw = 128;
    bn = pw;
    if (swap) {
      // Skinny problems stream X (the long operand) from HBM once; the whole
      // of Y fits one tile and split-K fills the waves.
    } else if (P->slow && P->Q > 128) {
      // Slow accumulation: held tiles of 192-256 columns (never split) when
      // they fill the SMs, else 128 (split-K can fill the waves).  A held
      // chunk's time follows its operand bytes (128 rows of X and BN of Y,
      // 128 bytes of K each), so the width with the fewest whole waves x
      // bytes per chunk wins; 128x128 Y scales need 128-aligned halves (256).
      // Pair tiles compete with one-CTA tiles by the same measure, a pair's
      // wave counted at kSlowPairWave of a one-CTA wave.  A 224-column held
      // tile stores its 112 columns per warp in 16-column chunks (the others
      // in 64 or 32): its waves count 12% longer, as measured on GB300
      // (4096^3 slow on pairs: 256 x 224 79.6 us against 256 x 256 75.4 us,
      // both four waves).
      constexpr double kHeld224Wave = 1.12;
      bn = 128;
      if (!mx && d.splitk <= 1 && tiles_r1 * cdiv(P->Q, 256) * L >= (int64_t)P->sms) {
        double best = 1e300;
        for (int c : {256, 224, 192}) {
          if (c != 256 && y_block128) continue;
          const int64_t tiles = tiles_r1 * cdiv(P->Q, c) * L;
          const double wide_cost = (kBlockM + c) * (c == 224 ? kHeld224Wave : 1.0);
          const double cost = (double)cdiv(tiles, P->sms) * wide_cost;
          if (cost < best * 0.999) {
            best = cost;
            bn = c;
            slow_pair = false;
          }
          if (d.cta_pair != 0) continue;
          const int64_t ptiles = pair_rows * cdiv(P->Q, c) * L;
          const double pcost = (double)cdiv(ptiles, P->sms / 2) * wide_cost * kSlowPairWave;
          if (pcost < best * 0.999) {
            best = pcost;
            bn = c;
            slow_pair = true;
          }
        }
      }
    } else if (!P->slow && P->Q > 128 && tiles_r1 * cdiv(P->Q, 256) * L > (int64_t)P->sms) {
      // (under one wave of 256-wide tiles the widest tile is the fastest)
      double best = 1e300;
      for (int c : {256, 224, 192, 128}) {
        if (mx && c == 192) continue;
        if (f4 && c == 224) continue;  // FP4 tiles are 128 or 256 columns
        const int64_t tiles = tiles_r1 * cdiv(P->Q, c) * L;
        const double cost = (double)cdiv(tiles, P->sms) * c / width_efficiency(c, mx);
        if (cost < best * 0.999) {
          best = cost;
          bn = c;
        }
      }
    }
  }
  // Slow accumulation keeps the promoted sums in registers: 192, 224 or 256
  // columns, on one CTA or a CTA pair, never swapped, split or MX; 192/224
  // only where no 128x128 Y-scale block straddles a half.
  const bool pair = d.cta_pair == 1 || auto_pair || slow_pair || auto_mx_pair;
  const bool slow_wide_ok = !swap && !mx && d.splitk <= 1 &&
                            (bn == 256 || ((bn == 224 || bn == 192) && !y_block128));
  if (P->slow && bn > 128 && !slow_wide_ok) {
    if (d.block_n != 0) return FP8MM_ERR_UNSUPPORTED;
    bn = 128;
  }
  // (a requested split needs the narrower MX tile: 256-column ones are held)
  if (mx && !P->slow && bn == 256 && d.block_n == 0 && d.splitk > 1) bn = 128;
  // MX tiles are 128 or 256 columns, or 224: the block-scaled MMA reads its
  // factors from a TMEM column aligned to an atom's four columns, so the
  // 224-column kernel gathers Y's factor atoms to start at the tile's first row.
  if (mx && bn != 128 && bn != 224 && bn != 256) return FP8MM_ERR_UNSUPPORTED;
  if (f4 && bn != 128 && bn != 256) return FP8MM_ERR_UNSUPPORTED;
  // FP8 outputs are stored in rows of at least 16 bytes that start on 16-byte
  // columns: unswapped tiles of 16 columns (8 per epilogue warp) are too narrow.
  if (fp8_out && !swap && bn < 32) {
    if (d.block_n != 0) return FP8MM_ERR_UNSUPPORTED;
    bn = 32;
  }
  P->bn = bn;

  if (pair) {
    if ((mx && !(mx_pairable && bn == 256)) || swap) return FP8MM_ERR_UNSUPPORTED;
    P->cg = 2;
  }
  // Epilogue warps: 16 for slow accumulation at 128 columns (more TMEM loads
  // in flight during the per-chunk promotion), else 8.
  const bool wide = wide_slow(bn, P->slow != 0);
  const bool wide_ycol = wide && blockwise && P->y_kind == kScaleRow;
  P->ew = d.epi_warps ? d.epi_warps : ((P->slow && !mx && bn == 128 && P->cg == 1) ? 16 : 8);
  KernelFn fn = select_kernel(P->bn, P->slow != 0, P->mx != 0, P->cg, P->ew, f4);
  if (!fn) return FP8MM_ERR_UNSUPPORTED;
  if (device_checks && held_tile(bn, P->slow != 0, mx)) {
    // The warpgroup register split only redistributes what the block was
    // launched with; refuse the plan if the compiled kernel holds fewer
    // registers per thread than the split hands out (its raise would wait
    // forever).
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, (const void*)fn) != cudaSuccess) {
      cudaGetLastError();
      return FP8MM_ERR_CUDA;
    }
    if (fa.numRegs * (P->ew + 4) < P->ew * epi_regs(P->ew) + 4 * kRegRoles) return FP8MM_ERR_UNSUPPORTED;
  }

  const int64_t tiles_r = std::max<int64_t>(1, cdiv(P->R, (int64_t)kBlockM * P->cg));
  const int64_t tiles_q = std::max<int64_t>(1, cdiv(P->Q, bn));
  P->tiles_r = (int)tiles_r;
  P->tiles_q = (int)tiles_q;
  const int64_t tiles = tiles_r * tiles_q * L;  // pair tiles when cg == 2

  // Split-K: contiguous 128-aligned K ranges.  Chosen to fill whole waves of
  // SMs when there are fewer than two waves of tiles and the partial tiles
  // are small next to the operand bytes they save.
  int S = d.splitk;
  const int64_t slots = P->sms / P->cg;  // concurrent work units (CTAs or CTA pairs)
  const bool held = held_tile(bn, P->slow != 0, mx);
  if (held && S > 1) return FP8MM_ERR_UNSUPPORTED;  // held tiles are never split
  if (S == 0) {
    S = 1;
    if (!held && tiles < 2 * slots && P->num_kb >= 8) {
      double best = (double)tiles / (double)(cdiv(tiles, slots) * slots);
      for (int sk = 2; sk <= 8; ++sk) {
        if (P->num_kb / sk < 4) break;
        if (bn > 128 && sk > 2) break;
        const int64_t u = tiles * sk;
        const double eff = (double)u / (double)(cdiv(u, slots) * slots);
        if (eff > best + 0.05) {
          best = eff;
          S = sk;
        }
      }
    }
  }
  S = std::max(1, std::min(S, std::max(1, P->num_kb)));
  P->kb_per_split = P->num_kb > 0 ? (int)cdiv(P->num_kb, S) : 0;
  P->splits = P->num_kb > 0 ? (int)cdiv(P->num_kb, P->kb_per_split) : 1;
  P->units = (long long)tiles * P->splits;
  P->grid = (int)std::min<long long>(P->units * P->cg, P->sms / P->cg * P->cg);
  // Grouped raster: consecutive work units walk a group of tile rows of one
  // tile column before moving to the next column, so a Y tile is read by the
  // group's CTAs while it is in L2: 8 one-CTA tile rows, 16 pair tile rows
  // (4096 rows; on GB300 the pair shapes of 1024-8192 x 28672 x 8192 ran
  // about 1% faster with 16 than with 8, 2-4% slower with 4 or 32).  (Groups
  // sized to keep all of X in L2 cut the DRAM re-reads of Y on the largest
  // shapes 4-8x but measured 2-5% slower.)
  P->group = swap ? 1 : (P->cg == 2 ? 16 : 8);

  // Pipeline depth: as many stages as fit in shared memory (at most 12).  The
  // MX form also keeps a 16-column TMEM slot per stage for its factors, next
  // to two accumulators when they fit in 512 columns (else one).
  // (Streaming skinny shapes measured best at 6-8 stages on GB300.)
  int stages = swap ? 8 : 12;
  while (stages > 2 && layout(P, stages) > (size_t)P->max_smem) --stages;
  if (d.stages > 0) {
    if (d.stages > stages) return FP8MM_ERR_UNSUPPORTED;
    stages = d.stages;
  } else if (wide && blockwise) {
    // Block-scaled slow 256-column tiles keep a shallow ring: the shared
    // memory left over becomes L1 for their per-chunk scale loads, which
    // measured faster on GB300 than a deeper ring (3 stages, 2 with
    // per-column scales).
    stages = std::min(stages, wide_ycol ? 2 : 3);
  }
  // Slow accumulation hands each 128-K chunk to the epilogue: with 128-column
  // tiles four chunk buffers fill the 512 TMEM columns and let the MMA run up
  // to three chunks ahead of the promotion.
  P->num_acc = (P->slow && !mx && 4 * bn <= 512) ? 4 : 2;
  // TMEM columns of one stage's factors (block-scaled forms)
  const uint32_t sf_cols = f4 ? 4u * (P->vec16 ? 4u : 2u) * (1u + (uint32_t)bn / 128u) : 16u;
  if (mx) {
    const int tmem_stages = (512 - 2 * bn) / (int)sf_cols;
    if (tmem_stages >= 3) {
      stages = std::min(stages, tmem_stages);
    } else {
      P->num_acc = 1;
      stages = std::min(stages, (512 - bn) / (int)sf_cols);
    }
  } else if (2 * bn > 512) {
    P->num_acc = 1;
  }
  P->stages = stages;
  P->smem_bytes = layout(P, stages);
  if (P->smem_bytes > (size_t)P->max_smem) return FP8MM_ERR_UNSUPPORTED;
  const uint32_t need = (uint32_t)(P->num_acc * bn) + (mx ? sf_cols * (uint32_t)stages : 0u);
  uint32_t cols = 32;
  while (cols < need) cols *= 2;
  if (cols > 512) return FP8MM_ERR_UNSUPPORTED;
  P->tmem_cols = cols;

  if (P->cg == 2 && !device_checks) {
    P->grid = 2 * (int)std::min<long long>(P->units, P->sms / 2);  // (one pair per two SMs)
  } else if (P->cg == 2) {
    // Persistent grid: as many CTA pairs as can be resident at once.
    int nclusters = 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)P->grid);
    cfg.blockDim = dim3(kernel_threads(P->ew, held_tile(P->bn, P->slow != 0, P->mx != 0)));
    cfg.dynamicSmemBytes = P->smem_bytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (ensure_smem_attr(fn, d.device, (size_t)P->max_smem) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&nclusters, (const void*)fn, &cfg) != cudaSuccess || nclusters < 1) {
      cudaGetLastError();
      return FP8MM_ERR_CUDA;
    }
    P->grid = 2 * (int)std::min<long long>(P->units, nclusters);
  }
  // Workspace: K-major copies of M/N-major operands first, then the split-K
  // partial tiles and their arrival counters.
  size_t ws = 0;
  if (d.a_major) {
    P->ws_ta_off = ws;
    ws += round256((size_t)L * d.M * d.K);
  }
  if (d.b_major) {
    P->ws_tb_off = ws;
    ws += round256((size_t)L * d.N * d.K);
  }
  P->ws_split_off = ws;
  if (P->splits > 1) {
    P->ws_partials_bytes = (size_t)tiles * P->cg * P->splits * kBlockM * bn * sizeof(float);
    P->ws_counters_off = ws + round256(P->ws_partials_bytes);
    P->ws_counters_bytes = (size_t)tiles * P->cg * sizeof(unsigned);
    ws = P->ws_counters_off + round256(P->ws_counters_bytes);
  }
  P->ws_bytes = ws;
  *out = P;
  P = nullptr;  // ownership passes to the caller
  return FP8MM_OK;
}

fp8mm_status fp8mm_plan(const fp8mm_desc* desc, fp8mm_plan_t** out) {
  return plan_impl(desc, 0, 0, true, out);
}

fp8mm_status fp8mm_plan_preview(const fp8mm_desc* desc, int32_t sms, int32_t max_smem_bytes,
                                fp8mm_plan_info* info) {
  if (!info || sms < 2 || max_smem_bytes <= 0) return FP8MM_ERR_INVALID;
  fp8mm_plan_t* P = nullptr;
  const fp8mm_status st = plan_impl(desc, sms, max_smem_bytes, false, &P);
  if (st != FP8MM_OK) return st;
  const fp8mm_status st2 = fp8mm_plan_get_info(P, info);
  delete P;
  return st2;
}

fp8mm_status fp8mm_workspace_size(const fp8mm_plan_t* plan, size_t* bytes) {
  if (!plan || !bytes) return FP8MM_ERR_INVALID;
  *bytes = plan->ws_bytes;
  return FP8MM_OK;
}

fp8mm_status fp8mm_plan_roofline(const fp8mm_plan_t* plan, double* flops, double* bytes) {
  if (!plan || !flops || !bytes) return FP8MM_ERR_INVALID;
  const fp8mm_desc& d = plan->d;
  const double L = (double)d.L, M = (double)d.M, N = (double)d.N, K = (double)d.K;
  const double kb = (double)cdiv(d.K, 128);
  double sbytes = 8.0;
  switch (d.scale_mode) {
    case FP8MM_SCALE_A1x128_B1x128: sbytes = 4.0 * L * (M + N) * kb; break;
    case FP8MM_SCALE_A1x128_B128x128: sbytes = 4.0 * L * (M + (double)cdiv(d.N, 128)) * kb; break;
    case FP8MM_SCALE_MX32_UE8M0:
    case FP8MM_SCALE_NV16_E4M3: {
      // one 512-byte atom per 128 rows and 4 factors along K
      const double atoms_k = (double)cdiv(d.K, 4 * (d.scale_mode == FP8MM_SCALE_NV16_E4M3 ? 16 : 32));
      sbytes = 512.0 * L * atoms_k * (double)(cdiv(d.M, 128) + cdiv(d.N, 128));
      break;
    }
    default: break;
  }
  const double opb = plan->f4 ? 0.5 : 1.0;  // operand bytes per element
  *flops = 2.0 * L * M * N * K;
  *bytes = opb * L * (M * K + N * K) + sbytes + (d.bias ? N * (double)plan->out_es : 0.0) +
           L * M * N * (double)plan->out_es + 4.0;
  return FP8MM_OK;
}

fp8mm_status fp8mm_plan_get_info(const fp8mm_plan_t* plan, fp8mm_plan_info* info) {
  if (!plan || !info) return FP8MM_ERR_INVALID;
  info->swap_ab = plan->swap;
  info->block_m = kBlockM;
  info->block_n = plan->bn;
  info->splitk = plan->splits;
  info->stages = plan->stages;
  info->grid = plan->grid;
  info->units = plan->units;
  info->slow = plan->slow;
  info->smem_bytes = (int32_t)plan->smem_bytes;
  info->cta_pair = plan->cg == 2 ? 1 : 0;
  info->epi_warps = plan->ew;
  return FP8MM_OK;
}

fp8mm_status fp8mm_plan_kernel_launches(const fp8mm_plan_t* plan, int32_t* launches) {
  if (!plan || !launches) return FP8MM_ERR_INVALID;
  const fp8mm_desc& d = plan->d;
  if (d.M == 0 || d.N == 0 || d.L == 0)
    *launches = 0;
  else if (d.K == 0)
    *launches = d.bias ? 1 : 0;  // the bias rows (C = 0 is a memset)
  else
    *launches = 1 + d.a_major + d.b_major;  // the K-major copies, then the GEMM
  return FP8MM_OK;
}

void fp8mm_destroy(fp8mm_plan_t* plan) { delete plan; }

fp8mm_status fp8mm_device_error(int device, uint32_t* code, int clear) {
  if (!code || device < 0) return FP8MM_ERR_INVALID;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return FP8MM_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return FP8MM_ERR_CUDA;
  fp8mm_status st = FP8MM_OK;
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(&v, g_fp8mm_abort_word, sizeof(v)) != cudaSuccess)
    st = FP8MM_ERR_CUDA;
  if (st == FP8MM_OK && clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_fp8mm_abort_word, &zero, sizeof(zero)) != cudaSuccess) st = FP8MM_ERR_CUDA;
  }
  *code = v;
  if (prev != device) cudaSetDevice(prev);
  return st;
}

fp8mm_status fp8mm_run(fp8mm_plan_t* P, const void* a, const void* b, const void* scale_a, const void* scale_b,
                       void* c, float* amax, void* workspace, size_t workspace_bytes, void* stream_) {
  return fp8mm_run_ex(P, a, b, scale_a, scale_b, nullptr, nullptr, c, amax, workspace, workspace_bytes, stream_);
}

fp8mm_status fp8mm_run_ex(fp8mm_plan_t* P, const void* a, const void* b, const void* scale_a, const void* scale_b,
                          const float* scale_result, const void* bias, void* c, float* amax, void* workspace,
                          size_t workspace_bytes, void* stream_) {
  if (!P || !amax) return FP8MM_ERR_INVALID;
  const fp8mm_desc& d = P->d;
  const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool empty = d.M == 0 || d.N == 0 || d.L == 0;
  // a bias exactly when the plan was made for one
  if ((bias != nullptr) != (d.bias != 0)) return FP8MM_ERR_INVALID;
  if (bias && !aligned(bias, (uintptr_t)P->out_es)) return FP8MM_ERR_ALIGNMENT;
  if (scale_result && !aligned(scale_result, 4)) return FP8MM_ERR_ALIGNMENT;
  if (!empty) {
    if (!c) return FP8MM_ERR_INVALID;
    if (d.K > 0 && (!a || !b || !scale_a || !scale_b)) return FP8MM_ERR_INVALID;
    if (!aligned(c, 16)) return FP8MM_ERR_ALIGNMENT;
    if (d.K > 0) {
      if (!aligned(a, 16) || !aligned(b, 16)) return FP8MM_ERR_ALIGNMENT;
      const uintptr_t sal = P->mx ? 16 : 4;
      if (!aligned(scale_a, sal) || !aligned(scale_b, sal)) return FP8MM_ERR_ALIGNMENT;
    }
  }
  if (!aligned(amax, 4)) return FP8MM_ERR_ALIGNMENT;
  if (P->ws_bytes > 0 && !empty && d.K > 0) {
    if (!workspace || workspace_bytes < P->ws_bytes) return FP8MM_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return FP8MM_ERR_ALIGNMENT;
  }

  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return FP8MM_ERR_CUDA;
  if (prev != d.device && cudaSetDevice(d.device) != cudaSuccess) return FP8MM_ERR_CUDA;
  struct Restore {
    int prev, dev;
    ~Restore() {
      if (prev != dev) cudaSetDevice(prev);
    }
  } restore{prev, d.device};

  if (cudaMemsetAsync(amax, 0, sizeof(float), stream) != cudaSuccess) return FP8MM_ERR_CUDA;
  if (empty) return FP8MM_OK;
  if (d.K == 0) {
    // An empty sum over K: every element of C is +0, plus the bias if any.
    if (bias)
      return launch_bias_rows(bias, c, (long long)d.L * d.M, (int)d.N, P->out_es, d.out_dtype == FP8MM_OUT_BF16,
                              reinterpret_cast<unsigned*>(amax), P->sms, stream) == cudaSuccess
                 ? FP8MM_OK
                 : FP8MM_ERR_CUDA;
    const size_t bytes = (size_t)d.L * d.M * d.N * P->out_es;
    return cudaMemsetAsync(c, 0, bytes, stream) == cudaSuccess ? FP8MM_OK : FP8MM_ERR_CUDA;
  }
  // M/N-major operands: copy them into K-major workspace, then read the copies.
  if (d.a_major) {
    void* ta = static_cast<uint8_t*>(workspace) + P->ws_ta_off;
    if (launch_transpose_to_kmajor(a, ta, (int)d.L, (int)d.K, (int)d.M, P->sms, stream) != cudaSuccess)
      return FP8MM_ERR_CUDA;
    a = ta;
  }
  if (d.b_major) {
    void* tb = static_cast<uint8_t*>(workspace) + P->ws_tb_off;
    if (launch_transpose_to_kmajor(b, tb, (int)d.L, (int)d.K, (int)d.N, P->sms, stream) != cudaSuccess)
      return FP8MM_ERR_CUDA;
    b = tb;
  }

  EncodeTiledFn enc = encode_fn();
  if (!enc) return FP8MM_ERR_CUDA;
  const void* xptr = P->swap ? b : a;
  const void* yptr = P->swap ? a : b;
  CUtensorMap tm_x, tm_y, tm_c, tm_sfx, tm_sfy;
  std::memset(&tm_sfx, 0, sizeof(tm_sfx));
  std::memset(&tm_sfy, 0, sizeof(tm_sfy));
  const int64_t kbytes = P->f4 ? d.K / 2 : d.K;  // bytes of K per operand row (FP4: two elements per byte)
  {
    cuuint64_t dims[3] = {(cuuint64_t)kbytes, (cuuint64_t)P->R, (cuuint64_t)d.L};
    cuuint64_t strides[2] = {(cuuint64_t)kbytes, (cuuint64_t)(kbytes * P->R)};
    cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)kBlockM, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(xptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FP8MM_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)kbytes, (cuuint64_t)P->Q, (cuuint64_t)d.L};
    cuuint64_t strides[2] = {(cuuint64_t)kbytes, (cuuint64_t)(kbytes * P->Q)};
    cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)(P->bn / P->cg), 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm_y, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(yptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FP8MM_ERR_CUDA;
  }
  // One TMA store per warp covers 32 tile rows x `cw` tile columns, staged in
  // shared memory with the swizzle that matches its row length.
  const int cw = chunk_cols(P->bn, P->out_es, P->ew, held_tile(P->bn, P->slow != 0, P->mx != 0), P->slow != 0);
  uint32_t rowbytes;
  cuuint32_t cbox[3];
  if (!P->swap) {
    rowbytes = (uint32_t)(cw * P->out_es);
    cbox[0] = (cuuint32_t)cw;
    cbox[1] = 32;
  } else {
    rowbytes = (uint32_t)(32 * P->out_es);
    cbox[0] = 32;
    cbox[1] = (cuuint32_t)cw;
  }
  cbox[2] = 1;
  CUtensorMapSwizzle cswz;
  uint32_t swz_mask;
  switch (rowbytes) {
    case 128: cswz = CU_TENSOR_MAP_SWIZZLE_128B; swz_mask = 7; break;
    case 64: cswz = CU_TENSOR_MAP_SWIZZLE_64B; swz_mask = 3; break;
    case 32: cswz = CU_TENSOR_MAP_SWIZZLE_32B; swz_mask = 1; break;
    default: cswz = CU_TENSOR_MAP_SWIZZLE_NONE; swz_mask = 0; break;
  }
  {
    const CUtensorMapDataType dt = d.out_dtype == FP8MM_OUT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : d.out_dtype == FP8MM_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : d.out_dtype == FP8MM_OUT_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[3] = {(cuuint64_t)d.N, (cuuint64_t)d.M, (cuuint64_t)d.L};
    cuuint64_t strides[2] = {(cuuint64_t)(d.N * P->out_es), (cuuint64_t)(d.N * d.M * P->out_es)};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm_c, dt, 3, c, dims, strides, cbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE, cswz,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FP8MM_ERR_CUDA;
  }

  KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.R = (int)P->R;
  kp.Q = (int)P->Q;
  kp.K = (int)d.K;
  kp.L = (int)d.L;
  kp.num_kb = P->num_kb;
  kp.kb_per_split = P->kb_per_split;
  kp.splits = P->splits;
  kp.tiles_r = P->tiles_r;
  kp.tiles_q = P->tiles_q;
  kp.group = P->group;
  kp.units = P->units;
  kp.swap = P->swap;
  kp.withhold_loads = g_withhold_loads.load() ? 1 : 0;
  kp.out_dtype = d.out_dtype;
  kp.out_es = P->out_es;
  kp.scale_result = scale_result;
  kp.bias = bias;
  kp.stages = P->stages;
  kp.num_acc = P->num_acc;
  kp.tmem_cols = P->tmem_cols;
  const uint32_t xf = (uint32_t)(P->swap ? d.b_fmt : d.a_fmt);
  const uint32_t yf = (uint32_t)(P->swap ? d.a_fmt : d.b_fmt);
  if (P->f4) {
    // kind::mxf4nvf4: E2M1 operands (format code 1 at bits 7-9 and 10-12), N>>3 at 17, scale type
    // at bit 23 (1 UE8M0 factors per 32 elements, 0 E4M3 factors per 16), M>>4 at 24; the
    // scale-factor ids of the 2X form are added per MMA in the kernel.
    kp.idesc = (1u << 7) | (1u << 10) | ((uint32_t)(P->bn >> 3) << 17) | ((P->vec16 ? 0u : 1u) << 23) |
               ((uint32_t)(kBlockM >> 4) << 24);
  } else if (P->mx) {
    // kind::mxf8f6f4: B scale id bits 4-5, formats 7-9 / 10-12, N>>3 at 17, UE8M0 scale type bit 23,
    // M>>4 at 24, A scale id bits 29-30 (ids added per K step in the kernel).
    kp.idesc = (xf << 7) | (yf << 10) | ((uint32_t)(P->bn >> 3) << 17) | (1u << 23) |
               ((uint32_t)((kBlockM * P->cg) >> 4) << 24);
  } else {
    // kind::f8f6f4: fp32 accumulator (bits 4-5 = 1), formats, K-major A and B, N>>3 at 17, M>>4 at 24.
    kp.idesc = (1u << 4) | (xf << 7) | (yf << 10) | ((uint32_t)(P->bn >> 3) << 17) |
               ((uint32_t)((kBlockM * P->cg) >> 4) << 24);
  }
  if (d.scale_mode == FP8MM_SCALE_TENSOR) {
    kp.sa_tensor = static_cast<const float*>(scale_a);
    kp.sb_tensor = static_cast<const float*>(scale_b);
  } else if (P->mx) {
    kp.sfx = static_cast<const uint8_t*>(P->swap ? scale_b : scale_a);
    kp.sfy = static_cast<const uint8_t*>(P->swap ? scale_a : scale_b);
  } else {
    kp.x_scale = static_cast<const float*>(P->swap ? scale_b : scale_a);
    kp.y_scale = static_cast<const float*>(P->swap ? scale_a : scale_b);
    kp.x_kind = P->x_kind;
    kp.y_kind = P->y_kind;
  }
  kp.scale_kb = P->f4 ? (int)cdiv(d.K, 4 * (P->vec16 ? 16 : 32)) : P->num_kb;
  kp.f4_vec16 = P->vec16;
  kp.sfx_mb = (int)cdiv(P->R, 128);
  kp.sfy_mb = (int)cdiv(P->Q, 128);
  kp.amax_bits = reinterpret_cast<unsigned*>(amax);
  kp.abort_word = abort_word_address(d.device);
  if (!kp.abort_word) return FP8MM_ERR_CUDA;
  if (P->splits > 1) {
    kp.ws_partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + P->ws_split_off);
    kp.ws_counters = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + P->ws_counters_off);
    if (cudaMemsetAsync(kp.ws_counters, 0, P->ws_counters_bytes, stream) != cudaSuccess) return FP8MM_ERR_CUDA;
  }
  kp.off_x = P->off_x;
  kp.off_y = P->off_y;
  kp.off_sf = P->off_sf;
  kp.off_out = P->off_out;
  kp.off_ys = P->off_ys;
  kp.off_bias = P->off_bias;
  kp.off_bar = P->off_bar;
  kp.x_stage_bytes = P->x_stage_bytes;
  kp.y_stage_bytes = P->y_stage_bytes;
  kp.sf_stage_bytes = P->sf_stage_bytes;
  kp.out_swz_mask = swz_mask;
  kp.out_rowbytes = rowbytes;

  KernelFn fn = select_kernel(P->bn, P->slow != 0, P->mx != 0, P->cg, P->ew, P->f4 != 0);
  if (!fn) return FP8MM_ERR_UNSUPPORTED;
  if (ensure_smem_attr(fn, d.device, (size_t)P->max_smem) != cudaSuccess) return FP8MM_ERR_CUDA;
  if (P->mx && !P->f4 && P->cg == 2) {
    // The factor atoms as a [atoms][2][256] byte tensor: one 512-byte box per
    // atom, loaded by the pair form of the TMA so that both CTAs' copies
    // complete on the leader's barrier.
    const void* sfx_ptr = P->swap ? scale_b : scale_a;
    const void* sfy_ptr = P->swap ? scale_a : scale_b;
    const int64_t kbn = P->num_kb;
    const int64_t natoms[2] = {(int64_t)d.L * cdiv(P->R, 128) * kbn, (int64_t)d.L * cdiv(P->Q, 128) * kbn};
    const void* ptrs[2] = {sfx_ptr, sfy_ptr};
    CUtensorMap* maps[2] = {&tm_sfx, &tm_sfy};
    for (int i = 0; i < 2; ++i) {
      cuuint64_t dims[3] = {256, 2, (cuuint64_t)natoms[i]};
      cuuint64_t strides[2] = {256, 512};
      cuuint32_t box[3] = {256, 2, 1};
      cuuint32_t es[3] = {1, 1, 1};
      if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptrs[i]), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return FP8MM_ERR_CUDA;
    }
  }
  void* args[6] = {&tm_x, &tm_y, &tm_c, &tm_sfx, &tm_sfy, &kp};
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P->cg;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)P->grid);
  cfg.blockDim = dim3(kernel_threads(P->ew, held_tile(P->bn, P->slow != 0, P->mx != 0)));
  cfg.dynamicSmemBytes = P->smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = P->cg == 2 ? 1 : 0;
  if (cudaLaunchKernelExC(&cfg, (const void*)fn, args) != cudaSuccess) return FP8MM_ERR_CUDA;
  return FP8MM_OK;
}

// ---------------------------------------------------------------------------
// Entry point for callers that may not allocate device memory.
//
// Split-K plans need scratch memory for their partial tiles and arrival
// counters.  fp8mm_run takes it from the caller; fp8mm_run_static_workspace
// instead uses this file-scope array, which every GPU that loads the library
// holds until the process exits.  Host code only sees a stand-in for the
// array's name, so its device address is looked up per device with
// cudaGetSymbolAddress, once, with that device current.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_fp8mm_static_workspace[FP8MM_STATIC_WORKSPACE_BYTES];

static fp8mm_status static_workspace_address(int device, void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  if (device < 0 || device >= 64) return FP8MM_ERR_INVALID;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fp8mm_static_workspace);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FP8MM_ERR_CUDA;
    }
    addr[device] = p;
  }
  *out = addr[device];
  return FP8MM_OK;
}

fp8mm_status fp8mm_run_static_workspace(fp8mm_plan_t* plan, const void* a, const void* b, const void* scale_a,
                                        const void* scale_b, void* c, float* amax, void* stream) {
  if (!plan) return FP8MM_ERR_INVALID;
  if (plan->ws_bytes > (size_t)FP8MM_STATIC_WORKSPACE_BYTES) return FP8MM_ERR_WORKSPACE;
  void* ws = nullptr;
  if (plan->ws_bytes > 0) {
    const int dev = plan->d.device;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return FP8MM_ERR_CUDA;
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return FP8MM_ERR_CUDA;
    const fp8mm_status st = static_workspace_address(dev, &ws);
    if (prev != dev) cudaSetDevice(prev);
    if (st != FP8MM_OK) return st;
  }
  // fp8mm_run zeroes the arrival counters on the stream before the kernel, and
  // every partial tile is written before it is read, so leftovers of an earlier
  // call never leak into this one.
  return fp8mm_run(plan, a, b, scale_a, scale_b, c, amax, ws, plan->ws_bytes, stream);
}

fp8mm_status fp8mm_gemm(const fp8mm_desc* desc, const void* a, const void* b, const void* scale_a,
                        const void* scale_b, void* c, float* amax, void* workspace, size_t workspace_bytes,
                        void* stream) {
  fp8mm_plan_t* plan = nullptr;
  fp8mm_status st = fp8mm_plan(desc, &plan);
  if (st != FP8MM_OK) return st;
  st = fp8mm_run(plan, a, b, scale_a, scale_b, c, amax, workspace, workspace_bytes, stream);
  fp8mm_destroy(plan);
  return st;
}

}  // extern "C"
