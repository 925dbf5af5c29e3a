/*
 * fp8mm.h -- C ABI of the GB300 (sm_103a) FP8 scaled matrix multiply with a
 * fused global amax.
 *
 *   C[l,m,n] = out_dtype( sum_c S_A(l,m,c) * S_B(l,n,c) * sum_{k in chunk c} A[l,m,k] * B[l,n,k] )
 *   amax     = max over l, m, n of |C[l,m,n]|        (taken over the stored C)
 *
 * Sources of the operation:
 *   - mmaemu "API reference (v0.1)", mmaemu.scaled_mm: torch._scaled_mm
 *     semantics -- FP8 operands, one-element fp32 scales that multiply the
 *     result, out_dtype, fast accumulation (one chain over K) or slow
 *     accumulation (128-element chunks), prior contents of the output never
 *     matter.
 *   - TileOPs "Linear Algebra Operators", GemmFP8FwdOp: a is [M x K], b is
 *     [N x K]; scales per tensor, per 1x128 block along K ([M x ceil(K/128)]),
 *     or for b per 128x128 block ([ceil(N/128) x ceil(K/128)]).
 *   - cuDNN "GEMM + Amax (SM100)", Shapes / Equations / Using JAX arrays:
 *     A (M,K,L) and B (N,K,L) K-major, scale factors per sf_vec_size = 32
 *     elements along K in the atom layout, C (M,N,L) N-major, Amax (1,1,1)
 *     fp32 = max |C|; A, B, C 16-byte aligned along the contiguous dimension;
 *     A and B of the same dtype for the block-scaled form.
 *
 *   - TileOPs "Linear Algebra Operators", GemmFP8FwdOp: an optional bias [N]
 *     in out_dtype, d = (a s_a) @ (b s_b)^T + bias; GemmFwdOp's layout table
 *     (NT, NN, TN, TT); BmmFP8FwdOp: a b that is not K-innermost is copied
 *     into a K-major buffer first (one extra read and write of it).
 *   - mmaemu "API reference (v0.1)", mmaemu.scaled_mm: out_dtype may also be
 *     float8_e4m3fn or float8_e5m2, and scale_result (one fp32) is used only
 *     for those FP8 outputs.
 *
 * Memory layout (all row-major, batch outermost):
 *   a        [L][M][K] FP8 codes (1 byte each), K contiguous (a_major = 0), or
 *            [L][K][M], M contiguous (a_major = 1: the "T" of TN / TT).
 *   b        [L][N][K] FP8 codes, K contiguous (b_major = 0), or [L][K][N], N
 *            contiguous (b_major = 1: the "N" of NN / TN).
 *   c        [L][M][N] of out_dtype, N contiguous.
 *   amax     one fp32.
 *   bias     [N] of out_dtype (fp32, bf16 or fp16 outputs only), when desc.bias = 1.
 *   scale_result  one fp32 (FP8 outputs; NULL means 1).
 *   scale_a / scale_b, by scale_mode:
 *     FP8MM_SCALE_TENSOR           one fp32 each.
 *     FP8MM_SCALE_A1x128_B1x128    fp32 [L][M][ceil(K/128)] and [L][N][ceil(K/128)].
 *     FP8MM_SCALE_A1x128_B128x128  fp32 [L][M][ceil(K/128)] and [L][ceil(N/128)][ceil(K/128)].
 *     FP8MM_SCALE_MX32_UE8M0       UE8M0 bytes (code e means 2^(e-127), 0xFF is NaN),
 *                                  [L][ceil(rows/128)][ceil(K/128)][32][4][4]: within one
 *                                  512-byte atom, byte i32*16 + i4*4 + j4 scales row
 *                                  i32 + 32*i4 of the 128-row block and the 32-element
 *                                  K block j4 of the 128-element K block.
 *     FP8MM_SCALE_NV16_E4M3        (FP4 operands only) E4M3 factor codes, positive (the
 *                                  tensor core reads them as unsigned E4M3), one per 16
 *                                  elements of K, in the same atoms: [L][ceil(rows/128)]
 *                                  [ceil(K/64)][32][4][4], j4 the 16-element block of the
 *                                  64-element K block.
 *
 * Ownership: the caller owns every buffer (inputs, outputs, workspace) and
 * every pointer above is a DEVICE pointer on the plan's device.  A plan holds
 * host state only and may be reused for any number of calls with the same
 * shapes; it is not thread-safe (one plan per host thread).
 *
 * Asynchrony: fp8mm_run only enqueues work on the given stream (amax is reset
 * on the stream, then the kernel runs).  It never synchronises.  Outputs are
 * valid once the stream reaches that point.
 *
 * Errors: every call returns an fp8mm_status; nothing throws across this ABI.
 * Validation failures return before any CUDA call.  A device-side abort (an
 * internal wait that exceeded its time limit) is recorded in a device word
 * that fp8mm_device_error reads; the outputs of that call are then undefined.
 */
#ifndef FP8MM_H
#define FP8MM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Operand formats.  FP8MM_E2M1 is packed FP4 (float4_e2m1fn_x2: two values per
 * byte along K, element 2i in the low four bits of byte i; cuDNN "GEMM + Amax
 * (SM100)", Dtypes and Layouts): A and B both E2M1, K-major, K % 64 == 0, a
 * block-scaled form (FP8MM_SCALE_MX32_UE8M0 = MXFP4 or FP8MM_SCALE_NV16_E4M3
 * = NVFP4), fast accumulation; a and b then hold K/2 bytes per row. */
typedef enum { FP8MM_E4M3 = 0, FP8MM_E5M2 = 1, FP8MM_E2M1 = 2 } fp8mm_fmt;

/* FP8 outputs (E4M3, E5M2): C = round_sat(fp32(alpha * acc) * scale_result), rounded once to
 * nearest even and saturated to the largest finite value (NaN stays NaN); amax is then
 * max |fp32(alpha * acc)|, before scale_result and the rounding (it sets the next quantisation
 * scale).  FP8 outputs need N % 16 == 0 and take no bias. */
typedef enum {
  FP8MM_OUT_F32 = 0,
  FP8MM_OUT_BF16 = 1,
  FP8MM_OUT_F16 = 2,
  FP8MM_OUT_E4M3 = 3,
  FP8MM_OUT_E5M2 = 4
} fp8mm_out;

typedef enum {
  FP8MM_SCALE_TENSOR = 0,
  FP8MM_SCALE_A1x128_B1x128 = 1,
  FP8MM_SCALE_A1x128_B128x128 = 2,
  FP8MM_SCALE_MX32_UE8M0 = 3,
  FP8MM_SCALE_NV16_E4M3 = 4
} fp8mm_scale_mode;

typedef enum {
  FP8MM_OK = 0,
  FP8MM_ERR_INVALID = 1,     /* null pointer, negative size, value out of range    */
  FP8MM_ERR_ALIGNMENT = 2,   /* a row or pointer is not 16-byte aligned (K % 16, N rows of C) */
  FP8MM_ERR_UNSUPPORTED = 3, /* outside this library: mixed formats in the MX form, sizes >= 2^31 */
  FP8MM_ERR_REJECTED = 4,    /* a format pair torch._scaled_mm refuses (only with strict_torch) */
  FP8MM_ERR_WORKSPACE = 5,   /* workspace missing or smaller than fp8mm_workspace_size */
  FP8MM_ERR_CUDA = 6,        /* a CUDA runtime call or the launch failed           */
  FP8MM_ERR_DEVICE = 7       /* the kernel aborted (see fp8mm_device_error)        */
} fp8mm_status;

/* Problem description.  Zero-initialise, then set the fields. */
typedef struct {
  int64_t M, N, K, L;  /* L = batch count (1 for a plain GEMM); M, N, L may be 0 */
  int32_t a_fmt;       /* fp8mm_fmt of A */
  int32_t b_fmt;       /* fp8mm_fmt of B */
  int32_t scale_mode;  /* fp8mm_scale_mode */
  int32_t out_dtype;   /* fp8mm_out */
  int32_t fast_accum;  /* 1: one fp32 chain over K; 0: 128-K chunks promoted into an fp32
                          register accumulator.  The block-scale modes always promote per
                          128-K chunk (their scales change per chunk). */
  int32_t splitk;      /* 0: choose; S >= 1: split K into S contiguous 128-aligned ranges */
  int32_t swap_ab;     /* 0: choose; 1: force on; 2: force off */
  int32_t block_n;     /* 0: choose; else the tile width on the MMA's N side, one the library
                          instantiates: fast 16, 32, 64, 128, 192, 224, 256 (CTA pairs 128, 192,
                          224, 256); slow 16, 32, 64, 128 (CTA pairs 128) and, unswapped and
                          unsplit, 192, 224, 256 on one CTA or a CTA pair (192/224 not with
                          128x128 B scales); MX 128, 224, 256 (CTA pairs 256, slow MX 128); FP4
                          128, 256.  Others: FP8MM_ERR_UNSUPPORTED. */
  int32_t device;      /* CUDA device ordinal the plan is for */
  int32_t cta_pair;    /* two-SM (CTA pair) tiles: 0 choose; 1 force on; 2 force off */
  int32_t epi_warps;   /* epilogue warps per CTA: 0 choose, 8 or 16 */
  int32_t stages;      /* shared-memory pipeline depth: 0 choose (as many as fit), else 2..12 */
  int32_t strict_torch; /* 0: accept all four E4M3/E5M2 pairs; 1: refuse with FP8MM_ERR_REJECTED
                           what torch._scaled_mm refuses: E5M2 x E5M2, and E4M3 x E4M3 with an
                           E5M2 output (mmaemu "Testing mmaemu", T1 hw_mini, expected error
                           classes) */
  int32_t bias;        /* 1: fp8mm_run_ex adds bias[n] (out_dtype, N values) to every row before the
                          one rounding (TileOPs GemmFP8FwdOp); not for FP8 outputs.  0: no bias. */
  int32_t a_major;     /* 0: a is [L][M][K] (K-major); 1: a is [L][K][M] (M-major, M % 16 == 0) */
  int32_t b_major;     /* 0: b is [L][N][K] (K-major); 1: b is [L][K][N] (N-major, N % 16 == 0).
                          An M/N-major operand is copied into K-major workspace by one extra
                          HBM-bound kernel before the GEMM (BmmFP8FwdOp's transposing copy). */
} fp8mm_desc;

typedef struct fp8mm_plan_s fp8mm_plan_t;

/* What a plan chose (for reports and tests). */
typedef struct {
  int32_t swap_ab;      /* 1 if B plays the MMA's A operand (skinny M) */
  int32_t block_m;      /* rows per CTA on the MMA's M side (128) */
  int32_t block_n;      /* tile width on the MMA's N side */
  int32_t splitk;       /* K ranges per output tile */
  int32_t stages;       /* shared-memory pipeline depth */
  int32_t grid;         /* persistent CTAs launched */
  int64_t units;        /* (tile, K range) work units */
  int32_t slow;         /* 1 if 128-K chunks are promoted in registers */
  int32_t smem_bytes;   /* dynamic shared memory per CTA */
  int32_t cta_pair;     /* 1 if tiles are computed by CTA pairs with two-SM MMAs (256-row tiles) */
  int32_t epi_warps;    /* epilogue warps per CTA */
} fp8mm_plan_info;

/* Validate desc and choose tiles, swap-AB and split-K for the device (the
 * check-support-then-compile step of cuDNN "GEMM + Amax (SM100)", Class API:
 * everything that can be refused is refused here, before any call).  On
 * success *out owns a new plan (free with fp8mm_destroy).  Reads the device's
 * SM count and kernel attributes; launches nothing.  Errors: INVALID (null
 * pointer, negative size, field out of range), ALIGNMENT (K % 16, rows of C
 * not 16-byte multiples, an M/N-major operand with M or N % 16), UNSUPPORTED
 * (a form or override this library does not build), REJECTED (strict_torch),
 * CUDA (a device query failed). */
fp8mm_status fp8mm_plan(const fp8mm_desc* desc, fp8mm_plan_t** out);

/* Device bytes the caller must pass as workspace to fp8mm_run (0 if none):
 * the K-major copies of M/N-major operands, then the split-K partial tiles
 * and their arrival counters (the workspace a profile states up front in
 * mmaemu "API reference (v0.1)", Profile; here the caller allocates it). */
fp8mm_status fp8mm_workspace_size(const fp8mm_plan_t* plan, size_t* bytes);

/* Enqueue one GEMM + amax on `stream` (a cudaStream_t; NULL = legacy default
 * stream): torch._scaled_mm's product (mmaemu "API reference (v0.1)",
 * mmaemu.scaled_mm) with TileOPs GemmFP8FwdOp's scale forms and cuDNN "GEMM +
 * Amax (SM100)"'s block-scaled form and Amax.  a, b, scale_a, scale_b, c,
 * amax, workspace: device pointers laid out as described above.  a, b and c
 * must be 16-byte aligned; scale pointers 4-byte aligned (MX factor atoms
 * 16-byte aligned), workspace 256-byte aligned; else FP8MM_ERR_ALIGNMENT.
 * c and amax are written, never read.  Plans with desc.bias = 1 must use
 * fp8mm_run_ex (FP8MM_ERR_INVALID here); FP8 outputs get scale_result = 1. */
fp8mm_status fp8mm_run(fp8mm_plan_t* plan, const void* a, const void* b, const void* scale_a,
                       const void* scale_b, void* c, float* amax, void* workspace,
                       size_t workspace_bytes, void* stream);

/* fp8mm_run with the two epilogue operands: scale_result (device, one fp32,
 * read only for FP8 outputs; NULL means 1) and bias (device, [N] of
 * out_dtype, 4-byte aligned for fp32, 2-byte for bf16/fp16; required exactly
 * when desc.bias = 1, else FP8MM_ERR_INVALID).  Sources: mmaemu.scaled_mm's
 * scale_result; TileOPs GemmFP8FwdOp's bias. */
fp8mm_status fp8mm_run_ex(fp8mm_plan_t* plan, const void* a, const void* b, const void* scale_a,
                          const void* scale_b, const float* scale_result, const void* bias, void* c,
                          float* amax, void* workspace, size_t workspace_bytes, void* stream);

/* Algorithmic work of one call (TileOPs "Linear Algebra Operators",
 * eval_roofline: the flops and bytes the op must do at least): flops =
 * 2*M*N*K*L; bytes = A + B + scales + bias + C + amax (workspace traffic --
 * split-K partials and K-major copies of M/N-major operands -- not counted). */
fp8mm_status fp8mm_plan_roofline(const fp8mm_plan_t* plan, double* flops, double* bytes);

fp8mm_status fp8mm_plan_get_info(const fp8mm_plan_t* plan, fp8mm_plan_info* info);

/* What fp8mm_plan would choose for a device with `sms` SMs and
 * `max_smem_bytes` of opt-in shared memory per block, without touching CUDA
 * (no device query, no kernel attribute or occupancy query: CTA-pair grids
 * assume one pair per two SMs, and the held kernels' register check is left
 * out).  For tests and planning tools; fp8mm_plan stays authoritative.
 * FP8MM_ERR_INVALID for sms < 2 or max_smem_bytes <= 0, else as fp8mm_plan. */
fp8mm_status fp8mm_plan_preview(const fp8mm_desc* desc, int32_t sms, int32_t max_smem_bytes,
                                fp8mm_plan_info* info);

void fp8mm_destroy(fp8mm_plan_t* plan);

/* Static string naming a status code. */
const char* fp8mm_status_string(fp8mm_status status);

/* Read (and with clear != 0, reset) the device's abort word: 0 when no kernel
 * on `device` has aborted since the last clear.  Synchronises the device. */
fp8mm_status fp8mm_device_error(int device, uint32_t* code, int clear);

/* Test support for the abort path.  While enabled (process-wide), GEMM kernels
 * launched afterwards issue no operand loads, so the MMA issuer's first wait
 * for a stage, and the epilogue's for the accumulator, never complete: the
 * first to reach its limit (2^31 SM cycles, about one second) records a
 * nonzero code in the abort word (fp8mm_device_error), and every role of the
 * kernel drains and returns; the CUDA context stays usable.  The outputs of
 * such calls are undefined.  Not for use outside tests. */
fp8mm_status fp8mm_test_withhold_loads(int enable);

/* Number of kernel launches fp8mm_run enqueues for this plan (the amax reset
 * and, with split-K, the counter reset are stream memsets, not kernels). */
fp8mm_status fp8mm_plan_kernel_launches(const fp8mm_plan_t* plan, int32_t* launches);

/* Largest split-K scratch fp8mm_run_static_workspace can serve (16 MiB). */
#define FP8MM_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)

/* fp8mm_run for callers that cannot allocate device memory -- for example a
 * plugin or custom-call host that owns every device buffer and hands an
 * operation only its inputs and outputs, or a service whose device-memory
 * budget is fixed once it has started.  The pages have no counterpart of this
 * entry point; it exists for such callers.
 *
 * Same arguments and results as fp8mm_run minus the workspace: split-K
 * scratch comes from one array of FP8MM_STATIC_WORKSPACE_BYTES bytes that the
 * library defines in device memory and that every GPU which loads the library
 * keeps until the process exits.  Nothing is allocated or freed by this call.
 *   - A plan whose fp8mm_workspace_size exceeds FP8MM_STATIC_WORKSPACE_BYTES
 *     is rejected with FP8MM_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device that needs scratch looks up the array's
 *     device address (cudaGetSymbolAddress, with that device current); make
 *     that first call before any stream capture.  The address is kept for
 *     the life of the process, so it assumes the device's primary context is
 *     not reset (cudaDeviceReset) in between.
 *   - Plans with M/N-major operands need workspace for their K-major copies
 *     too; it counts against the same limit.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents.  Each call resets the parts that must start at zero on its
 *     stream, so calls in stream order are independent; calls that may run
 *     at the same time on the GPU (other streams, other threads) race on the
 *     array and give undefined results. */
fp8mm_status fp8mm_run_static_workspace(fp8mm_plan_t* plan, const void* a, const void* b,
                                        const void* scale_a, const void* scale_b, void* c,
                                        float* amax, void* stream);

/* One-shot form: plan, run, destroy.  Same arguments as fp8mm_plan + fp8mm_run. */
fp8mm_status fp8mm_gemm(const fp8mm_desc* desc, const void* a, const void* b,
                        const void* scale_a, const void* scale_b, void* c, float* amax,
                        void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8MM_H */
