/*
 * fp4q.h -- C ABI of libfp4q.so: UE5M3-scaled FP4 (E2M1) quantisation and the
 * block-scaled GEMM on a GB300 (sm_103a).
 *
 * Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
 * Abstract.  Linear-layer operands are stored as E2M1 payloads with one
 * unsigned E5M3 (UE5M3) scale per block of 16 elements under an FP32 tensor
 * scale refreshed periodically; forward operands round to nearest even and
 * backward gradients round stochastically; all internal linears run their
 * matrix multiplications (fprop, dgrad, wgrad) on these operands, with UE5M3
 * emulated in software because tensor cores take only E4M3/E8M0 block scales.
 *
 * Conventions shared by every call
 *  - Every pointer argument except `stream` and those documented as host
 *    pointers is a DEVICE pointer, owned by the caller; the library never
 *    allocates or frees memory, and never synchronises the stream (except
 *    fp4q_get_device_status, which waits for its own stream).  Calls are asynchronous on `stream`
 *    (a cudaStream_t; NULL = the legacy default stream).
 *  - Data-dependent scalars (amax, tensor scale) stay on the device, so that a
 *    whole quantise -> GEMM sequence needs no host round trip.
 *  - Tensors are row-major and densely packed.  Every tensor pointer must be
 *    16-byte aligned; scalar pointers (amax, tensor scales) 4-byte aligned,
 *    stats 8-byte aligned.  BF16 is the IEEE bfloat16 bit pattern (uint16).
 *  - Validation errors (bad enum, shape, null or misaligned pointer) are
 *    returned synchronously before any launch and nothing is written.
 *    Launch failures return FP4Q_ERR_CUDA.  Conditions only the GPU can see
 *    (non-finite input, a pipeline wait that ran out) are latched in a device
 *    status word read by fp4q_get_device_status.
 *
 * Formats (readings of the method where the abstract leaves them open)
 *  - E2M1 element: sign bit 3, 2-bit exponent (bias 1), 1-bit mantissa;
 *    magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  Packed two per byte, the
 *    element with the even index in the low nibble.
 *  - UE5M3 scale: 5-bit exponent (bias 15), 3-bit mantissa, subnormals
 *    m/8 * 2^-14, 0xFF reserved (never produced), largest 0xFE = 114688.
 *    UE4M3 (bias 7, largest 0x7E = 448) is available for comparison.
 *  - Tensor scale T = amax / (6 * Smax / H), T = 1 for an all-zero tensor,
 *    raised to 2^-100 if smaller.
 *  - Block of 16: s* = amax_b / (6 T) rounded to the scale format (nearest,
 *    ties to even, saturating); element q = x * (1 / (s T)); RNE or
 *    stochastic rounding to E2M1, saturating at 6.  Every product, quotient
 *    and reciprocal is one IEEE binary32 operation rounded to nearest even.
 *  - Stochastic rounding draws Philox4x32-10 (key = seed), counter
 *    (i/4, i/4 >> 32, axis, 0), word i % 4, for the element with row-major
 *    index i of the input; round up iff (word >> 8) * 2^-24 < fractional
 *    position between the two neighbouring grid points.
 */
#ifndef FP4Q_H
#define FP4Q_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP4Q_OK = 0,
    FP4Q_ERR_ARG = 1,        /* null pointer or unknown enum value */
    FP4Q_ERR_SHAPE = 2,      /* a size is not a supported multiple or too large */
    FP4Q_ERR_ALIGN = 3,      /* a pointer is misaligned (see conventions) */
    FP4Q_ERR_CUDA = 4,       /* a CUDA runtime/driver call failed */
    FP4Q_ERR_NONFINITE = 5,  /* device status: an input element was inf/NaN */
    FP4Q_ERR_TIMEOUT = 6     /* device status: a bounded pipeline wait gave up */
} fp4q_status;

typedef enum { FP4Q_AXIS_ROW = 0, FP4Q_AXIS_COL = 1, FP4Q_AXIS_BOTH = 2, FP4Q_AXIS_BOTH_2D = 3 } fp4q_axis;
typedef enum { FP4Q_RNE = 0, FP4Q_SR = 1 } fp4q_rounding;
typedef enum { FP4Q_SCALE_UE5M3 = 0, FP4Q_SCALE_UE4M3 = 1 } fp4q_scale_fmt;

/* Per-quantisation counters, device resident. */
typedef struct {
    unsigned long long scale_sat_blocks;    /* blocks with s* above the largest scale */
    unsigned long long scale_uflow_blocks;  /* nonzero blocks whose scale encoded to 0 */
    unsigned long long elem_clamped;        /* elements with |q| > 6 (saturated) */
    unsigned long long elem_flushed;        /* nonzero elements encoded as (+-)0 */
} fp4q_stats;

/* amax = max |x| over n BF16 elements (the current-tensor-scaling pass of the
 * method's TE baseline, and the first refresh of periodic scaling).
 * in_bf16: device, n elements.  out_amax: device float, overwritten.
 * n may be 0 (amax = 0).  A non-finite element latches FP4Q_ERR_NONFINITE. */
fp4q_status fp4q_amax(const void* in_bf16, int64_t n, float* out_amax, void* stream);

/* Tensor scale from an amax (periodic tensor scaling, Abstract):
 * *out_scale = amax / (6 * Smax(fmt) / headroom) with the zero and floor
 * rules above.  amax, out_scale: device floats.  headroom: host value, a
 * power of two >= 1. */
fp4q_status fp4q_tensor_scale(const float* amax, fp4q_scale_fmt fmt, float headroom,
                              float* out_scale, void* stream);

/* Block-16 quantisation of a rows x cols BF16 tensor (E2M1 + UE5M3 block
 * scales, Abstract).  rows and cols: multiples of 16, >= 0; for every axis
 * but ROW, ceil(rows/128) * ceil(cols/128) <= 2^31 - 1 (FP4Q_ERR_SHAPE
 * otherwise).  Element indices are 64-bit throughout.
 *  axis ROW : blocks along a row.  out_payload_row [rows, cols/2] bytes,
 *             out_scales_row [rows, cols/16] bytes.
 *  axis COL : blocks along a column, written as the row-wise quantisation of
 *             the transpose: out_payload_col [cols, rows/2],
 *             out_scales_col [cols, rows/16].
 *  axis BOTH: both outputs from one read of the input.
 *  axis BOTH_2D: both outputs, one scale per 16 x 16 tile (the
 *             transposition-invariant block scaling listed among the related
 *             work of the UE5M3 page): the tile's amax picks its code by the
 *             block rule, every element is quantised once with it (FP4Q_SR
 *             with the row-wise stream, axis id 0), and the result is written
 *             in both layouts -- the column payload is the nibble transpose
 *             of the row payload; out_scales_row repeats a tile's code on its
 *             16 rows, out_scales_col on its 16 columns.
 * Unused output pointers may be NULL.  tensor_scale: device float (T).
 * rnd/seed: FP4Q_SR draws its bits as stated above (row-wise uses axis id 0,
 * column-wise 1); seed is ignored for FP4Q_RNE.
 * out_stats (nullable): zeroed, then filled; for BOTH it points to TWO structs
 * (row-wise, column-wise); for BOTH_2D to one (scale counts per 16 x 16
 * tile, element counts once per element).  out_amax (nullable): zeroed, then set to max |x|
 * of this input -- the by-product periodic scaling keeps for its next
 * refresh. */
fp4q_status fp4q_quantize(const void* in_bf16, int64_t rows, int64_t cols, fp4q_axis axis,
                          fp4q_scale_fmt fmt, const float* tensor_scale, fp4q_rounding rnd,
                          uint64_t seed,
                          uint8_t* out_payload_row, uint8_t* out_scales_row,
                          uint8_t* out_payload_col, uint8_t* out_scales_col,
                          fp4q_stats* out_stats, float* out_amax, void* stream);

/* Dequantisation of a [rows, cols] block-scaled tensor quantised along its
 * rows: v = (e * s) * T, each product rounded to binary32, written as BF16
 * (rounded to nearest even) or binary32 (out_is_f32 != 0).
 * payload [rows, cols/2], scales [rows, cols/16], tensor_scale device float. */
fp4q_status fp4q_dequantize(const uint8_t* payload, const uint8_t* scales, int64_t rows,
                            int64_t cols, fp4q_scale_fmt fmt, const float* tensor_scale,
                            void* out, int out_is_f32, void* stream);

/* Block-scaled GEMM, the method's FP4 matrix multiplication (fprop
 * Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X, each written as C = A B^T):
 *   C[m, n] = (T_A * T_B) * sum_k deq(A)[m, k] * deq(B)[n, k]
 * A: payload [M, K/2] + scales [M, K/16], B: payload [N, K/2] + scales
 * [N, K/16], both quantised along K; A_tscale, B_tscale device floats.
 * The UE5M3 scales are applied in software: each tile is expanded in shared
 * memory to FP16 as e*s*2^-4 (exact: at most 6 significant bits, within the
 * FP16 range and on its subnormal grid) and multiplied on the tcgen05 tensor
 * cores with binary32 accumulation; the 2^-8 returns in the epilogue.  out: [M, N] BF16
 * (out_is_f32 == 0) or binary32.  M, N >= 0 (any value up to 2^31 - 1;
 * M at most 65535 * 256), K a multiple of 64 up to 2^31 - 64 (K = 0 writes
 * zeros); FP4Q_ERR_SHAPE otherwise.  Every internal pipeline wait is bounded (about 2 s);
 * one that runs out latches FP4Q_ERR_TIMEOUT and the kernel exits, leaving
 * `out` unspecified.  Test hooks (environment, read per call):
 * FP4Q_TEST_GEMM_WAIT_CYCLES shortens the bound, FP4Q_TEST_GEMM_SKIP_LOADS=1
 * withholds the operand loads so that the waits run out. */
fp4q_status fp4q_gemm(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                      const uint8_t* B, const uint8_t* B_scales, const float* B_tscale,
                      int64_t M, int64_t N, int64_t K, fp4q_scale_fmt fmt,
                      void* out, int out_is_f32, void* stream);

/* fp4q_gemm whose epilogue also quantises the BF16 result for the next layer
 * (quantisation fused into the producing GEMM -- the "format-aware fusion"
 * direction the UE5M3 page lists among related work): C is rounded to BF16
 * as fp4q_gemm writes it and quantised row-wise, blocks of 16 along N, round
 * to nearest even, with the device tensor scale c_tscale (e.g. refreshed
 * periodically from an earlier out_amax):
 *   out_payload [M, N/2], out_scales [M, N/16] = fp4q_quantize(bf16(C), ROW,
 *   fmt, c_tscale, RNE) byte for byte;
 *   out_bf16 (nullable) = bf16(C) [M, N]; out_amax (nullable) = max |bf16(C)|
 *   (zeroed, then set; a non-finite element latches FP4Q_ERR_NONFINITE).
 * Operands, fmt (also the format of the output scales) and K as fp4q_gemm;
 * N must be a multiple of 32. */
fp4q_status fp4q_gemm_quantize(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                               const uint8_t* B, const uint8_t* B_scales, const float* B_tscale,
                               int64_t M, int64_t N, int64_t K, fp4q_scale_fmt fmt,
                               const float* c_tscale, void* out_bf16, uint8_t* out_payload,
                               uint8_t* out_scales, float* out_amax, void* stream);

/* Native NVFP4 GEMM: the same contraction as fp4q_gemm on operands whose
 * block scales are UE4M3 (the NVFP4 format of the TE recipe the method is
 * compared against, and of the abstract's native-NVFP4 execution ablation),
 * multiplied by the tensor cores' own block-scaled MMA -- no software
 * expansion:
 *   C[m, n] = (T_A * T_B) * sum_k (e s)_A[m, k] * (e s)_B[n, k]
 * A: payload [M, K/2] + UE4M3 scales [M, K/16]; B: [N, K/2] + [N, K/16]
 * (fp4q_quantize with FP4Q_SCALE_UE4M3 writes exactly this layout);
 * A_tscale, B_tscale device floats.  Binary32 accumulation; out [M, N] BF16
 * (out_is_f32 == 0) or binary32.  M, N >= 0 (M at most 65535 * 128), K a
 * multiple of 256 (K = 0 writes zeros); FP4Q_ERR_SHAPE otherwise.  Waits are
 * bounded as in fp4q_gemm, with the same test hooks
 * (FP4Q_TEST_GEMM_WAIT_CYCLES, FP4Q_TEST_GEMM_SKIP_LOADS). */
fp4q_status fp4q_gemm_nvfp4(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                            const uint8_t* B, const uint8_t* B_scales, const float* B_tscale,
                            int64_t M, int64_t N, int64_t K, void* out, int out_is_f32, void* stream);

/* Exponent rebias of UE5M3 block-scale codes, so that a UE5M3-scaled GEMM can
 * run exactly on the tensor cores' UE4M3 block-scaled MMA ("UE5M3 FP4 Block
 * Scaling for Stable Language Model Pretraining", Abstract: the hardware
 * takes E4M3/E8M0 block scales, which is why UE5M3 is emulated).  UE5M3 and
 * UE4M3 share their 3 mantissa bits, so a group of scales whose non-zero
 * values lie in 14 consecutive binades [e_top - 13, e_top] is exactly
 * factor * (UE4M3 values) with factor = 2^(e_top - 7); the group's largest
 * binade lands in UE4M3 exponent field 14.  Groups:
 *   per_row != 0: each row; e_top is the row's largest binade; a row with no
 *                 non-zero scale gets factor 1 and zero codes;
 *   per_row == 0: the whole tensor, with the fixed window e_top = 16 (the
 *                 binade of UE5M3's largest finite scale, where the tensor
 *                 scale puts the tensor's amax): factor 2^9, binades 3..16.
 * scales: UE5M3 codes [rows, nblocks] (device); out_scales: UE4M3 codes of
 * the same shape (device; must not overlap `scales`); out_factor: binary32
 * [rows] (per_row) or [1] (device).  Zero codes stay zero.  A group that does
 * not fit sets *inout_nofit to 1 (a device int, OR-ed, never cleared here: the
 * caller zeroes it, then may rebias several operands into the same flag); the
 * codes and factor of such a group are unspecified.  nblocks a multiple of 16
 * (K = 16 nblocks a multiple of 256, as fp4q_gemm_nvfp4 needs); scales and
 * out_scales 16-byte aligned, out_factor and inout_nofit 4-byte aligned.
 * Asynchronous on `stream`; nothing is read back to the host. */
fp4q_status fp4q_rebias_scales(const uint8_t* scales, int64_t rows, int64_t nblocks, int per_row,
                               uint8_t* out_scales, float* out_factor, int* inout_nofit, void* stream);

/* fp4q_gemm_nvfp4 on rebiased operands: A's UE4M3 codes with one power-of-two
 * factor per row (A_factor [M]), B's with one for the tensor (B_factor [1]),
 * as fp4q_rebias_scales writes them:
 *   C[m, n] = (T_A * T_B * fb * fa[m]) * sum_k (e s4)_A[m, k] * (e s4)_B[n, k]
 * the factors applied to the binary32 accumulator after T_A * T_B (exact
 * products of powers of two while the result stays in binary32's normal
 * range).  With codes and factors from fp4q_rebias_scales that fitted, this
 * is the UE5M3 contraction of fp4q_gemm on the original scales, up to the
 * accumulation order.  skip_if_set (nullable device int): when it is non-zero
 * as the kernel starts, the launch writes nothing (K = 0 still writes zeros);
 * it is read once on the device, never on the host.  Shapes, alignment, waits
 * and test hooks as fp4q_gemm_nvfp4; A_factor, B_factor 4-byte aligned. */
fp4q_status fp4q_gemm_nvfp4_rebiased(const uint8_t* A, const uint8_t* A_scales4, const float* A_factor,
                                     const float* A_tscale, const uint8_t* B, const uint8_t* B_scales4,
                                     const float* B_factor, const float* B_tscale, int64_t M, int64_t N,
                                     int64_t K, const int* skip_if_set, void* out, int out_is_f32,
                                     void* stream);

/* fp4q_gemm that runs only when the device int *run_if_set is non-zero as the
 * kernel starts (read once on the device, never on the host); otherwise the
 * launch writes nothing (K = 0 still writes zeros).  With the flag of
 * fp4q_rebias_scales it is the exact fallback of fp4q_gemm_nvfp4_rebiased
 * into the same `out`: issued after it on one stream, exactly one of the two
 * writes C.  Arguments otherwise as fp4q_gemm; run_if_set 4-byte aligned. */
fp4q_status fp4q_gemm_if(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                         const uint8_t* B, const uint8_t* B_scales, const float* B_tscale, int64_t M,
                         int64_t N, int64_t K, fp4q_scale_fmt fmt, const int* run_if_set, void* out,
                         int out_is_f32, void* stream);

/* fp4q_gemm_nvfp4_rebiased whose epilogue also quantises the BF16 result for
 * the next layer, as fp4q_gemm_quantize does for the emulated GEMM (the
 * "format-aware fusion" direction the UE5M3 page lists among related work):
 * bf16(C) row-wise, blocks of 16 along N, round to nearest even, scale
 * format fmt, device tensor scale c_tscale:
 *   out_payload [M, N/2], out_scales [M, N/16] = fp4q_quantize(bf16(C), ROW,
 *   fmt, c_tscale, RNE) byte for byte; out_bf16 (nullable) = bf16(C);
 *   out_amax (nullable): max-ed with max |bf16(C)| -- NOT zeroed first, so
 *   that this call and fp4q_gemm_quantize_if (its fallback) can share it;
 *   the caller zeroes it before the pair (a non-finite element latches
 *   FP4Q_ERR_NONFINITE).
 * skip_if_set as fp4q_gemm_nvfp4_rebiased (a skipped launch writes none of
 * the outputs); N must be a multiple of 32; otherwise as that call. */
fp4q_status fp4q_gemm_nvfp4_rebiased_quantize(const uint8_t* A, const uint8_t* A_scales4, const float* A_factor,
                                              const float* A_tscale, const uint8_t* B, const uint8_t* B_scales4,
                                              const float* B_factor, const float* B_tscale, int64_t M, int64_t N,
                                              int64_t K, const int* skip_if_set, fp4q_scale_fmt fmt,
                                              const float* c_tscale, void* out_bf16, uint8_t* out_payload,
                                              uint8_t* out_scales, float* out_amax, void* stream);

/* fp4q_gemm_quantize run only when the device int *run_if_set is non-zero
 * (read once on the device), its out_amax max-ed into rather than zeroed
 * first: the exact fallback of fp4q_gemm_nvfp4_rebiased_quantize into the
 * same outputs.  K = 0 still writes zero outputs (out_amax unchanged).
 * Arguments otherwise as fp4q_gemm_quantize; run_if_set 4-byte aligned. */
fp4q_status fp4q_gemm_quantize_if(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                                  const uint8_t* B, const uint8_t* B_scales, const float* B_tscale, int64_t M,
                                  int64_t N, int64_t K, fp4q_scale_fmt fmt, const int* run_if_set,
                                  const float* c_tscale, void* out_bf16, uint8_t* out_payload,
                                  uint8_t* out_scales, float* out_amax, void* stream);

/* Two-window exponent rebias of UE5M3 block-scale codes, per row, for an
 * operand whose rows span more binades than one UE4M3 window holds (the
 * column-wise codes of a gradient whose per-token magnitudes differ by many
 * decades, the A operand of wgrad).  Same reading of the page as
 * fp4q_rebias_scales (its Abstract: UE5M3 is emulated because the hardware
 * takes E4M3/E8M0 block scales), with two 14-binade windows under each row's
 * largest binade e_top:
 *   high window [e_top - 13, e_top]:      out_hi code, factor 2^(e_top - 7)
 *   low window  [e_top - 27, e_top - 14]: out_lo code, factor 2^(e_top - 21)
 * each non-zero code going to exactly one of out_hi, out_lo (zero in the
 * other), so that
 *   s = factor_hi * UE4M3(out_hi) + factor_lo * UE4M3(out_lo)   exactly.
 * factor_lo = factor_hi * 2^-14 always (a row with no non-zero scale: 1 and
 * 2^-14, zero codes).  A non-zero code below both windows sets *inout_nofit to
 * 1 (OR-ed, never cleared here) and is zero in both outputs.
 * scales: UE5M3 codes [rows, nblocks]; out_hi, out_lo: UE4M3 codes of the
 * same shape; out_factor_hi, out_factor_lo: binary32 [rows]; all device.  The
 * three code arrays must not overlap (FP4Q_ERR_ARG).  nblocks a multiple of
 * 16; code arrays 16-byte aligned, factors and inout_nofit 4-byte aligned.
 * Asynchronous on `stream`; nothing is read back to the host. */
fp4q_status fp4q_rebias_scales_two_windows(const uint8_t* scales, int64_t rows, int64_t nblocks, uint8_t* out_hi,
                                           uint8_t* out_lo, float* out_factor_hi, float* out_factor_lo,
                                           int* inout_nofit, void* stream);

/* The UE5M3 GEMM on the native block-scaled MMA with A's codes in two windows
 * (fp4q_rebias_scales_two_windows) and B's in one (fp4q_rebias_scales,
 * per_row == 0): each K step multiplies the same E2M1 operand tiles twice,
 * once with A's high-window codes and once with its low-window codes, into
 * two binary32 accumulators, and the epilogue forms
 *   C[m, n] = (T_A * T_B * fb * fa_hi[m]) * (acc_hi[m, n] + 2^-14 acc_lo[m, n])
 * (the 2^-14 scaling exact, the sum rounded once in binary32), which is the
 * UE5M3 contraction of fp4q_gemm on the original scales up to the
 * accumulation order.  A_factor_hi: the per-row high-window factors [M];
 * skip_if_set, shapes (K a multiple of 256), alignment, waits, test hooks and
 * out as fp4q_gemm_nvfp4_rebiased; A_scales_lo 16-byte aligned. */
fp4q_status fp4q_gemm_nvfp4_two_windows(const uint8_t* A, const uint8_t* A_scales_hi, const uint8_t* A_scales_lo,
                                        const float* A_factor_hi, const float* A_tscale, const uint8_t* B,
                                        const uint8_t* B_scales4, const float* B_factor, const float* B_tscale,
                                        int64_t M, int64_t N, int64_t K, const int* skip_if_set, void* out,
                                        int out_is_f32, void* stream);

/* Reads the device status word of the current device in the order of
 * `stream` (after every call already issued on it), waits for `stream` alone
 * (no other stream of the device is synchronised), returns the latched
 * condition in *out (FP4Q_ERR_TIMEOUT, else FP4Q_ERR_NONFINITE, else
 * FP4Q_OK) and clears the bits it reported (an atomic AND on the stream,
 * waited for before returning).  The word is shared by every stream of the
 * device: a condition latched by work on another stream is seen once that
 * work has completed, and one latched between the read and the clear stays
 * set for the next call.  out: HOST pointer.  Returns FP4Q_ERR_ARG for a
 * null out, FP4Q_ERR_CUDA if a copy, launch or wait fails. */
fp4q_status fp4q_get_device_status(int* out, void* stream);

/* Static description of a status code.  Never NULL. */
const char* fp4q_status_string(fp4q_status s);

#ifdef __cplusplus
}
#endif

#endif /* FP4Q_H */
