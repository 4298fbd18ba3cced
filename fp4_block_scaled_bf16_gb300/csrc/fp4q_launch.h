// fp4q_launch.h -- host-side launch interface between the C ABI (fp4q_api.cu)
// and the kernel translation units (quantize.cu, gemm.cu, gemm_native.cu,
// rebias.cu).  Internal to libfp4q.so; arguments are validated by the ABI
// layer before they get here.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp4q {

struct StatsDev;

struct QuantArgs {
  const void* in;       // BF16 [rows, cols]
  int64_t rows, cols;   // multiples of 16
  int axis;             // 0 row, 1 col, 2 both
  int fmt;              // 0 UE5M3, 1 UE4M3
  const float* tscale;  // device T
  bool sr;
  uint64_t seed;
  uint8_t *pay_row, *sc_row, *pay_col, *sc_col;
  StatsDev* stats;      // nullable; two structs for axis 2
  float* amax_out;      // nullable
  int* status;          // device status word
};

cudaError_t launch_amax(const void* in, int64_t n, float* out, int* status, cudaStream_t st);
cudaError_t launch_tensor_scale(const float* amax, float denom, float* out, cudaStream_t st);
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st);
cudaError_t launch_dequantize(const uint8_t* payload, const uint8_t* scales, int64_t rows,
                              int64_t cols, int fmt, const float* tscale, void* out, bool f32,
                              cudaStream_t st);

struct GemmArgs {
  const uint8_t *A, *As, *B, *Bs;   // payloads [M, K/2], [N, K/2]; scales [., K/16]
  const float *TA, *TB;             // device tensor scales
  int64_t M, N, K;                  // K multiple of 64
  int fmt;
  void* out;                        // [M, N] BF16 or binary32
  bool out_f32;
  int* status;
  // epilogue quantisation of the BF16 result (null qpay: none); out may then be null
  const float* TC = nullptr;        // device tensor scale of C
  uint8_t *qpay = nullptr, *qsc = nullptr;   // [M, N/2], [M, N/16], row-wise, RNE
  float* qamax = nullptr;           // nullable: max |bf16(C)|
  long long wait_cycles;            // budget of every pipeline wait (clock64 cycles)
  bool skip_loads;                  // test hook: the producer issues no loads
  // native GEMM, rebiased operands: per-A-row and per-B-tensor power-of-two
  // factors (nullable), and a device flag that makes the launch a no-op
  const float *fa = nullptr, *fb = nullptr;
  const int* skip_if = nullptr;
  // emulated GEMM: a device flag without which the launch is a no-op (nullable)
  const int* run_if = nullptr;
  // epilogue quantisation: the scale format of the quantised result (the
  // emulated GEMM uses fmt), and whether the launch zeroes qamax first
  // (false: qamax is max-ed into as the caller left it)
  int fmt_out = 0;
  bool zero_qamax = true;
  // native GEMM, two-window rebiased A (nullable): A's low-window codes, the
  // high-window codes in As and their per-row factor in fa, the low window's
  // factor fa * 2^-14
  const uint8_t* As_lo = nullptr;
};

// The driver's cuTensorMapEncodeTiled (looked up once through the runtime);
// null when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn();

// Returns cudaErrorNotSupported when the driver entry point for tensor maps
// is missing.
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st);

// The native NVFP4 GEMM (gemm_native.cu): UE4M3-scaled E2M1 operands on the
// tensor cores' block-scaled MMA.  K % 256 == 0.
cudaError_t launch_gemm_nvfp4(const GemmArgs& a, cudaStream_t st);

// UE5M3 scale codes [rows, nb] -> UE4M3 codes and power-of-two factors
// (rebias.cu): per row (factor[rows]) or for the whole tensor (factor[1]);
// ORs 1 into *nofit when a group does not fit.  nb % 16 == 0.
cudaError_t launch_rebias(const uint8_t* scales, int64_t rows, int64_t nb, bool per_row, uint8_t* out,
                          float* factor, int* nofit, cudaStream_t st);

// The same per row with two windows (rebias.cu): high-window codes and
// factor (out_hi, f_hi), low-window codes and factor (out_lo, f_lo).
cudaError_t launch_rebias2(const uint8_t* scales, int64_t rows, int64_t nb, uint8_t* out_hi, uint8_t* out_lo,
                           float* f_hi, float* f_lo, int* nofit, cudaStream_t st);

}  // namespace fp4q
