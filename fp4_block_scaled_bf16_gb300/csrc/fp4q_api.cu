// fp4q_api.cu -- the extern "C" entry points of libfp4q.so (declared and
// documented in include/fp4q.h): argument validation, device status word,
// dispatch to the kernel launchers.  No entry point allocates memory.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "fp4q.h"
#include "fp4q_device.cuh"
#include "fp4q_launch.h"

// Built with -DFP4Q_NVTX (FP4Q_NVTX=1 in the environment of the build), every
// entry point is an NVTX range named after it, for timeline profilers; the
// default build has none.
#ifdef FP4Q_NVTX
#include <nvtx3/nvToolsExt.h>
namespace {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace
#define FP4Q_RANGE(name) NvtxRange fp4q_nvtx_range_(name)
#else
#define FP4Q_RANGE(name) ((void)0)
#endif

namespace {

// Latched by kernels (non-finite input, bounded-wait timeout) with atomicOr;
// read and cleared by fp4q_get_device_status.
__device__ int g_status_word;

__global__ void clear_status_kernel(int* word, int bits) { atomicAnd(word, ~bits); }

int* status_ptr() {
  // One address per device; looked up on each call (cheap) so that a caller
  // switching devices gets the right copy.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// scalars (amax, tensor scales) need their natural 4-byte alignment, the
// stats counters 8 bytes
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

fp4q_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA; }

float scale_max_host(fp4q_scale_fmt f) { return f == FP4Q_SCALE_UE5M3 ? 114688.0f : 448.0f; }

bool valid_fmt(int f) { return f == FP4Q_SCALE_UE5M3 || f == FP4Q_SCALE_UE4M3; }

}  // namespace

extern "C" {

const char* fp4q_status_string(fp4q_status s) {
  switch (s) {
    case FP4Q_OK: return "ok";
    case FP4Q_ERR_ARG: return "invalid argument (null pointer or unknown enum)";
    case FP4Q_ERR_SHAPE: return "unsupported shape";
    case FP4Q_ERR_ALIGN: return "misaligned pointer";
    case FP4Q_ERR_CUDA: return "CUDA error";
    case FP4Q_ERR_NONFINITE: return "non-finite input element";
    case FP4Q_ERR_TIMEOUT: return "device pipeline wait timed out";
  }
  return "unknown status";
}

fp4q_status fp4q_amax(const void* in_bf16, int64_t n, float* out_amax, void* stream) {
  FP4Q_RANGE("fp4q_amax");
  if (!out_amax || n < 0 || (n > 0 && !in_bf16)) return FP4Q_ERR_ARG;
  if ((n > 0 && !aligned16(in_bf16)) || !aligned4(out_amax)) return FP4Q_ERR_ALIGN;
  int* st = status_ptr();
  if (!st) return FP4Q_ERR_CUDA;
  return from_cuda(fp4q::launch_amax(in_bf16, n, out_amax, st, static_cast<cudaStream_t>(stream)));
}

fp4q_status fp4q_tensor_scale(const float* amax, fp4q_scale_fmt fmt, float headroom, float* out_scale,
                              void* stream) {
  FP4Q_RANGE("fp4q_tensor_scale");
  if (!amax || !out_scale || !valid_fmt(fmt)) return FP4Q_ERR_ARG;
  // headroom must be a power of two >= 1 so that 6 * Smax / H is exact
  int e = 0;
  if (!(headroom >= 1.0f) || frexpf(headroom, &e) != 0.5f) return FP4Q_ERR_ARG;
  if (!aligned4(amax) || !aligned4(out_scale)) return FP4Q_ERR_ALIGN;
  const float denom = (6.0f * scale_max_host(fmt)) / headroom;
  return from_cuda(fp4q::launch_tensor_scale(amax, denom, out_scale, static_cast<cudaStream_t>(stream)));
}

fp4q_status fp4q_quantize(const void* in_bf16, int64_t rows, int64_t cols, fp4q_axis axis,
                          fp4q_scale_fmt fmt, const float* tensor_scale, fp4q_rounding rnd,
                          uint64_t seed, uint8_t* out_payload_row, uint8_t* out_scales_row,
                          uint8_t* out_payload_col, uint8_t* out_scales_col, fp4q_stats* out_stats,
                          float* out_amax, void* stream) {
  FP4Q_RANGE("fp4q_quantize");
  if (axis != FP4Q_AXIS_ROW && axis != FP4Q_AXIS_COL && axis != FP4Q_AXIS_BOTH && axis != FP4Q_AXIS_BOTH_2D)
    return FP4Q_ERR_ARG;
  if (!valid_fmt(fmt) || (rnd != FP4Q_RNE && rnd != FP4Q_SR) || !tensor_scale) return FP4Q_ERR_ARG;
  if (rows < 0 || cols < 0 || rows % 16 || cols % 16) return FP4Q_ERR_SHAPE;
  if (axis != FP4Q_AXIS_ROW) {   // the tile kernels number 128 x 128 tiles in 32 bits
    const int64_t tr = (rows + 127) / 128, tc = (cols + 127) / 128;
    if (tc > 0 && tr > INT32_MAX / tc) return FP4Q_ERR_SHAPE;
  }
  const bool row = axis != FP4Q_AXIS_COL, col = axis != FP4Q_AXIS_ROW;
  const bool empty = rows == 0 || cols == 0;
  if (!empty) {
    if (!in_bf16) return FP4Q_ERR_ARG;
    if (row && (!out_payload_row || !out_scales_row)) return FP4Q_ERR_ARG;
    if (col && (!out_payload_col || !out_scales_col)) return FP4Q_ERR_ARG;
    if (!aligned16(in_bf16)) return FP4Q_ERR_ALIGN;
    if (row && (!aligned16(out_payload_row) || !aligned16(out_scales_row))) return FP4Q_ERR_ALIGN;
    if (col && (!aligned16(out_payload_col) || !aligned16(out_scales_col))) return FP4Q_ERR_ALIGN;
  }
  if (!aligned4(tensor_scale) || (out_stats && !aligned8(out_stats)) ||
      (out_amax && !aligned4(out_amax)))
    return FP4Q_ERR_ALIGN;
  int* st = status_ptr();
  if (!st) return FP4Q_ERR_CUDA;
  fp4q::QuantArgs a;
  a.in = in_bf16;
  a.rows = rows;
  a.cols = cols;
  a.axis = (int)axis;
  a.fmt = (int)fmt;
  a.tscale = tensor_scale;
  a.sr = rnd == FP4Q_SR;
  a.seed = seed;
  a.pay_row = out_payload_row;
  a.sc_row = out_scales_row;
  a.pay_col = out_payload_col;
  a.sc_col = out_scales_col;
  a.stats = reinterpret_cast<fp4q::StatsDev*>(out_stats);
  a.amax_out = out_amax;
  a.status = st;
  return from_cuda(fp4q::launch_quantize(a, static_cast<cudaStream_t>(stream)));
}

fp4q_status fp4q_dequantize(const uint8_t* payload, const uint8_t* scales, int64_t rows, int64_t cols,
                            fp4q_scale_fmt fmt, const float* tensor_scale, void* out, int out_is_f32,
                            void* stream) {
  FP4Q_RANGE("fp4q_dequantize");
  if (!valid_fmt(fmt) || !tensor_scale) return FP4Q_ERR_ARG;
  if (rows < 0 || cols < 0 || rows % 16 || cols % 16) return FP4Q_ERR_SHAPE;
  if (rows > 0 && cols > 0) {
    if (!payload || !scales || !out) return FP4Q_ERR_ARG;
    if (!aligned16(payload) || !aligned16(scales) || !aligned16(out)) return FP4Q_ERR_ALIGN;
  }
  if (!aligned4(tensor_scale)) return FP4Q_ERR_ALIGN;
  return from_cuda(fp4q::launch_dequantize(payload, scales, rows, cols, (int)fmt, tensor_scale, out,
                                           out_is_f32 != 0, static_cast<cudaStream_t>(stream)));
}

// Shared by fp4q_gemm and fp4q_gemm_quantize: validation of the operands and
// the launch arguments; q* are the epilogue-quantisation outputs (or null).
static fp4q_status gemm_common(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                               const uint8_t* B, const uint8_t* B_scales, const float* B_tscale,
                               int64_t M, int64_t N, int64_t K, fp4q_scale_fmt fmt, void* out,
                               int out_is_f32, const float* c_tscale, uint8_t* qpay, uint8_t* qsc,
                               float* qamax, void* stream, const int* run_if = nullptr,
                               bool zero_qamax = true) {
  if (!valid_fmt(fmt)) return FP4Q_ERR_ARG;
  if (run_if && !aligned4(run_if)) return FP4Q_ERR_ALIGN;
  if (M < 0 || N < 0 || K < 0 || K % 64 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
    return FP4Q_ERR_SHAPE;
  if ((M + 255) / 256 > 65535) return FP4Q_ERR_SHAPE;   // 256-row tiles on the grid's y dimension
  if (qpay && N % 32) return FP4Q_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (qamax && !aligned4(qamax)) return FP4Q_ERR_ALIGN;
  if (M == 0 || N == 0) {
    if (qamax && zero_qamax) return from_cuda(cudaMemsetAsync(qamax, 0, sizeof(float), st));
    return FP4Q_OK;
  }
  if (!out && !qpay) return FP4Q_ERR_ARG;
  if (out && !aligned16(out)) return FP4Q_ERR_ALIGN;
  if (qpay) {
    if (!qsc || !c_tscale) return FP4Q_ERR_ARG;
    if (!aligned16(qpay) || !aligned16(qsc) || !aligned4(c_tscale)) return FP4Q_ERR_ALIGN;
  }
  if (K == 0) {   // C = 0: zero output, zero payload (+0 nibbles), zero scale codes, amax 0
    cudaError_t e = cudaSuccess;
    if (out) e = cudaMemsetAsync(out, 0, (size_t)M * N * (out_is_f32 ? 4 : 2), st);
    if (e == cudaSuccess && qpay) e = cudaMemsetAsync(qpay, 0, (size_t)M * N / 2, st);
    if (e == cudaSuccess && qpay) e = cudaMemsetAsync(qsc, 0, (size_t)M * N / 16, st);
    if (e == cudaSuccess && qamax && zero_qamax) e = cudaMemsetAsync(qamax, 0, sizeof(float), st);
    return from_cuda(e);
  }
  if (!A || !A_scales || !A_tscale || !B || !B_scales || !B_tscale) return FP4Q_ERR_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(A_scales) || !aligned16(B_scales) ||
      !aligned4(A_tscale) || !aligned4(B_tscale))
    return FP4Q_ERR_ALIGN;
  int* status = status_ptr();
  if (!status) return FP4Q_ERR_CUDA;
  fp4q::GemmArgs a;
  a.run_if = run_if;
  a.zero_qamax = zero_qamax;
  a.TC = c_tscale;
  a.qpay = qpay;
  a.qsc = qsc;
  a.qamax = qamax;
  a.A = A;
  a.As = A_scales;
  a.B = B;
  a.Bs = B_scales;
  a.TA = A_tscale;
  a.TB = B_tscale;
  a.M = M;
  a.N = N;
  a.K = K;
  a.fmt = (int)fmt;
  a.out = out;
  a.out_f32 = out_is_f32 != 0;
  a.status = status;
  // Every pipeline wait gives up after about 2 s (4e9 cycles) unless the
  // test hooks below shorten it; FP4Q_TEST_GEMM_SKIP_LOADS makes the producer
  // issue no loads so that the consumers' waits run out (failure-path test).
  a.wait_cycles = 4000000000LL;
  a.skip_loads = false;
  if (const char* e = getenv("FP4Q_TEST_GEMM_WAIT_CYCLES")) {
    const long long v = atoll(e);
    if (v > 0) a.wait_cycles = v;
  }
  if (const char* e = getenv("FP4Q_TEST_GEMM_SKIP_LOADS")) a.skip_loads = atoi(e) != 0;
  return from_cuda(fp4q::launch_gemm(a, st));
}

fp4q_status fp4q_gemm(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale, const uint8_t* B,
                      const uint8_t* B_scales, const float* B_tscale, int64_t M, int64_t N, int64_t K,
                      fp4q_scale_fmt fmt, void* out, int out_is_f32, void* stream) {
  FP4Q_RANGE("fp4q_gemm");
  return gemm_common(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, out, out_is_f32,
                     nullptr, nullptr, nullptr, nullptr, stream);
}

fp4q_status fp4q_gemm_quantize(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                               const uint8_t* B, const uint8_t* B_scales, const float* B_tscale,
                               int64_t M, int64_t N, int64_t K, fp4q_scale_fmt fmt,
                               const float* c_tscale, void* out_bf16, uint8_t* out_payload,
                               uint8_t* out_scales, float* out_amax, void* stream) {
  FP4Q_RANGE("fp4q_gemm_quantize");
  if (M > 0 && N > 0 && !out_payload) return FP4Q_ERR_ARG;
  return gemm_common(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, out_bf16, 0,
                     c_tscale, out_payload, out_scales, out_amax, stream);
}

fp4q_status fp4q_gemm_if(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale, const uint8_t* B,
                         const uint8_t* B_scales, const float* B_tscale, int64_t M, int64_t N, int64_t K,
                         fp4q_scale_fmt fmt, const int* run_if_set, void* out, int out_is_f32, void* stream) {
  FP4Q_RANGE("fp4q_gemm_if");
  if (!run_if_set) return FP4Q_ERR_ARG;
  return gemm_common(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, out, out_is_f32,
                     nullptr, nullptr, nullptr, nullptr, stream, run_if_set);
}

fp4q_status fp4q_gemm_quantize_if(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                                  const uint8_t* B, const uint8_t* B_scales, const float* B_tscale, int64_t M,
                                  int64_t N, int64_t K, fp4q_scale_fmt fmt, const int* run_if_set,
                                  const float* c_tscale, void* out_bf16, uint8_t* out_payload,
                                  uint8_t* out_scales, float* out_amax, void* stream) {
  FP4Q_RANGE("fp4q_gemm_quantize_if");
  if (!run_if_set) return FP4Q_ERR_ARG;
  if (M > 0 && N > 0 && !out_payload) return FP4Q_ERR_ARG;
  return gemm_common(A, A_scales, A_tscale, B, B_scales, B_tscale, M, N, K, fmt, out_bf16, 0, c_tscale,
                     out_payload, out_scales, out_amax, stream, run_if_set, /*zero_qamax=*/false);
}

}  // extern "C"

namespace {

fp4q_status gemm_native_common(const uint8_t* A, const uint8_t* A_scales, const float* A_factor,
                               const float* A_tscale, const uint8_t* B, const uint8_t* B_scales,
                               const float* B_factor, const float* B_tscale, int64_t M, int64_t N,
                               int64_t K, const int* skip_if, void* out, int out_is_f32, void* stream,
                               const float* c_tscale = nullptr, uint8_t* qpay = nullptr, uint8_t* qsc = nullptr,
                               float* qamax = nullptr, int qfmt = 0, const uint8_t* A_scales_lo = nullptr) {
  if (M < 0 || N < 0 || K < 0 || K % 256 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
    return FP4Q_ERR_SHAPE;
  if ((M + 127) / 128 > 65535) return FP4Q_ERR_SHAPE;   // 128-row tiles on the grid's y dimension
  if (qpay && N % 32) return FP4Q_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (qamax && !aligned4(qamax)) return FP4Q_ERR_ALIGN;
  if (M == 0 || N == 0) return FP4Q_OK;
  if (!out && !qpay) return FP4Q_ERR_ARG;
  if (out && !aligned16(out)) return FP4Q_ERR_ALIGN;
  if (qpay) {
    if (!qsc || !c_tscale) return FP4Q_ERR_ARG;
    if (!aligned16(qpay) || !aligned16(qsc) || !aligned4(c_tscale)) return FP4Q_ERR_ALIGN;
  }
  if (K == 0) {   // C = 0: zero output, payload and scale codes; qamax (max-ed into) unchanged
    cudaError_t e = cudaSuccess;
    if (out) e = cudaMemsetAsync(out, 0, (size_t)M * N * (out_is_f32 ? 4 : 2), st);
    if (e == cudaSuccess && qpay) e = cudaMemsetAsync(qpay, 0, (size_t)M * N / 2, st);
    if (e == cudaSuccess && qpay) e = cudaMemsetAsync(qsc, 0, (size_t)M * N / 16, st);
    return from_cuda(e);
  }
  if (!A || !A_scales || !A_tscale || !B || !B_scales || !B_tscale) return FP4Q_ERR_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(A_scales) || !aligned16(B_scales) ||
      !aligned16(A_scales_lo) || !aligned4(A_tscale) || !aligned4(B_tscale) || !aligned4(A_factor) ||
      !aligned4(B_factor) || !aligned4(skip_if))
    return FP4Q_ERR_ALIGN;
  int* status = status_ptr();
  if (!status) return FP4Q_ERR_CUDA;
  fp4q::GemmArgs a;
  a.A = A;
  a.As = A_scales;
  a.B = B;
  a.Bs = B_scales;
  a.TA = A_tscale;
  a.TB = B_tscale;
  a.fa = A_factor;
  a.fb = B_factor;
  a.skip_if = skip_if;
  a.M = M;
  a.N = N;
  a.K = K;
  a.fmt = FP4Q_SCALE_UE4M3;
  a.out = out;
  a.out_f32 = out_is_f32 != 0;
  a.status = status;
  a.TC = c_tscale;
  a.qpay = qpay;
  a.qsc = qsc;
  a.qamax = qamax;
  a.fmt_out = qfmt;
  a.As_lo = A_scales_lo;
  a.wait_cycles = 4000000000LL;   // about 2 s per wait, as fp4q_gemm
  a.skip_loads = false;
  if (const char* e = getenv("FP4Q_TEST_GEMM_WAIT_CYCLES")) {
    const long long v = atoll(e);
    if (v > 0) a.wait_cycles = v;
  }
  if (const char* e = getenv("FP4Q_TEST_GEMM_SKIP_LOADS")) a.skip_loads = atoi(e) != 0;
  return from_cuda(fp4q::launch_gemm_nvfp4(a, st));
}

}  // namespace

extern "C" {

fp4q_status fp4q_gemm_nvfp4(const uint8_t* A, const uint8_t* A_scales, const float* A_tscale,
                            const uint8_t* B, const uint8_t* B_scales, const float* B_tscale, int64_t M,
                            int64_t N, int64_t K, void* out, int out_is_f32, void* stream) {
  FP4Q_RANGE("fp4q_gemm_nvfp4");
  return gemm_native_common(A, A_scales, nullptr, A_tscale, B, B_scales, nullptr, B_tscale, M, N, K, nullptr,
                            out, out_is_f32, stream);
}

fp4q_status fp4q_gemm_nvfp4_rebiased(const uint8_t* A, const uint8_t* A_scales4, const float* A_factor,
                                     const float* A_tscale, const uint8_t* B, const uint8_t* B_scales4,
                                     const float* B_factor, const float* B_tscale, int64_t M, int64_t N,
                                     int64_t K, const int* skip_if_set, void* out, int out_is_f32,
                                     void* stream) {
  FP4Q_RANGE("fp4q_gemm_nvfp4_rebiased");
  if (M > 0 && N > 0 && K > 0 && (!A_factor || !B_factor)) return FP4Q_ERR_ARG;
  return gemm_native_common(A, A_scales4, A_factor, A_tscale, B, B_scales4, B_factor, B_tscale, M, N, K,
                            skip_if_set, out, out_is_f32, stream);
}

fp4q_status fp4q_gemm_nvfp4_rebiased_quantize(const uint8_t* A, const uint8_t* A_scales4, const float* A_factor,
                                              const float* A_tscale, const uint8_t* B, const uint8_t* B_scales4,
                                              const float* B_factor, const float* B_tscale, int64_t M, int64_t N,
                                              int64_t K, const int* skip_if_set, fp4q_scale_fmt fmt,
                                              const float* c_tscale, void* out_bf16, uint8_t* out_payload,
                                              uint8_t* out_scales, float* out_amax, void* stream) {
  FP4Q_RANGE("fp4q_gemm_nvfp4_rebiased_quantize");
  if (!valid_fmt(fmt)) return FP4Q_ERR_ARG;
  if (M > 0 && N > 0 && !out_payload) return FP4Q_ERR_ARG;
  if (M > 0 && N > 0 && K > 0 && (!A_factor || !B_factor)) return FP4Q_ERR_ARG;
  return gemm_native_common(A, A_scales4, A_factor, A_tscale, B, B_scales4, B_factor, B_tscale, M, N, K,
                            skip_if_set, out_bf16, 0, stream, c_tscale, out_payload, out_scales, out_amax,
                            (int)fmt);
}

fp4q_status fp4q_gemm_nvfp4_two_windows(const uint8_t* A, const uint8_t* A_scales_hi, const uint8_t* A_scales_lo,
                                        const float* A_factor_hi, const float* A_tscale, const uint8_t* B,
                                        const uint8_t* B_scales4, const float* B_factor, const float* B_tscale,
                                        int64_t M, int64_t N, int64_t K, const int* skip_if_set, void* out,
                                        int out_is_f32, void* stream) {
  FP4Q_RANGE("fp4q_gemm_nvfp4_two_windows");
  if (M > 0 && N > 0 && K > 0 && (!A_factor_hi || !B_factor || !A_scales_lo)) return FP4Q_ERR_ARG;
  return gemm_native_common(A, A_scales_hi, A_factor_hi, A_tscale, B, B_scales4, B_factor, B_tscale, M, N, K,
                            skip_if_set, out, out_is_f32, stream, nullptr, nullptr, nullptr, nullptr, 0,
                            A_scales_lo);
}

fp4q_status fp4q_rebias_scales_two_windows(const uint8_t* scales, int64_t rows, int64_t nblocks, uint8_t* out_hi,
                                           uint8_t* out_lo, float* out_factor_hi, float* out_factor_lo,
                                           int* inout_nofit, void* stream) {
  FP4Q_RANGE("fp4q_rebias_scales_two_windows");
  if (rows < 0 || nblocks < 0 || nblocks % 16 || nblocks > INT32_MAX) return FP4Q_ERR_SHAPE;
  if (!inout_nofit || (rows > 0 && (!out_factor_hi || !out_factor_lo))) return FP4Q_ERR_ARG;
  if (rows > 0 && nblocks > 0 && (!scales || !out_hi || !out_lo)) return FP4Q_ERR_ARG;
  if (!aligned16(scales) || !aligned16(out_hi) || !aligned16(out_lo) || !aligned4(out_factor_hi) ||
      !aligned4(out_factor_lo) || !aligned4(inout_nofit))
    return FP4Q_ERR_ALIGN;
  if (rows > 0 && nblocks > 0) {
    const int64_t n = rows * nblocks;
    auto overlap = [n](const void* x, const void* y) {
      const uint8_t *a = static_cast<const uint8_t*>(x), *b = static_cast<const uint8_t*>(y);
      return a < b + n && b < a + n;
    };
    // the input is read after outputs are written; the two outputs are written together
    if (overlap(scales, out_hi) || overlap(scales, out_lo) || overlap(out_hi, out_lo)) return FP4Q_ERR_ARG;
  }
  return from_cuda(fp4q::launch_rebias2(scales, rows, nblocks, out_hi, out_lo, out_factor_hi, out_factor_lo,
                                        inout_nofit, static_cast<cudaStream_t>(stream)));
}

fp4q_status fp4q_rebias_scales(const uint8_t* scales, int64_t rows, int64_t nblocks, int per_row,
                               uint8_t* out_scales, float* out_factor, int* inout_nofit, void* stream) {
  FP4Q_RANGE("fp4q_rebias_scales");
  if (rows < 0 || nblocks < 0 || nblocks % 16 || nblocks > INT32_MAX) return FP4Q_ERR_SHAPE;
  if (!out_factor || !inout_nofit) return FP4Q_ERR_ARG;
  if (rows > 0 && nblocks > 0 && (!scales || !out_scales)) return FP4Q_ERR_ARG;
  if (!aligned16(scales) || !aligned16(out_scales) || !aligned4(out_factor) || !aligned4(inout_nofit))
    return FP4Q_ERR_ALIGN;
  if (scales && out_scales && rows > 0 && nblocks > 0) {
    const uint8_t *a0 = scales, *a1 = scales + rows * nblocks, *b0 = out_scales, *b1 = out_scales + rows * nblocks;
    if (a0 < b1 && b0 < a1) return FP4Q_ERR_ARG;   // the input is read after outputs are written
  }
  return from_cuda(fp4q::launch_rebias(scales, rows, nblocks, per_row != 0, out_scales, out_factor,
                                       inout_nofit, static_cast<cudaStream_t>(stream)));
}

fp4q_status fp4q_get_device_status(int* out, void* stream) {
  FP4Q_RANGE("fp4q_get_device_status");
  if (!out) return FP4Q_ERR_ARG;
  int* st = status_ptr();
  if (!st) return FP4Q_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  // stream-ordered read of the word, then a wait on this stream only
  if (cudaMemcpyAsync(&v, st, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FP4Q_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FP4Q_ERR_CUDA;
  if (v) {
    // clear only the bits reported here, atomically: a condition latched by
    // another stream in the meantime stays set for the next read
    clear_status_kernel<<<1, 1, 0, s>>>(st, v);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return FP4Q_ERR_CUDA;
  }
  *out = (v & fp4q::kStatusTimeout) ? FP4Q_ERR_TIMEOUT
         : (v & fp4q::kStatusNonFinite) ? FP4Q_ERR_NONFINITE
                                        : FP4Q_OK;
  return FP4Q_OK;
}

}  // extern "C"
