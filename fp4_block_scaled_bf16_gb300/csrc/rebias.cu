// rebias.cu -- UE5M3 block-scale codes re-expressed as UE4M3 codes times a
// power of two, so that a UE5M3-scaled GEMM can run exactly on the tensor
// cores' UE4M3 block-scaled MMA (gemm_native.cu) with the power of two applied
// to its result.
//
// Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
// Abstract -- UE5M3 is emulated because the tensor cores take only E4M3/E8M0
// block scales.  The two scale formats share their 3 mantissa bits: a group of
// UE5M3 scales whose non-zero values lie in 14 consecutive binades
// [e_top - 13, e_top] equals f * (UE4M3 values) with f = 2^(e_top - 7), the
// largest landing in UE4M3's exponent field 14.  Groups:
//   per row   -- e_top is the row's largest binade (one warp per row: a
//                warp-wide max and min over the row's codes, then the codes);
//   per tensor -- e_top = 16, the binade of the largest finite UE5M3 scale,
//                where the tensor scale puts the tensor's amax: f = 2^9 and
//                every code is checked on its own.
// A group that does not fit sets *nofit (never cleared here); its codes and
// factor are then unspecified.
// Two windows per row (rebias_rows2_kernel): the 14 binades under the row's
// top as above (factor f_hi = 2^(e_top - 7)) and the 14 below them
// [e_top - 27, e_top - 14] (factor f_lo = 2^(e_top - 21) = f_hi 2^-14), each
// code in exactly one of the two outputs and zero in the other; a code below
// both windows sets *nofit and is zero in both.
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp4q_device.cuh"
#include "fp4q_launch.h"

namespace fp4q {
namespace rebias {

constexpr int kNone = -1000;   // binade of "no non-zero scale"

// Binade e = floor(log2 v) of a non-zero UE5M3 code and its 3 mantissa bits
// once normalised (a subnormal m/8 * 2^-14 has at most 3 significant bits).
__device__ __forceinline__ int binade(uint32_t c, uint32_t& mn) {
  const uint32_t E = c >> 3, m = c & 7u;
  if (E != 0) {
    mn = m;
    return (int)E - 15;
  }
  const int lz = 31 - __clz((int)m);   // floor(log2 m), m in 1..7
  mn = (m << (3 - lz)) & 7u;
  return lz - 17;
}

// The UE4M3 code of v / 2^(etop - 7) for a non-zero UE5M3 code; 0 stays 0.
// Outside the group's window the exponent field is clamped (the group does
// not fit and its codes are unspecified).
__device__ __forceinline__ uint32_t recode(uint32_t c, int etop) {
  if (c == 0) return 0;
  uint32_t mn;
  const int e = binade(c, mn);
  const int f = min(max(e - etop + 14, 0), 15);
  return ((uint32_t)f << 3) | mn;
}

__device__ __forceinline__ float pow2(int k) { return __int_as_float((k + 127) << 23); }

__device__ __forceinline__ uint32_t word_at(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Four codes per 32-bit word.  Codes order like their values (zero lowest),
// so a group's largest and smallest non-zero binades are those of its
// largest and smallest non-zero codes: a bytewise max, and a bytewise min
// with the zero bytes raised to 0xFF (not a value).  When every non-zero code
// of a fitting group is normal, the re-encode is the same for each of them --
// exponent field E -> E - (E_top - 14), mantissa kept -- one bytewise add per
// word, with the zero bytes masked back to zero.
__device__ __forceinline__ uint32_t max_byte(uint32_t v) {
  return max(max(v & 0xFFu, (v >> 8) & 0xFFu), max((v >> 16) & 0xFFu, v >> 24));
}
__device__ __forceinline__ uint32_t min_byte(uint32_t v) {
  return min(min(v & 0xFFu, (v >> 8) & 0xFFu), min((v >> 16) & 0xFFu, v >> 24));
}
__device__ __forceinline__ uint4 add_nonzero4(const uint4& v, uint32_t k) {
  return make_uint4(__vadd4(v.x, k) & __vcmpne4(v.x, 0u), __vadd4(v.y, k) & __vcmpne4(v.y, 0u),
                    __vadd4(v.z, k) & __vcmpne4(v.z, 0u), __vadd4(v.w, k) & __vcmpne4(v.w, 0u));
}

// One warp per row (grid-stride over rows); nb % 16 == 0, rows 16-byte aligned.
__global__ void __launch_bounds__(256) rebias_rows_kernel(const uint8_t* __restrict__ in, int64_t rows, int nb,
                                                          uint8_t* __restrict__ out, float* __restrict__ factor,
                                                          int* nofit) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int chunks = nb >> 4;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
    const uint4* src = reinterpret_cast<const uint4*>(in + r * nb);
    uint32_t vmax = 0u, vmin = 0xFFFFFFFFu;
    for (int j = lane; j < chunks; j += 32) {
      const uint4 v = __ldg(src + j);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t word = word_at(v, w);
        vmax = __vmaxu4(vmax, word);
        vmin = __vminu4(vmin, word | ~__vcmpne4(word, 0u));
      }
    }
    const uint32_t cmax = __reduce_max_sync(0xFFFFFFFFu, max_byte(vmax));
    const uint32_t cmin = __reduce_min_sync(0xFFFFFFFFu, min_byte(vmin));
    uint32_t mn;
    const bool any = cmax != 0u;
    const int emax = any ? binade(cmax, mn) : kNone;
    if (lane == 0) {
      factor[r] = any ? pow2(emax - 7) : 1.0f;
      if (any && binade(cmin, mn) < emax - 13) atomicOr(nofit, 1);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + r * nb);
    if (cmin >= 8u) {   // every non-zero code normal (an all-zero row: cmin = 0xFF)
      const uint32_t k = ((14u - (cmax >> 3)) << 3 & 0xFFu) * 0x01010101u;
      for (int j = lane; j < chunks; j += 32) dst[j] = add_nonzero4(__ldg(src + j), k);
    } else {            // subnormal codes: normalised code by code
      for (int j = lane; j < chunks; j += 32) {
        const uint4 v = __ldg(src + j);
        uint32_t o[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t word = word_at(v, w);
          o[w] = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b) o[w] |= recode((word >> (8 * b)) & 0xFFu, emax) << (8 * b);
        }
        dst[j] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// The whole tensor with the fixed window (binades 3..16, factor 2^9): a
// non-zero code fits iff its exponent field is at least 18, and then its
// field drops by 17 (the code by 0x88); grid-stride over 16-code chunks.
__global__ void __launch_bounds__(256) rebias_tensor_kernel(const uint4* __restrict__ in, int64_t chunks,
                                                            uint4* __restrict__ out, float* __restrict__ factor,
                                                            int* nofit) {
  constexpr int kTop = 16;
  if (blockIdx.x == 0 && threadIdx.x == 0) factor[0] = pow2(kTop - 7);
  uint32_t bad = 0u;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < chunks; j += stride) {
    const uint4 v = __ldg(in + j);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t word = word_at(v, w);
      bad |= __vcmpltu4(word, 0x90909090u) & __vcmpne4(word, 0u);   // binade below 3
    }
    out[j] = add_nonzero4(v, 0x78787878u);   // - 0x88 per byte
  }
  if (__any_sync(0xFFFFFFFFu, bad != 0u) && (threadIdx.x & 31) == 0) atomicOr(nofit, 1);
}

// The UE4M3 codes of a non-zero UE5M3 code in the two windows of a row with
// top binade etop (exactly one of hi, lo non-zero, or neither below both).
__device__ __forceinline__ void recode2(uint32_t c, int etop, uint32_t& hi, uint32_t& lo) {
  hi = lo = 0;
  if (c == 0) return;
  uint32_t mn;
  const int e = binade(c, mn);
  if (e >= etop - 13)
    hi = ((uint32_t)(e - etop + 14) << 3) | mn;
  else if (e >= etop - 27)
    lo = ((uint32_t)(e - etop + 28) << 3) | mn;
}

// Two windows per row, one warp per row (grid-stride); layout as
// rebias_rows_kernel.  When every non-zero code is normal, a code's window is
// decided by a bytewise compare of the code against the first code of the
// window (E_top - 13 and E_top - 27 exponent fields, clamped at 0), and each
// window's re-encode is one bytewise add: fields drop by E_top - 14 (high)
// and E_top - 28 (low).
__global__ void __launch_bounds__(256) rebias_rows2_kernel(const uint8_t* __restrict__ in, int64_t rows, int nb,
                                                           uint8_t* __restrict__ out_hi,
                                                           uint8_t* __restrict__ out_lo, float* __restrict__ f_hi,
                                                           float* __restrict__ f_lo, int* nofit) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int chunks = nb >> 4;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
    const uint4* src = reinterpret_cast<const uint4*>(in + r * nb);
    uint32_t vmax = 0u, vmin = 0xFFFFFFFFu;
    for (int j = lane; j < chunks; j += 32) {
      const uint4 v = __ldg(src + j);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t word = word_at(v, w);
        vmax = __vmaxu4(vmax, word);
        vmin = __vminu4(vmin, word | ~__vcmpne4(word, 0u));
      }
    }
    const uint32_t cmax = __reduce_max_sync(0xFFFFFFFFu, max_byte(vmax));
    const uint32_t cmin = __reduce_min_sync(0xFFFFFFFFu, min_byte(vmin));
    uint32_t mn;
    const bool any = cmax != 0u;
    const int emax = any ? binade(cmax, mn) : kNone;
    if (lane == 0) {
      f_hi[r] = any ? pow2(emax - 7) : 1.0f;
      f_lo[r] = any ? pow2(emax - 21) : pow2(-14);
      if (any && binade(cmin, mn) < emax - 27) atomicOr(nofit, 1);
    }
    uint4* dh = reinterpret_cast<uint4*>(out_hi + r * nb);
    uint4* dl = reinterpret_cast<uint4*>(out_lo + r * nb);
    if (cmin >= 8u) {   // every non-zero code normal (an all-zero row: cmin = 0xFF)
      const int et = (int)(cmax >> 3);
      const uint32_t thi = (uint32_t)(max(et - 13, 0) << 3) * 0x01010101u;
      const uint32_t tlo = (uint32_t)(max(et - 27, 0) << 3) * 0x01010101u;
      const uint32_t khi = ((uint32_t)(14 - et) << 3 & 0xFFu) * 0x01010101u;
      const uint32_t klo = ((uint32_t)(28 - et) << 3 & 0xFFu) * 0x01010101u;
      for (int j = lane; j < chunks; j += 32) {
        const uint4 v = __ldg(src + j);
        uint32_t h[4], l[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t word = word_at(v, w);
          const uint32_t nz = __vcmpne4(word, 0u);
          const uint32_t inhi = __vcmpgeu4(word, thi) & nz;
          const uint32_t inlo = __vcmpgeu4(word, tlo) & nz & ~inhi;
          h[w] = __vadd4(word, khi) & inhi;
          l[w] = __vadd4(word, klo) & inlo;
        }
        dh[j] = make_uint4(h[0], h[1], h[2], h[3]);
        dl[j] = make_uint4(l[0], l[1], l[2], l[3]);
      }
    } else {            // subnormal codes: normalised code by code
      for (int j = lane; j < chunks; j += 32) {
        const uint4 v = __ldg(src + j);
        uint32_t h[4], l[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t word = word_at(v, w);
          h[w] = l[w] = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t ch, cl;
            recode2((word >> (8 * b)) & 0xFFu, emax, ch, cl);
            h[w] |= ch << (8 * b);
            l[w] |= cl << (8 * b);
          }
        }
        dh[j] = make_uint4(h[0], h[1], h[2], h[3]);
        dl[j] = make_uint4(l[0], l[1], l[2], l[3]);
      }
    }
  }
}

}  // namespace rebias

cudaError_t launch_rebias2(const uint8_t* scales, int64_t rows, int64_t nb, uint8_t* out_hi, uint8_t* out_lo,
                           float* f_hi, float* f_lo, int* nofit, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (rows + 7) / 8;   // eight rows (warps) per 256-thread block
  const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  rebias::rebias_rows2_kernel<<<grid, 256, 0, st>>>(scales, rows, (int)nb, out_hi, out_lo, f_hi, f_lo, nofit);
  return cudaGetLastError();
}

cudaError_t launch_rebias(const uint8_t* scales, int64_t rows, int64_t nb, bool per_row, uint8_t* out,
                          float* factor, int* nofit, cudaStream_t st) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (per_row) {
    if (rows == 0) return cudaSuccess;
    const int64_t want = (rows + 7) / 8;   // eight rows (warps) per 256-thread block
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    rebias::rebias_rows_kernel<<<grid, 256, 0, st>>>(scales, rows, (int)nb, out, factor, nofit);
  } else {
    const int64_t chunks = rows * nb / 16;
    const int64_t want = (chunks + 255) / 256;
    int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    if (grid < 1) grid = 1;   // the factor is written even for an empty tensor
    rebias::rebias_tensor_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(scales), chunks,
                                                       reinterpret_cast<uint4*>(out), factor, nofit);
  }
  return cudaGetLastError();
}

}  // namespace fp4q
