// fp4q_device.cuh -- device-side format helpers shared by the quantiser,
// dequantiser and GEMM kernels of libfp4q.so (sm_103a).
//
// Formats follow "UE5M3 FP4 Block Scaling for Stable Language Model
// Pretraining", Abstract: E2M1 elements, unsigned E5M3 block scales on blocks
// of 16, an FP32 tensor scale.  Every floating-point step is one IEEE binary32
// operation rounded to nearest even (explicit __f*_rn intrinsics, so that no
// multiply-add is ever contracted), which makes the encoded bytes a pure
// function of the input.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp4q {

enum : int { kUE5M3 = 0, kUE4M3 = 1 };

// Device status bits latched by kernels (read back by fp4q_get_device_status).
enum : int { kStatusNonFinite = 1, kStatusTimeout = 2 };

struct StatsDev {
  unsigned long long scale_sat, scale_uflow, elem_clamped, elem_flushed;
};

// ---------------------------------------------------------------- loads/stores
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream_u32(void* p, uint32_t v) {
  asm volatile("st.global.L1::no_allocate.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// BF16 pair (one 32-bit word) -> two binary32 values, exactly.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- scale format
// UE5M3: bias 15, largest 0xFE = 114688, subnormal step 2^-17.
// UE4M3: bias 7, largest 0x7E = 448, subnormal step 2^-9.
__device__ __forceinline__ float scale_max(int fmt) { return fmt == kUE5M3 ? 114688.0f : 448.0f; }

// Round a non-negative binary32 s* to the scale format: nearest, ties to the
// even code, saturating to the largest finite code (flagged in *sat).
__device__ __forceinline__ uint32_t encode_scale(float s, int fmt, bool* sat) {
  const bool ue5 = (fmt == kUE5M3);
  *sat = s > scale_max(fmt);
  if (!(s > 0.0f)) return 0u;
  if (*sat) return ue5 ? 0xFEu : 0x7Eu;
  if (s < (ue5 ? 0x1p-14f : 0x1p-6f)) {
    // subnormal range: integer multiples of the subnormal step (exact scaling)
    return (uint32_t)__float2int_rn(__fmul_rn(s, ue5 ? 0x1p17f : 0x1p9f));
  }
  // normal range: round the binary32 pattern to 3 mantissa bits (ties to
  // even; a mantissa carry moves into the exponent), then re-bias.
  const uint32_t b = __float_as_uint(s);
  const uint32_t t = (b + 0x7FFFFu + ((b >> 20) & 1u)) >> 20;
  return t - (ue5 ? (112u << 3) : (120u << 3));
}

__device__ __forceinline__ float decode_scale(uint32_t code, int fmt) {
  const bool ue5 = (fmt == kUE5M3);
  const uint32_t e = code >> 3, m = code & 7u;
  if (e == 0) return __fmul_rn(__uint2float_rn(m), ue5 ? 0x1p-17f : 0x1p-9f);
  return __uint_as_float(((e + (ue5 ? 112u : 120u)) << 23) | (m << 20));
}

// ---------------------------------------------------------------- E2M1
// Eight binary32 values -> eight E2M1 nibbles (round to nearest even,
// saturating at +-6, sign kept), element 2j in the low nibble of byte j.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float q[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return out;
}

// Stochastic rounding with a 16-bit uniform U (u = U * 2^-16, round up iff
// u < p, p the position of the magnitude between its grid neighbours).  On
// [1, 8) the E2M1 grid points are the binary32 values with one mantissa bit:
// p * 2^16 = D / 64 for the 22 dropped mantissa bits D, and
//   U < ceil(D / 64)  <=>  D + ((2^16 - 1 - U) << 6 | 63) carries into bit 22,
// so one integer add of that addend and one mask round the pattern (a carry
// into the exponent is the step to the next binade; results of 8 saturate in
// the caller's conversion).  Below 1 the grid is uniform with step 1/2, the
// same as on [1, 2): adding 1 rounded upward maps a onto [1, 2] keeping the
// fraction that decides (ceil at 2^-22, which leaves ceil(p * 2^16)
// unchanged), and subtracting 1 afterwards is exact.
// The addend of the uniform in the low (HI = false) or high half of the word.
template <bool HI>
__device__ __forceinline__ uint32_t sr_addend(uint32_t w) {
  return HI ? ((((~w) >> 10) & 0x3FFFC0u) | 0x3Fu) : ((((~w) << 6) & 0x3FFFC0u) | 0x3Fu);
}
__device__ __forceinline__ float sr_round_mag(float a, uint32_t addend) {
  float c;   // 1.0 below 1, else 0.0
  asm("set.lt.f32.f32 %0, %1, 0f3F800000;" : "=f"(c) : "f"(a));
  const float z = __fadd_ru(a, c);
  const float zr = __uint_as_float((__float_as_uint(z) + addend) & 0xFFC00000u);
  return __fsub_rn(zr, c);
}

// ---------------------------------------------------------------- Philox4x32-10
// Salmon et al., "Parallel random numbers: as easy as 1, 2, 3" (SC 2011):
// ten rounds of two 32x32->64 multiplies and a key-xor permutation, the key
// bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The four random words of counter block ctr (= element index / 4): word j
// belongs to element 4 ctr + j; the row-wise layout rounds with its low 16
// bits, the column-wise layout with its high 16 bits.
__device__ __forceinline__ uint4 sr_words4(uint64_t ctr, uint64_t seed) {
  return philox4x32_10(make_uint4((uint32_t)ctr, (uint32_t)(ctr >> 32), 0u, 0u),
                       (uint32_t)seed, (uint32_t)(seed >> 32));
}

// ---------------------------------------------------------------- one block
// The exact rule for a block with amax a (a BF16 value) under tensor scale T:
//   code = encode(RN(a / RN(6 T))),  r = RN(1 / RN(decode(code) T)).
// Per block the kernels use a multiply by RN(1 / (6 T)) instead of the
// division: the product differs from RN(a / (6 T)) by at most two binary32
// ulps, so it rounds to the same code unless it lies within a few ulps of a
// code's rounding midpoint (or of the largest scale, for the saturation
// flag) -- then, rarely, the exact division is taken.  The binary32 image
// of s * 2^-(127 - bias), shifted right by 20, is the scale code (subnormal
// codes included), so "a few ulps from a midpoint" is a test on its low 20
// bits.  The reciprocal r is tabulated per code once per CTA.
struct BlockScale {
  uint32_t code;
  float r;        // 1 / (s T); 0 for a zero scale: x * 0 is the signed zero of a
                  // finite x, and a block holding inf or NaN never gets code 0
  bool sat;
};

struct ScaleTab {
  float recip[256];    // RN(1 / RN(s_c T)), 0 where s_c = 0
  float six_t;         // RN(6 T)
  float inv6t;         // RN(1 / RN(6 T))
  float unbias;        // 2^-(127 - bias)
  float smax;          // largest finite scale
  uint32_t cmax;       // its code
  int fmt;
};

__device__ __forceinline__ uint32_t exact_code(uint32_t a16, float six_t, int fmt, bool* sat) {
  return encode_scale(__fdiv_rn(__uint_as_float(a16 << 16), six_t), fmt, sat);
}

// Block-wide: every thread of the CTA calls it (it ends with __syncthreads).
__device__ __forceinline__ void build_scale_tab(ScaleTab* tab, float T, int fmt) {
  const uint32_t cmax = (fmt == kUE5M3) ? 0xFEu : 0x7Eu;
  for (uint32_t c = threadIdx.x; c < 256; c += blockDim.x) {
    const float sc = decode_scale(c, fmt);
    tab->recip[c] = (sc == 0.0f || c > cmax) ? 0.0f : __frcp_rn(__fmul_rn(sc, T));
  }
  if (threadIdx.x == 0) {
    tab->six_t = __fmul_rn(6.0f, T);
    tab->inv6t = __frcp_rn(tab->six_t);
    tab->unbias = (fmt == kUE5M3) ? 0x1p-112f : 0x1p-120f;
    tab->smax = scale_max(fmt);
    tab->cmax = cmax;
    tab->fmt = fmt;
  }
  __syncthreads();
}

// Kept out of line: the call is taken by a few blocks in a million, and
// inlining it makes every block pay for the division's instructions.
static __device__ __noinline__ uint32_t exact_code_slow(uint32_t a16, const ScaleTab& tab, bool* sat) {
  return exact_code(a16, tab.six_t, tab.fmt, sat);
}

// With STATS the saturation flag is exact as well; without it, a block
// whose s* lies near the largest scale needs no exact division, because both
// sides of the largest scale round to the same (clamped) code.
// The table's scalars, read once into registers by each kernel (the table
// itself stays in shared memory).
struct ScaleRegs { float inv6t, unbias, smax; uint32_t cmax; };
__device__ __forceinline__ ScaleRegs scale_regs(const ScaleTab& tab) {
  return ScaleRegs{tab.inv6t, tab.unbias, tab.smax, tab.cmax};
}
template <bool STATS>
__device__ __forceinline__ BlockScale block_scale(uint32_t a16, const ScaleTab& tab, const ScaleRegs& k) {
  BlockScale bs;
  const float sa = __fmul_rn(__uint_as_float(a16 << 16), k.inv6t);
  const uint32_t x = __float_as_uint(__fmul_rn(sa, k.unbias));
  const bool near_mid = ((x & 0xFFFFFu) - 0x7FFF8u) < 16u;                     // within 8 of the midpoint
  const bool near_max = STATS && (__float_as_uint(sa) - __float_as_uint(k.smax) + 8u) < 16u;
  if (near_mid || near_max) {
    bs.code = exact_code_slow(a16, tab, &bs.sat);
  } else {
    bs.code = min((x + 0x80000u) >> 20, k.cmax);
    bs.sat = sa > k.smax;
  }
  bs.r = tab.recip[bs.code];
  return bs;
}

// q = x * r for a BF16 pair, as one packed binary32x2 multiply (each lane
// rounded to nearest even, exactly like two scalar multiplies).
__device__ __forceinline__ void mul2(uint32_t pair, float r, float& q0, float& q1) {
  unsigned long long x, rr, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(pair << 16), "r"(pair & 0xFFFF0000u));
  asm("mov.b64 %0, {%1, %1};" : "=l"(rr) : "f"(r));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(x), "l"(rr));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(q0), "=f"(q1) : "l"(y));
}

// (a, b) * r as one packed binary32x2 multiply.
__device__ __forceinline__ void mul2f(float a, float b, float r, float& qa, float& qb) {
  unsigned long long x, rr, y;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(rr) : "f"(r));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(x), "l"(rr));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(qa), "=f"(qb) : "l"(y));
}

// Two binary32 values -> one byte of two E2M1 nibbles (lo in the low nibble),
// in bits 0..7 of the result.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t out;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\t"
      "cvt.u32.u8 %0, b;\n\t}"
      : "=r"(out) : "f"(lo), "f"(hi));
  return out;
}

// Quantises eight elements (four BF16 words) with multiplier r.  Returns the
// eight nibbles; with STATS, adds clamped/flushed element counts.
template <bool SR, bool STATS>
__device__ __forceinline__ uint32_t quantize8(const uint32_t w[4], float r, const uint32_t* rb,
                                              uint32_t* clamped, uint32_t* flushed) {
  float q[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) mul2(w[j], r, q[2 * j], q[2 * j + 1]);
  if (STATS) {
#pragma unroll
    for (int j = 0; j < 8; ++j) *clamped += (fabsf(q[j]) > 6.0f) ? 1u : 0u;
  }
  if (SR) {   // row-wise: the uniforms are the low halves of the words
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float m = sr_round_mag(fabsf(q[j]), sr_addend<false>(rb[j]));
      q[j] = __uint_as_float(__float_as_uint(m) | (__float_as_uint(q[j]) & 0x80000000u));
    }
  }
  const uint32_t nib = cvt_e2m1x8(q);
  if (STATS) {
    // one flag bit per element, bit 3 of its nibble: magnitude 0 (adding 7
    // to a 3-bit magnitude sets bit 3 unless it is 0, with no carry out of
    // the nibble), and a nonzero input (the two BF16 halves of word j are
    // elements 2j and 2j + 1, nibbles 2j and 2j + 1)
    const uint32_t zero_mag = ~((nib & 0x77777777u) + 0x77777777u) & 0x88888888u;
    uint32_t nonzero = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t m = __vsetne2(w[j] & 0x7FFF7FFFu, 0u);     // 1 in each nonzero half
      nonzero |= ((m | (m >> 12)) & 0x11u) << (8 * j + 3);
    }
    *flushed += __popc(zero_mag & nonzero);
  }
  return nib;
}

// max of |bf16| over four words, as a 16-bit pattern (finite values order
// like their patterns; inf/NaN patterns compare above every finite one).
__device__ __forceinline__ uint32_t absmax16(const uint32_t w[4]) {
  uint32_t m = __vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu);
  m = __vmaxu2(m, __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

}  // namespace fp4q
