/*
 * fp4q_oracle.c -- plain, slow, scalar CPU oracle for UE5M3-scaled FP4
 * quantisation and the block-scaled GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * reference leg use it.  It shares no code, header, table or helper with the
 * CUDA library; it is written from the method's statement and the format
 * definitions, one step at a time, so that it can be checked by eye.
 *
 * Source of the method: "UE5M3 FP4 Block Scaling for Stable Language Model
 * Pretraining", Abstract -- E2M1 payloads, unsigned E5M3 (UE5M3) block scales
 * on blocks of 16 elements, a periodically refreshed per-tensor scale, and
 * stochastic rounding selectively on backward gradients.  The abstract fixes
 * only these ingredients; every numeric convention below that it leaves open
 * is a stated reading (bias, specials, rounding of the scale, the tensor-scale
 * formula, the stochastic-rounding bit usage, the nibble order).
 *
 * Arithmetic: IEEE binary32 with round-to-nearest-even, one rounding per
 * operation, no FMA contraction (build with -ffp-contract=off); the GEMM
 * accumulates in binary64.  BF16 inputs are widened to binary32 exactly.
 *
 * Parity status: every function here is pinned by tests/test_oracle_*.py
 * against something other than itself (exact rational models of the formats,
 * brute force, an independent Philox implementation, statistics, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Formats                                                                   */
/* ------------------------------------------------------------------------ */

enum { ORC_UE5M3 = 0, ORC_UE4M3 = 1 };

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* BF16 -> binary32 is exact: the BF16 pattern is the top half of the binary32. */
static float bf16_to_f32(uint16_t h) { return f32_from_bits(((uint32_t)h) << 16); }

/* binary32 -> BF16, round to nearest, ties to even (used by dequantise only). */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = bits_from_f32(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))  /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* E2M1 element (OCP FP4 E2M1 definition): bit 3 sign, bits 2..1 exponent with
 * bias 1, bit 0 mantissa.  Exponent 0 is subnormal (m * 0.5).  No inf, no NaN.
 * Magnitudes of codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_decode(uint8_t nib) {
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* Scale formats.  UE5M3: 8 bits, 5-bit exponent with bias 15, 3-bit mantissa,
 * exponent 0 subnormal (m/8 * 2^-14), code 0xFF reserved as NaN and never
 * produced; largest finite 0xFE = 1.75 * 2^16 = 114688.  UE4M3: the unsigned
 * E4M3 (bias 7, 0x7F NaN, largest finite 0x7E = 448, bit 7 unused). */
static int scale_bias(int fmt) { return fmt == ORC_UE5M3 ? 15 : 7; }
static int scale_nan_code(int fmt) { return fmt == ORC_UE5M3 ? 0xFF : 0x7F; }
static int scale_max_code(int fmt) { return fmt == ORC_UE5M3 ? 0xFE : 0x7E; }

double orc_scale_decode(uint8_t code, int fmt) {
    if (fmt == ORC_UE4M3 && code > 0x7F) return NAN;
    if (code == scale_nan_code(fmt)) return NAN;
    int e = code >> 3, m = code & 7, bias = scale_bias(fmt);
    if (e == 0) return ldexp((double)m / 8.0, 1 - bias);
    return ldexp(1.0 + (double)m / 8.0, e - bias);
}

double orc_scale_max(int fmt) { return orc_scale_decode((uint8_t)scale_max_code(fmt), fmt); }

/* Encode a non-negative binary32 scale s* to the scale format: round to the
 * nearest representable value, ties to the even code, saturating to the
 * largest finite value (no NaN is ever produced).  *sat is set when s* lies
 * above the largest finite value. */
uint8_t orc_scale_encode(float s, int fmt, int *sat) {
    int bias = scale_bias(fmt);
    int max_code = scale_max_code(fmt);
    double smax = orc_scale_decode((uint8_t)max_code, fmt);
    double x = (double)s;
    if (sat) *sat = 0;
    if (!(x > 0.0)) return 0;                    /* zero (and negative zero) */
    if (x > smax) { if (sat) *sat = 1; return (uint8_t)max_code; }
    double min_normal = ldexp(1.0, 1 - bias);
    if (x < min_normal) {
        /* subnormal range: multiples of 2^(1-bias)/8; q == 8 is the min normal */
        double q = rint(x / ldexp(1.0, 1 - bias - 3));   /* rint: ties to even */
        return (uint8_t)q;
    }
    int e2;
    double f = frexp(x, &e2);                    /* x = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;                              /* x = (2f) * 2^E, 2f in [1, 2) */
    double q = rint((2.0 * f - 1.0) * 8.0);      /* 3 mantissa bits, ties even */
    if (q == 8.0) { q = 0.0; E += 1; }
    int code = ((E + bias) << 3) | (int)q;
    if (code > max_code) code = max_code;        /* unreachable once x <= smax */
    return (uint8_t)code;
}

/* E2M1 round to nearest, ties to the even code, saturating at 6.  Returns the
 * nibble with the sign of q (so a negative value that rounds to zero keeps
 * its sign: 0x8). */
uint8_t orc_e2m1_rne(float q) {
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t sign = signbit(q) ? 8 : 0;
    double a = fabs((double)q);
    if (a >= 6.0) return sign | 7;
    int lo = 0;
    while (lo < 7 && grid[lo + 1] <= a) lo++;     /* grid[lo] <= a < grid[lo+1] */
    double dlo = a - grid[lo], dhi = grid[lo + 1] - a;
    int code;
    if (dlo < dhi) code = lo;
    else if (dhi < dlo) code = lo + 1;
    else code = (lo % 2 == 0) ? lo : lo + 1;     /* tie: the even code */
    return sign | (uint8_t)code;
}

/* E2M1 stochastic rounding.  With lo <= |q| < hi adjacent grid points and
 * p = (|q| - lo) / (hi - lo) (exact: the step is a power of two), the result
 * is hi when u < p and lo otherwise, u = U * 2^-16 for the 16-bit uniform
 * integer U (the low 16 bits of the argument).  Magnitudes at or above 6
 * saturate to 6.  Reading: the abstract fixes no random-bit width; 16 bits
 * keep E[result] within 2^-16 of a grid step of q. */
uint8_t orc_e2m1_sr(float q, uint32_t u16) {
    static const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    uint8_t sign = signbit(q) ? 8 : 0;
    float a = fabsf(q);
    if (a >= 6.0f) return sign | 7;
    int lo = 0;
    while (lo < 7 && grid[lo + 1] <= a) lo++;
    float p = (a - grid[lo]) / (grid[lo + 1] - grid[lo]);
    float u = (float)(u16 & 0xFFFFu) * 0x1p-16f;
    return sign | (uint8_t)(u < p ? lo + 1 : lo);
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 and Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel     */
/* random numbers: as easy as 1, 2, 3", SC 2011, section on the Philox        */
/* family): a 10-round counter-based generator.  Each round multiplies        */
/* counter words 0 and 2 by fixed constants, and the new counter is           */
/* (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)); between  */
/* rounds the key is bumped by the Weyl constants.  The 64-bit variant exists */
/* here only so that the round structure can be checked against numpy's       */
/* independent Philox4x64 implementation.                                     */
/* ------------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static void mul64_hilo(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo) {
    uint64_t a0 = (uint32_t)a, a1 = a >> 32, b0 = (uint32_t)b, b1 = b >> 32;
    uint64_t p00 = a0 * b0, p01 = a0 * b1, p10 = a1 * b0, p11 = a1 * b1;
    uint64_t mid = (p00 >> 32) + (uint32_t)p01 + (uint32_t)p10;
    *lo = (mid << 32) | (uint32_t)p00;
    *hi = p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
}

void orc_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2], uint64_t out[4]) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint64_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t hi0, lo0, hi1, lo1;
        mul64_hilo(M0, c0, &hi0, &lo0);
        mul64_hilo(M1, c2, &hi1, &lo1);
        uint64_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 16-bit uniform an element draws.  Reading (the abstract does not say
 * how random bits are assigned): key = (seed low 32, seed high 32); element
 * (r, c) of the rows x cols input has logical index i = r*cols + c and draws
 * word i % 4 of the block with counter (i/4 low 32, i/4 high 32, 0, 0); the
 * row-wise quantisation (axis 0) uses the word's low 16 bits, the
 * column-wise one (axis 1) its high 16 bits, so that the two layouts of the
 * same element round with independent bits from one draw.  The draw depends
 * only on the element and the axis, never on how the work is split or laid
 * out. */
uint32_t orc_sr_uniform(uint64_t seed, uint64_t i, uint32_t axis) {
    uint32_t ctr[4] = {(uint32_t)(i >> 2), (uint32_t)(i >> 34), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t w = out[i & 3];
    return axis == 0 ? (w & 0xFFFFu) : (w >> 16);
}

/* ------------------------------------------------------------------------ */
/* Tensor scale                                                              */
/* ------------------------------------------------------------------------ */

/* amax = max |x| over a BF16 tensor (exact).  *nonfinite is set when any
 * element is inf or NaN (out of contract). */
float orc_amax_bf16(const uint16_t *x, int64_t n, int *nonfinite) {
    float m = 0.0f;
    int bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(bf16_to_f32(x[i]));
        if (!isfinite(a)) { bad = 1; continue; }
        if (a > m) m = a;
    }
    if (nonfinite) *nonfinite = bad;
    return m;
}

/* Per-tensor FP32 scale.  Reading: T = amax / (6 * Smax / H), rounded once,
 * so that the tensor's largest block lands on the top of the block-scale
 * range (H = headroom, a power of two; H = 1 gives T = amax / (6 * Smax)).
 * A zero amax gives T = 1; a T below 2^-100 is raised to 2^-100 so that every
 * later product s * T stays a normal number. */
float orc_tensor_scale(float amax, int fmt, float headroom) {
    float d = (float)(6.0 * orc_scale_max(fmt)) / headroom;   /* exact */
    if (amax == 0.0f) return 1.0f;
    float t = amax / d;
    if (t < 0x1p-100f) t = 0x1p-100f;
    return t;
}

/* ------------------------------------------------------------------------ */
/* Block quantisation                                                        */
/* ------------------------------------------------------------------------ */

enum { ORC_ROW = 0, ORC_COL = 1 };
enum { ORC_RNE = 0, ORC_SR = 1 };
enum { ST_SCALE_SAT = 0, ST_SCALE_UFLOW = 1, ST_ELEM_CLAMP = 2, ST_ELEM_FLUSH = 3 };

/* Quantise one block of 16 binary32 values v[0..15] (already widened from
 * BF16) with tensor scale T.  Writes 16 nibbles and returns the scale code.
 * rbits[j] is the 16-bit uniform of element j (used only for SR). */
static uint8_t quantize_block16(const float v[16], float T, int fmt, int rnd,
                                const uint32_t rbits[16], uint8_t nib[16],
                                uint64_t stats[4]) {
    /* block amax (exact) */
    float amax_b = 0.0f;
    for (int j = 0; j < 16; ++j) { float a = fabsf(v[j]); if (a > amax_b) amax_b = a; }
    /* decode scale s* = amax_b / (6 T), each product/quotient rounded once */
    float six_t = 6.0f * T;
    float s_star = amax_b / six_t;
    int sat = 0;
    uint8_t code = orc_scale_encode(s_star, fmt, &sat);
    if (sat) stats[ST_SCALE_SAT]++;
    if (amax_b > 0.0f && code == 0) stats[ST_SCALE_UFLOW]++;
    float s = (float)orc_scale_decode(code, fmt);
    if (s == 0.0f) {
        for (int j = 0; j < 16; ++j) {
            nib[j] = signbit(v[j]) ? 8 : 0;
            if (v[j] != 0.0f) stats[ST_ELEM_FLUSH]++;
        }
        return code;
    }
    /* element: q = x * (1 / (s * T)) */
    float den = s * T;
    float r = 1.0f / den;
    for (int j = 0; j < 16; ++j) {
        float q = v[j] * r;
        if (fabsf(q) > 6.0f) stats[ST_ELEM_CLAMP]++;
        uint8_t n = (rnd == ORC_SR) ? orc_e2m1_sr(q, rbits[j]) : orc_e2m1_rne(q);
        if (v[j] != 0.0f && (n & 7) == 0) stats[ST_ELEM_FLUSH]++;
        nib[j] = n;
    }
    return code;
}

/* Quantise a rows x cols row-major BF16 tensor.
 *  axis ROW: blocks of 16 consecutive columns of a row.  payload[r, j] holds
 *            elements (r, 2j) in the low and (r, 2j+1) in the high nibble
 *            ([rows, cols/2] bytes); scales[r, b] covers columns 16b..16b+15
 *            ([rows, cols/16] bytes).
 *  axis COL: blocks of 16 consecutive rows of a column -- the row-wise
 *            quantisation of the transpose: payload[c, i] holds (2i, c) low
 *            and (2i+1, c) high ([cols, rows/2]); scales[c, b] covers rows
 *            16b..16b+15 ([cols, rows/16]).
 * stats[4] accumulates {scale saturations, scale underflows, clamped
 * elements, flushed elements}.  rows and cols are multiples of 16. */
void orc_quantize_band(const uint16_t *x, int64_t row_base, int64_t rows, int64_t cols, int axis,
                       int fmt, float T, int rnd, uint64_t seed,
                       uint8_t *payload, uint8_t *scales, uint64_t stats[4]);

void orc_quantize(const uint16_t *x, int64_t rows, int64_t cols, int axis, int fmt,
                  float T, int rnd, uint64_t seed,
                  uint8_t *payload, uint8_t *scales, uint64_t stats[4]) {
    orc_quantize_band(x, 0, rows, cols, axis, fmt, T, rnd, seed, payload, scales, stats);
}

/* The same for rows row_base .. row_base + rows - 1 of a larger tensor with
 * `cols` columns, x pointing at the first of them (row_base a multiple of
 * 16, so that the band holds whole column blocks).  Only the logical index
 * of an element, and with it the stochastic-rounding counter, depends on
 * row_base; the outputs are the band's rows (ROW) or the band's span of each
 * column (COL). */
void orc_quantize_band(const uint16_t *x, int64_t row_base, int64_t rows, int64_t cols, int axis,
                       int fmt, float T, int rnd, uint64_t seed,
                       uint8_t *payload, uint8_t *scales, uint64_t stats[4]) {
    int64_t outer = (axis == ORC_ROW) ? rows : cols;   /* rows of the output */
    int64_t inner = (axis == ORC_ROW) ? cols : rows;   /* the blocked length */
    for (int64_t o = 0; o < outer; ++o) {
        for (int64_t b = 0; b < inner / 16; ++b) {
            float v[16];
            uint32_t rb[16];
            uint8_t nib[16];
            for (int j = 0; j < 16; ++j) {
                int64_t r = (axis == ORC_ROW) ? o : 16 * b + j;
                int64_t c = (axis == ORC_ROW) ? 16 * b + j : o;
                int64_t i = (row_base + r) * cols + c;        /* logical index */
                v[j] = bf16_to_f32(x[r * cols + c]);
                rb[j] = (rnd == ORC_SR) ? orc_sr_uniform(seed, (uint64_t)i, (uint32_t)axis) : 0u;
            }
            uint8_t code = quantize_block16(v, T, fmt, rnd, rb, nib, stats);
            scales[o * (inner / 16) + b] = code;
            for (int j = 0; j < 8; ++j)
                payload[o * (inner / 2) + 8 * b + j] =
                    (uint8_t)(nib[2 * j] | (nib[2 * j + 1] << 4));
        }
    }
}

/* Two-dimensional (16 x 16) block scaling -- the transposition-invariant
 * variant named among the related work of "UE5M3 FP4 Block Scaling for Stable
 * Language Model Pretraining" (Related papers: "Stable FP4 Training via
 * Transposition-Invariant Block Quantization").  Reading: one UE5M3 scale per
 * 16 x 16 tile, chosen by the block rule above with the tile's amax, and one
 * quantisation per element with that scale (SR with the row-wise uniform,
 * the low 16 bits of the element's word); the result is written in both
 * layouts, so that the
 * column-wise operand is exactly the transpose of the row-wise one.
 *   pay_row/sc_row: as axis ROW, sc_row[r, b] = code of tile (r/16, b);
 *   pay_col/sc_col: as axis COL, sc_col[c, b] = code of tile (b, c/16).
 * stats[4]: scale counts per tile, element counts once per element. */
void orc_quantize_2d(const uint16_t *x, int64_t rows, int64_t cols, int fmt, float T, int rnd,
                     uint64_t seed, uint8_t *pay_row, uint8_t *sc_row, uint8_t *pay_col,
                     uint8_t *sc_col, uint64_t stats[4]) {
    for (int64_t tr = 0; tr < rows / 16; ++tr) {
        for (int64_t tc = 0; tc < cols / 16; ++tc) {
            /* tile amax (exact) and its scale, as for a block of 16 */
            float amax_t = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    float a = fabsf(bf16_to_f32(x[(16 * tr + i) * cols + 16 * tc + j]));
                    if (a > amax_t) amax_t = a;
                }
            float six_t = 6.0f * T;
            float s_star = amax_t / six_t;
            int sat = 0;
            uint8_t code = orc_scale_encode(s_star, fmt, &sat);
            if (sat) stats[ST_SCALE_SAT]++;
            if (amax_t > 0.0f && code == 0) stats[ST_SCALE_UFLOW]++;
            float s = (float)orc_scale_decode(code, fmt);
            float r = (s == 0.0f) ? 0.0f : 1.0f / (s * T);
            for (int i = 0; i < 16; ++i) {
                int64_t row = 16 * tr + i;
                for (int j = 0; j < 16; ++j) {
                    int64_t col = 16 * tc + j;
                    int64_t idx = row * cols + col;            /* logical index */
                    float v = bf16_to_f32(x[idx]);
                    uint8_t n;
                    if (s == 0.0f) {
                        n = signbit(v) ? 8 : 0;
                        if (v != 0.0f) stats[ST_ELEM_FLUSH]++;
                    } else {
                        float q = v * r;
                        if (fabsf(q) > 6.0f) stats[ST_ELEM_CLAMP]++;
                        n = (rnd == ORC_SR) ? orc_e2m1_sr(q, orc_sr_uniform(seed, (uint64_t)idx, 0u))
                                            : orc_e2m1_rne(q);
                        if (v != 0.0f && (n & 7) == 0) stats[ST_ELEM_FLUSH]++;
                    }
                    /* row layout: byte (row, col/2); column layout: byte (col, row/2) */
                    uint8_t *br = &pay_row[row * (cols / 2) + col / 2];
                    *br = (col & 1) ? (uint8_t)((*br & 0x0f) | (n << 4)) : (uint8_t)((*br & 0xf0) | n);
                    uint8_t *bc = &pay_col[col * (rows / 2) + row / 2];
                    *bc = (row & 1) ? (uint8_t)((*bc & 0x0f) | (n << 4)) : (uint8_t)((*bc & 0xf0) | n);
                }
                sc_row[row * (cols / 16) + tc] = code;
            }
            for (int j = 0; j < 16; ++j) sc_col[(16 * tc + j) * (rows / 16) + tr] = code;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Dequantisation and the GEMM                                               */
/* ------------------------------------------------------------------------ */

/* Element (o, k) of a quantised [outer, inner] operand as e * s, exact in
 * binary64 (and in binary32: at most 6 significant bits). */
static double deq_es(const uint8_t *payload, const uint8_t *scales, int64_t inner,
                     int64_t o, int64_t k, int fmt) {
    uint8_t byte = payload[o * (inner / 2) + k / 2];
    uint8_t nib = (k & 1) ? (byte >> 4) : (byte & 15);
    return orc_e2m1_decode(nib) * orc_scale_decode(scales[o * (inner / 16) + k / 16], fmt);
}

/* v = RN32(RN32(e * s) * T), written as binary32 and as its BF16 rounding. */
void orc_dequantize(const uint8_t *payload, const uint8_t *scales, int64_t outer,
                    int64_t inner, int fmt, float T, float *out_f32, uint16_t *out_bf16) {
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t k = 0; k < inner; ++k) {
            float es = (float)deq_es(payload, scales, inner, o, k, fmt);
            float v = es * T;
            if (out_f32) out_f32[o * inner + k] = v;
            if (out_bf16) out_bf16[o * inner + k] = f32_to_bf16_rne(v);
        }
}

/* R[m, n] = (T_A * T_B) * sum_k deq(A)[m, k] * deq(B)[n, k], all in binary64
 * (T_A * T_B is exact in binary64).  A is [M, K] and B is [N, K], both
 * quantised along K (the "TN" form C = A . B^T).  Only the (m, n) pairs in
 * ms/ns are computed (count of them); pass ms == NULL for the full M x N
 * matrix in row-major order. */
void orc_gemm(const uint8_t *A, const uint8_t *As, float TA,
              const uint8_t *B, const uint8_t *Bs, float TB,
              int64_t M, int64_t N, int64_t K, int fmt,
              const int64_t *ms, const int64_t *ns, int64_t count, double *out) {
    double alpha = (double)TA * (double)TB;
    int64_t total = ms ? count : M * N;
    for (int64_t t = 0; t < total; ++t) {
        int64_t m = ms ? ms[t] : t / N;
        int64_t n = ms ? ns[t] : t % N;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += deq_es(A, As, K, m, k, fmt) * deq_es(B, Bs, K, n, k, fmt);
        out[t] = alpha * acc;
    }
}

/* Dequantised operand e * s in binary64, [outer, inner] row-major, so that a
 * library matmul can serve as the (exact-product, binary64-sum) contraction. */
void orc_deq_es_matrix(const uint8_t *payload, const uint8_t *scales, int64_t outer,
                       int64_t inner, int fmt, double *out) {
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t k = 0; k < inner; ++k)
            out[o * inner + k] = deq_es(payload, scales, inner, o, k, fmt);
}

/* ------------------------------------------------------------------------ */
/* Re-expressing UE5M3 block scales as UE4M3 scales times a power of two      */
/* ------------------------------------------------------------------------ */

/* The two scale formats share their 3 mantissa bits, so a group of UE5M3
 * scales whose non-zero values v all lie in 14 consecutive binades,
 * e = floor(log2 v) in [e_top - 13, e_top], is exactly f * v4 with one factor
 * f = 2^(e_top - 7) and UE4M3 values v4 = v / f in [2^-6, 240]: the
 * dequantised operand e * s is unchanged, so the same GEMM can run on the
 * tensor cores' UE4M3 block scales with f applied to its result.  (This is the
 * route to native execution that the method's closing argument motivates;
 * the abstract gives no procedure for it.)
 *   per_row != 0: each row is a group, e_top = the largest binade of the
 *     row's non-zero scales (a row of zeros: f = 1);
 *   per_row == 0: the whole tensor is one group with the fixed e_top = 16,
 *     the binade of the largest finite UE5M3 scale -- where the tensor scale
 *     puts the tensor's own amax -- so f = 2^9 and the group fits when every
 *     non-zero scale lies in binades 3..16.
 * out_factor[g] = f (one per row, or one); out_codes = the UE4M3 encoding of
 * v / f (exact: at most 4 significant bits, UE4M3's normal range), 0 for
 * v = 0; *nofit is set to 1 when a group does not fit (its codes and factor
 * are then unspecified).  *nofit is never cleared. */
void orc_rebias_scales(const uint8_t *codes, int64_t rows, int64_t nb, int per_row,
                       uint8_t *out_codes, float *out_factor, int *nofit) {
    const int64_t groups = per_row ? rows : 1;
    const int64_t glen = per_row ? nb : rows * nb;
    for (int64_t g = 0; g < groups; ++g) {
        const uint8_t *c = codes + g * glen;
        uint8_t *o = out_codes + g * glen;
        int emax = -1000, emin = 1000;
        for (int64_t i = 0; i < glen; ++i) {
            const double v = orc_scale_decode(c[i], ORC_UE5M3);
            if (v == 0.0) continue;
            const int e = ilogb(v);
            if (e > emax) emax = e;
            if (e < emin) emin = e;
        }
        if (emax == -1000) {   /* every scale of the group is zero */
            out_factor[g] = per_row ? 1.0f : 512.0f;
            for (int64_t i = 0; i < glen; ++i) o[i] = 0;
            continue;
        }
        const int etop = per_row ? emax : 16;
        if (emin < etop - 13 || emax > etop) *nofit = 1;
        const double f = ldexp(1.0, etop - 7);
        out_factor[g] = (float)f;
        for (int64_t i = 0; i < glen; ++i) {
            const double v = orc_scale_decode(c[i], ORC_UE5M3);
            int sat = 0;
            o[i] = v == 0.0 ? 0 : orc_scale_encode((float)(v / f), ORC_UE4M3, &sat);
        }
    }
}

/* Two windows per row: the row's top 14 binades [e_top - 13, e_top] as in
 * orc_rebias_scales (factor 2^(e_top - 7)), and the 14 below them
 * [e_top - 27, e_top - 14] (factor 2^(e_top - 21), its top binade again in
 * UE4M3's exponent field 14).  Every non-zero UE5M3 value equals
 * hi[i] * f_hi + lo[i] * f_lo with exactly one of the two UE4M3 codes
 * non-zero, so a GEMM on the row splits into two block-scaled contractions
 * of the same payload, one with the hi codes and one with the lo codes,
 * scaled by their factors.  A value below both windows sets *nofit (its
 * codes are then unspecified); a zero row gets factors 1 and 2^-14 and zero
 * codes. */
void orc_rebias_scales2(const uint8_t *codes, int64_t rows, int64_t nb, uint8_t *out_hi, uint8_t *out_lo,
                        float *f_hi, float *f_lo, int *nofit) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t *c = codes + r * nb;
        uint8_t *h = out_hi + r * nb, *l = out_lo + r * nb;
        int emax = -1000;
        for (int64_t i = 0; i < nb; ++i) {
            const double v = orc_scale_decode(c[i], ORC_UE5M3);
            if (v != 0.0 && ilogb(v) > emax) emax = ilogb(v);
        }
        if (emax == -1000) {
            f_hi[r] = 1.0f;
            f_lo[r] = (float)ldexp(1.0, -14);
            for (int64_t i = 0; i < nb; ++i) h[i] = l[i] = 0;
            continue;
        }
        const double fh = ldexp(1.0, emax - 7), fl = ldexp(1.0, emax - 21);
        f_hi[r] = (float)fh;
        f_lo[r] = (float)fl;
        for (int64_t i = 0; i < nb; ++i) {
            const double v = orc_scale_decode(c[i], ORC_UE5M3);
            int sat = 0;
            h[i] = l[i] = 0;
            if (v == 0.0) continue;
            const int e = ilogb(v);
            if (e >= emax - 13) {
                h[i] = orc_scale_encode((float)(v / fh), ORC_UE4M3, &sat);
            } else if (e >= emax - 27) {
                l[i] = orc_scale_encode((float)(v / fl), ORC_UE4M3, &sat);
            } else {
                *nofit = 1;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Array forms of the scalar steps, so that the tests can sweep many values  */
/* through exactly the functions above.                                      */
/* ------------------------------------------------------------------------ */

void orc_e2m1_rne_array(const float *q, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_rne(q[i]);
}

void orc_e2m1_sr_array(const float *q, const uint32_t *u16, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_sr(q[i], u16[i]);
}

void orc_scale_encode_array(const float *s, int64_t n, int fmt, uint8_t *out, uint8_t *sat) {
    for (int64_t i = 0; i < n; ++i) {
        int st = 0;
        out[i] = orc_scale_encode(s[i], fmt, &st);
        if (sat) sat[i] = (uint8_t)st;
    }
}

void orc_sr_uniform_array(uint64_t seed, const uint64_t *idx, int64_t n, uint32_t axis, uint32_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_sr_uniform(seed, idx[i], axis);
}
