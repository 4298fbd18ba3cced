// quantize.cu -- memory-bound kernels of libfp4q.so: tensor amax, tensor
// scale, block-16 E2M1/UE5M3 quantisation (row-wise, column-wise, both from
// one read; RNE or Philox stochastic rounding) and dequantisation.
//
// Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
// Abstract -- E2M1 payloads with UE5M3 block-16 scales under a periodically
// refreshed FP32 tensor scale; stochastic rounding on backward gradients.
//
// Design (GB300): every kernel streams BF16 with 128-bit coalesced loads that
// bypass L1 and keeps blocks in registers.  The row-wise quantiser treats the
// tensor as flat (a block never straddles a row), so that one warp covers 256
// consecutive elements and a lane pair shares one block (one shuffle for the
// block amax).  The column-wise / dual-axis quantisers give each thread a
// piece of a 128 x 128 tile (8 x 8 for round to nearest, 16 x 4 for
// stochastic rounding); lanes that share a block combine their maxima with
// shuffles, so that neither axis needs shared memory.
#include "fp4q_device.cuh"
#include "fp4q_launch.h"

namespace fp4q {

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ void flush_stats(StatsDev* g, uint32_t sat, uint32_t uflow,
                                            uint32_t clamped, uint32_t flushed) {
  __shared__ unsigned long long s[4];
  if (threadIdx.x < 4) s[threadIdx.x] = 0ull;
  __syncthreads();
  sat = __reduce_add_sync(0xFFFFFFFFu, sat);
  uflow = __reduce_add_sync(0xFFFFFFFFu, uflow);
  clamped = __reduce_add_sync(0xFFFFFFFFu, clamped);
  flushed = __reduce_add_sync(0xFFFFFFFFu, flushed);
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&s[0], (unsigned long long)sat);
    atomicAdd(&s[1], (unsigned long long)uflow);
    atomicAdd(&s[2], (unsigned long long)clamped);
    atomicAdd(&s[3], (unsigned long long)flushed);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (s[0]) atomicAdd(&g->scale_sat, s[0]);
    if (s[1]) atomicAdd(&g->scale_uflow, s[1]);
    if (s[2]) atomicAdd(&g->elem_clamped, s[2]);
    if (s[3]) atomicAdd(&g->elem_flushed, s[3]);
  }
}

// Publishes a CTA's max |x| (16-bit pattern): device float amax via an
// unsigned max on the binary32 pattern (valid for non-negative values), and
// the non-finite flag.
__device__ __forceinline__ void flush_amax(float* amax_out, int* status, uint32_t m16) {
  __shared__ uint32_t s_m;
  if (threadIdx.x == 0) s_m = 0u;
  __syncthreads();
  m16 = __reduce_max_sync(0xFFFFFFFFu, m16);
  if ((threadIdx.x & 31) == 0) atomicMax(&s_m, m16);
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t m = s_m;
    if (m >= 0x7F80u) atomicOr(status, kStatusNonFinite);
    if (amax_out && m) atomicMax(reinterpret_cast<unsigned int*>(amax_out), m << 16);
  }
}

// ---------------------------------------------------------------- amax
// Streams the tensor with 128-bit loads, eight in flight per thread.
__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ in, int64_t nchunks,
                                                   const uint16_t* __restrict__ tail, int ntail,
                                                   float* amax_out, int* status) {
  uint32_t m = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; g + 7 * stride < nchunks; g += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = ld_stream_v4(in + g + u * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      m = max(m, absmax16(w));
    }
  }
  for (; g < nchunks; g += stride) {
    const uint4 v = ld_stream_v4(in + g);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    m = max(m, absmax16(w));
  }
  if (blockIdx.x == 0 && (int)threadIdx.x < ntail) m = max(m, (uint32_t)(tail[threadIdx.x] & 0x7FFFu));
  flush_amax(amax_out, status, m);
}

__global__ void tensor_scale_kernel(const float* amax, float denom, float* out) {
  const float a = *amax;
  float t = (a == 0.0f) ? 1.0f : __fdiv_rn(a, denom);
  if (t < 0x1p-100f) t = 0x1p-100f;
  *out = t;
}

// ---------------------------------------------------------------- row-wise
// One chunk = 8 consecutive elements (16 bytes of BF16) per lane; lanes 2k
// and 2k+1 hold one block of 16.  The warp loop is uniform so that every
// lane takes part in the shuffle; inactive lanes carry zeros.
constexpr int kRowThreads = 512;

template <bool SR, bool STATS>
__global__ void __launch_bounds__(kRowThreads, 2) quantize_row_kernel(
    const uint4* __restrict__ in, int64_t nchunks, int fmt, const float* __restrict__ tscale,
    uint64_t seed, uint32_t* __restrict__ payload, uint8_t* __restrict__ scales, StatsDev* stats,
    float* amax_out, int* status) {
  __shared__ ScaleTab tab;
  build_scale_tab(&tab, __ldg(tscale), fmt);
  const ScaleRegs kr = scale_regs(tab);
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  constexpr int U = SR ? 2 : 4;  // chunks in flight per lane
  uint32_t tmax = 0, n_sat = 0, n_uflow = 0, n_clamp = 0, n_flush = 0;

  for (int64_t base = warp * 32 * U; base < nchunks; base += nwarps * 32 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = base + u * 32 + lane;
      v[u] = (g < nchunks) ? ld_stream_v4(in + g) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = base + u * 32 + lane;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t m = absmax16(w);
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      tmax = max(tmax, m);
      const BlockScale bs = block_scale<STATS>(m, tab, kr);
      uint32_t rb[8];
      if (SR) {
        const uint4 a = sr_words4((uint64_t)g * 2, seed);
        const uint4 b = sr_words4((uint64_t)g * 2 + 1, seed);
        rb[0] = a.x; rb[1] = a.y; rb[2] = a.z; rb[3] = a.w;
        rb[4] = b.x; rb[5] = b.y; rb[6] = b.z; rb[7] = b.w;
      }
      uint32_t c = 0, f = 0;
      const uint32_t nib = quantize8<SR, STATS>(w, bs.r, rb, &c, &f);
      if (g < nchunks) {
        st_stream_u32(payload + g, nib);
        if ((lane & 1) == 0) scales[g >> 1] = (uint8_t)bs.code;
        if (STATS) {
          n_clamp += c;
          n_flush += f;
          if ((lane & 1) == 0) {
            n_sat += bs.sat ? 1u : 0u;
            n_uflow += (m != 0u && bs.code == 0u) ? 1u : 0u;
          }
        }
      }
    }
  }
  if (STATS) flush_stats(stats, n_sat, n_uflow, n_clamp, n_flush);
  flush_amax(amax_out, status, tmax);
}

// ---------------------------------------------------------------- tiles
// Column-wise and dual-axis round-to-nearest quantisation, register-resident.
// A tile is 128 rows x 128 columns (each persistent CTA walks tiles with a
// stride of the grid); warp w takes rows 16 w .. +15 of it.  Lane l
// holds an 8 x 8 piece: rows 16 w + 8 (l / 16) .. +7, columns 8 (l % 16) .. +7,
// loaded with eight 128-bit loads (each warp load reads two 256-byte row
// segments).
//   magnitudes: one pass over the masked BF16 words gives, per word column,
//     the maxima of its two columns over the lane's eight rows, and per row
//     pair the two row maxima, each packed two to a word;
//   column blocks: lanes l and l ^ 16 hold the two 8-row halves of the same
//     eight columns; one shuffle per word column completes both columns'
//     block maxima, lane l computes the scale of the even (l < 16) or odd
//     column of each word column and one more shuffle hands the reciprocal
//     to its partner;
//   row blocks (dual axis): lanes l and l ^ 1 hold the two 8-column halves of
//     the same rows; per row pair one shuffle completes both maxima and each
//     lane computes one of the two scales, exchanged the same way;
//   conversion: each 2 x 2 group (two BF16 words of consecutive rows) is
//     unpacked once and multiplied by the row reciprocal (packed binary32x2
//     multiplies) and the column reciprocal (scalar); a row payload word is eight nibbles of
//     one row, a column payload word eight nibbles of one column.
// Row outputs go straight to global memory; the column payload and codes of
// a tile are staged in shared memory (ColStage, double-buffered) and leave
// as 64 contiguous bytes per column.  The block-scale reciprocals come from
// a per-CTA table.
constexpr int kRcRows = 128, kRcCols = 128, kRcThreads = 256;

__device__ __forceinline__ uint32_t word_of(const uint4& v, int q) {
  return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// max(|a|, |b|) of two BF16 pairs lane by lane, on the FP16/BF16 pipe (one
// instruction instead of a sign mask and an integer max on the ALU): the
// magnitudes are exact, a NaN input propagates (so that the non-finite flag
// still sees it), and the sign bits of the result are the XOR of the inputs'
// -- callers mask them off once, after accumulating.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Places bits 0..7 of b into byte k of acc.
__device__ __forceinline__ uint32_t put_byte(uint32_t acc, uint32_t b, int k) {
  return __byte_perm(acc, b, k == 0 ? 0x3214 : k == 1 ? 0x3240 : k == 2 ? 0x3410 : 0x4210);
}

// Flushed-element count of one converted byte: inputs of non-zero magnitude
// whose nibble has zero magnitude.
__device__ __forceinline__ uint32_t flushed2(float x0, float x1, uint32_t byte) {
  return ((__float_as_uint(x0) & 0x7FFFFFFFu) != 0u && (byte & 7u) == 0u ? 1u : 0u) +
         ((__float_as_uint(x1) & 0x7FFFFFFFu) != 0u && (byte & 0x70u) == 0u ? 1u : 0u);
}

__device__ __forceinline__ uint32_t clamped2(float q0, float q1) {
  return (fabsf(q0) > 6.0f ? 1u : 0u) + (fabsf(q1) > 6.0f ? 1u : 0u);
}

// Column-wise outputs of one 128 x 128 tile, staged in shared memory so that
// they leave as contiguous runs per column (the 8 x 8 pieces of a warp belong
// to 32 different columns).  pay: per column 128 bytes of which 64 are used
// (16 words of eight row nibbles); word g of column c sits at
// 32 c + (g ^ 2 ((c >> 3) & 15)), which keeps word pairs (2k, 2k + 1) adjacent
// and makes the writes of a warp conflict-free.  sc: 8 block codes per column.
struct ColStage {
  uint32_t pay[128 * 32];
  uint8_t sc[128 * 8];
};

__device__ __forceinline__ int stage_word(int c, int g) { return 32 * c + (g ^ (2 * ((c >> 3) & 15))); }

// Every thread of the CTA: the staged column outputs of the tile whose first
// row and column are tr, tc -> global, 8-byte pieces (16 rows of a column).
__device__ __forceinline__ void write_col_stage(const ColStage& st, int64_t R, int64_t C, int64_t tr,
                                                int64_t tc, uint8_t* __restrict__ pay_col,
                                                uint8_t* __restrict__ sc_col) {
  // thread t writes piece t & 7 of columns t / 8 + 32 i, i < 4: one base
  // pointer, advanced by 32 column rows of R / 2 bytes
  const int c_t = (int)threadIdx.x >> 3, piece = (int)threadIdx.x & 7;
  uint8_t* dst = pay_col + (tc + c_t) * (R / 2) + tr / 2 + 8 * piece;
  const int64_t step = 32 * (R / 2);
  const bool rows_in = tr + 16 * piece < R;
#pragma unroll
  for (int i = 0; i < 4; ++i, dst += step) {
    const int c = c_t + 32 * i;
    if (rows_in && tc + c < C) {
      const uint2 w = *reinterpret_cast<const uint2*>(&st.pay[stage_word(c, 2 * piece)]);
      *reinterpret_cast<uint2*>(dst) = w;
    }
  }
  if (threadIdx.x < 128) {
    const int c = threadIdx.x;
    if (tc + c < C) {
      uint8_t* dst = sc_col + (tc + c) * (R / 16) + tr / 16;
      const int nb = (int)((R - tr) / 16 < 8 ? (R - tr) / 16 : 8);
      if (nb == 8 && (reinterpret_cast<uintptr_t>(dst) & 7) == 0) {
        *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(&st.sc[8 * c]);
      } else {
        for (int b = 0; b < nb; ++b) dst[b] = st.sc[8 * c + b];
      }
    }
  }
}

// Per-thread counters of the tile quantisers.
struct TileCounts {
  uint32_t tmax = 0;
  uint32_t r_sat = 0, r_uflow = 0, r_clamp = 0, r_flush = 0;
  uint32_t c_sat = 0, c_uflow = 0, c_clamp = 0, c_flush = 0;
};

// One lane's 8 x 8 piece of a 128 x 128 tile: rows r0 .. r0 + 7 (r0 = rb or
// rb + 8, rb the first row of the 16-row column block), columns c0 .. c0 + 7.
// TWO_D: one scale per 16 x 16 tile (lanes l, l ^ 1, l ^ 16, l ^ 17), used by
// both layouts, which then hold the same nibbles transposed.
template <bool STATS, bool DO_ROW, bool TWO_D>
__device__ __forceinline__ void rne_piece(const uint4 (&v)[8], int64_t R, int64_t C, int64_t rb,
                                          int64_t r0, int64_t c0, bool ok, int half, int par,
                                          const ScaleTab& tab, uint32_t* __restrict__ pay_row,
                                          uint8_t* __restrict__ sc_row, ColStage& stage, int warp, int cg,
                                          TileCounts& cnt) {
  const ScaleRegs kr = scale_regs(tab);
  // ---- magnitudes: cmx[q] = maxima of columns 2q (low) and 2q + 1 (high);
  // rpx[p] = maxima of rows 2p (low) and 2p + 1 (high) over the lane's columns
  uint32_t cmx[4] = {0u, 0u, 0u, 0u}, rpx[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint32_t rm[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        w[q] = word_of(v[2 * p + k], q);
        cmx[q] = absmax_bf16x2(cmx[q], w[q]);
      }
      rm[k] = absmax_bf16x2(absmax_bf16x2(w[0], w[1]), absmax_bf16x2(w[2], w[3]));
    }
    rpx[p] = absmax_bf16x2(__byte_perm(rm[0], rm[1], 0x5410), __byte_perm(rm[0], rm[1], 0x7632)) & 0x7FFF7FFFu;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) cmx[q] &= 0x7FFF7FFFu;
  const uint32_t tm = __vmaxu2(__vmaxu2(cmx[0], cmx[1]), __vmaxu2(cmx[2], cmx[3]));
  cnt.tmax = max(cnt.tmax, max(tm & 0xFFFFu, tm >> 16));

  BlockScale ts;   // the 16 x 16 tile's scale (TWO_D)
  if (TWO_D) {
    uint32_t m = max(tm & 0xFFFFu, tm >> 16);
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
    ts = block_scale<STATS>(m, tab, kr);
    if (STATS && ok && par == 0 && half == 0) {
      cnt.r_sat += ts.sat ? 1u : 0u;
      cnt.r_uflow += (m != 0u && ts.code == 0u) ? 1u : 0u;
    }
  }

  // ---- column scales: this lane computes column 2q + half of word column q
  const uint32_t pick = half ? 0x4432u : 0x4410u;   // high or low 16 bits, zero-extended
  float colr[8];
#pragma unroll
  for (int q = 0; q < 4 && TWO_D; ++q) {
    colr[2 * q] = colr[2 * q + 1] = ts.r;
    stage.sc[8 * (8 * cg + 2 * q + half) + warp] = (uint8_t)ts.code;
  }
#pragma unroll
  for (int q = 0; q < 4 && !TWO_D; ++q) {
    const uint32_t full = __vmaxu2(cmx[q], __shfl_xor_sync(0xFFFFFFFFu, cmx[q], 16));
    const uint32_t cm = __byte_perm(full, 0u, pick);
    const BlockScale bs = block_scale<STATS>(cm, tab, kr);
    const float other = __shfl_xor_sync(0xFFFFFFFFu, bs.r, 16);
    colr[2 * q] = half ? other : bs.r;
    colr[2 * q + 1] = half ? bs.r : other;
    stage.sc[8 * (8 * cg + 2 * q + half) + warp] = (uint8_t)bs.code;
    if (ok) {
      if (STATS) {
        cnt.c_sat += bs.sat ? 1u : 0u;
        cnt.c_uflow += (cm != 0u && bs.code == 0u) ? 1u : 0u;
      }
    }
  }

  // ---- conversion, one row pair at a time.  Row outputs through base
  // pointers advanced by two rows per pair: payload words of rows r0 + 2p
  // (+ 1) at prow, scale code of row r0 + 2p + par at srow.
  const uint32_t rpick = par ? 0x4432u : 0x4410u;
  uint32_t pcol[8];
  uint32_t* prow = pay_row + ((r0 * C + c0) >> 3);
  uint8_t* srow = sc_row + (((r0 + par) * C + (c0 & ~(int64_t)15)) >> 4);
  const int64_t pstep = C >> 3, sstep = C >> 3;   // one row of payload words; two rows of codes
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float re = 0.0f, ro = 0.0f;   // row reciprocals of rows 2p and 2p + 1
    if (DO_ROW && TWO_D) {
      re = ro = ts.r;
      if (ok) srow[p * sstep] = (uint8_t)ts.code;
    } else if (DO_ROW) {
      const uint32_t full = __vmaxu2(rpx[p], __shfl_xor_sync(0xFFFFFFFFu, rpx[p], 1));
      const uint32_t m = __byte_perm(full, 0u, rpick);          // row 2p + par
      const BlockScale bs = block_scale<STATS>(m, tab, kr);
      const float other = __shfl_xor_sync(0xFFFFFFFFu, bs.r, 1);
      re = par ? other : bs.r;
      ro = par ? bs.r : other;
      if (ok) {
        srow[p * sstep] = (uint8_t)bs.code;
        if (STATS) {
          cnt.r_sat += bs.sat ? 1u : 0u;
          cnt.r_uflow += (m != 0u && bs.code == 0u) ? 1u : 0u;
        }
      }
    }
    float xe[8], xo[8];   // row products of rows 2p and 2p + 1
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t wa = word_of(v[2 * p], q), wb = word_of(v[2 * p + 1], q);
      const float a0 = bf16_lo(wa), a1 = bf16_hi(wa), b0 = bf16_lo(wb), b1 = bf16_hi(wb);
      if (DO_ROW) {
        mul2f(a0, a1, re, xe[2 * q], xe[2 * q + 1]);
        mul2f(b0, b1, ro, xo[2 * q], xo[2 * q + 1]);
      }
      // column products as scalar multiplies: their operand pairs are not
      // the register pairs the row products use
      const float y0 = __fmul_rn(a0, colr[2 * q]), y1 = __fmul_rn(b0, colr[2 * q]);
      const float z0 = __fmul_rn(a1, colr[2 * q + 1]), z1 = __fmul_rn(b1, colr[2 * q + 1]);
      const uint32_t by = e2m1x2(y0, y1), bz = e2m1x2(z0, z1);
      pcol[2 * q] = p == 0 ? by : put_byte(pcol[2 * q], by, p);
      pcol[2 * q + 1] = p == 0 ? bz : put_byte(pcol[2 * q + 1], bz, p);
      if (STATS && !TWO_D && ok) {
        cnt.c_clamp += clamped2(y0, y1) + clamped2(z0, z1);
        cnt.c_flush += flushed2(a0, b0, by) + flushed2(a1, b1, bz);
      }
    }
    if (DO_ROW) {
      const uint32_t ne = cvt_e2m1x8(xe), no = cvt_e2m1x8(xo);
      if (ok) {
        st_stream_u32(prow + (2 * p) * pstep, ne);
        st_stream_u32(prow + (2 * p + 1) * pstep, no);
        if (STATS) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t wa = word_of(v[2 * p], q), wb = word_of(v[2 * p + 1], q);
            cnt.r_clamp += clamped2(xe[2 * q], xe[2 * q + 1]) + clamped2(xo[2 * q], xo[2 * q + 1]);
            cnt.r_flush += flushed2(bf16_lo(wa), bf16_hi(wa), (ne >> (8 * q)) & 0xFFu) +
                       flushed2(bf16_lo(wb), bf16_hi(wb), (no >> (8 * q)) & 0xFFu);
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) stage.pay[stage_word(8 * cg + j, 2 * warp + half)] = pcol[j];
}

// Persistent: each CTA walks tiles with a stride of the grid, the loads of
// its next piece in flight while it converts the current one; the scale table
// is built and the amax and counts are published once per CTA.
template <bool STATS, bool DO_ROW, bool TWO_D>
__global__ void __launch_bounds__(kRcThreads, 2) quantize_tile_kernel(
    const uint16_t* __restrict__ in, int64_t R, int64_t C, int fmt,
    const float* __restrict__ tscale, uint32_t* __restrict__ pay_row,
    uint8_t* __restrict__ sc_row, uint8_t* __restrict__ pay_col, uint8_t* __restrict__ sc_col,
    StatsDev* stats, float* amax_out, int* status) {
  __shared__ ScaleTab tab;
  __shared__ ColStage stage[2];   // double-buffered: one barrier per tile
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int half = lane >> 4, cg = lane & 15, par = cg & 1;
  // tile counts fit in 32 bits (the ABI rejects more than 2^31 - 1 tiles)
  const uint32_t tiles_x = (uint32_t)((C + kRcCols - 1) / kRcCols);
  const uint32_t ntiles = tiles_x * (uint32_t)((R + kRcRows - 1) / kRcRows);
  TileCounts cnt;
  // Tile coordinates walk with the grid stride: one 32-bit division per CTA
  // for the first tile and the stride, then a carry per step (a 64-bit
  // division per tile would cost more than a piece's conversion).
  const uint32_t stride = gridDim.x;
  const uint32_t dy = stride / tiles_x, dx = stride - dy * tiles_x;
  auto advance = [&](uint32_t& ty, uint32_t& tx) {
    tx += dx;
    ty += dy;
    if (tx >= tiles_x) { tx -= tiles_x; ++ty; }
  };
  // piece coordinates of tile (ty, tx); sizes are multiples of 16, so a
  // 16 x 16 region is wholly inside or outside
  auto coords = [&](uint32_t ty, uint32_t tx, int64_t& rb, int64_t& r0, int64_t& c0) {
    rb = (int64_t)ty * kRcRows + warp * 16;
    r0 = rb + 8 * half;
    c0 = (int64_t)tx * kRcCols + cg * 8;
    return rb < R && c0 < C;
  };
  auto load = [&](uint4 (&v)[8], int64_t r0, int64_t c0, bool ok) {
    const uint16_t* src = in + r0 * C + c0;
#pragma unroll
    for (int rr = 0; rr < 8; ++rr)
      v[rr] = ok ? ld_stream_v4(src + rr * C) : make_uint4(0, 0, 0, 0);
  };
  uint4 va[8], vb[8];
  uint32_t tile = blockIdx.x;
  uint32_t ty = tile / tiles_x, tx = tile - ty * tiles_x;   // tile being converted (buffer a)
  int64_t rb, r0, c0;
  bool ok = tile < ntiles && coords(ty, tx, rb, r0, c0);
  load(va, r0, c0, ok);
  build_scale_tab(&tab, __ldg(tscale), fmt);   // while the first piece is in flight
  // two tiles per trip, so that the two register buffers swap roles without copies
  auto flush_tile = [&](const ColStage& st, uint32_t fy, uint32_t fx) {
    __syncthreads();
    write_col_stage(st, R, C, (int64_t)fy * kRcRows, (int64_t)fx * kRcCols, pay_col, sc_col);
  };
  for (; tile < ntiles; tile += 2 * stride) {
    uint32_t ty1 = ty, tx1 = tx;
    advance(ty1, tx1);
    int64_t rb1, r01, c01;
    const bool ok1 = tile + stride < ntiles && coords(ty1, tx1, rb1, r01, c01);
    load(vb, r01, c01, ok1);
    rne_piece<STATS, DO_ROW, TWO_D>(va, R, C, rb, r0, c0, ok, half, par, tab, pay_row, sc_row, stage[0], warp, cg, cnt);
    flush_tile(stage[0], ty, tx);
    if (tile + stride >= ntiles) break;
    ty = ty1;
    tx = tx1;
    advance(ty, tx);
    ok = tile + 2 * stride < ntiles && coords(ty, tx, rb, r0, c0);
    load(va, r0, c0, ok);
    rne_piece<STATS, DO_ROW, TWO_D>(vb, R, C, rb1, r01, c01, ok1, half, par, tab, pay_row, sc_row, stage[1], warp, cg, cnt);
    flush_tile(stage[1], ty1, tx1);
  }
  if (STATS) {
    if (DO_ROW) flush_stats(stats, cnt.r_sat, cnt.r_uflow, cnt.r_clamp, cnt.r_flush);
    if (!TWO_D) flush_stats(stats + (DO_ROW ? 1 : 0), cnt.c_sat, cnt.c_uflow, cnt.c_clamp, cnt.c_flush);
  }
  flush_amax(amax_out, status, cnt.tmax);
}

// ---------------------------------------------------------------- tiles, 16 x 4 pieces
// Column-wise and dual-axis stochastic-rounding quantisation,
// register-resident; the narrower piece leaves the registers that the Philox
// work needs.  A CTA covers 128 rows x 128 columns: warp w takes rows
// 16 w .. +15 and lane l columns 4 l .. +3 (sixteen coalesced 64-bit loads,
// each warp load one 256-byte row segment).
//   magnitudes: one pass over the masked BF16 words gives the four column
//     maxima over the lane's sixteen rows (each column block whole in the
//     lane) and the row maxima over its four columns, packed two rows to a
//     word;
//   row blocks (dual axis): four consecutive lanes hold the 16 columns of a
//     block; two butterfly shuffles per packed word complete the maxima of
//     two rows, lane l computes the scales of the rows r with r % 4 = l % 4,
//     and one shuffle per row pair hands each lane the reciprocals it lacks;
//   conversion: one row pair at a time, each BF16 word of the pair is
//     unpacked once and multiplied by its row and its column reciprocal; the
//     row and the column products are rounded with the words of their own
//     Philox streams.
// Stochastic rounding draws one Philox block per row and axis: the four
// words of counter (row C + 4 l) / 4 are exactly the lane's four elements.
// Row outputs go straight to global memory; the column payload and codes of
// the tile are staged in shared memory (ColStage) and leave as 64
// contiguous bytes per column.  The block-scale reciprocals come from a
// per-CTA table.

// Stochastic rounding of the pair (q0, q1) with the uniforms in the low
// (HI = false, row-wise) or high halves of the random words w0, w1 -> one
// byte of two E2M1 nibbles (q0 low).
template <bool HI>
__device__ __forceinline__ uint32_t sr_e2m1x2(float q0, float q1, uint32_t w0, uint32_t w1) {
  const float m0 = sr_round_mag(fabsf(q0), sr_addend<HI>(w0));
  const float m1 = sr_round_mag(fabsf(q1), sr_addend<HI>(w1));
  return e2m1x2(__uint_as_float(__float_as_uint(m0) | (__float_as_uint(q0) & 0x80000000u)),
                __uint_as_float(__float_as_uint(m1) | (__float_as_uint(q1) & 0x80000000u)));
}

// TWO_D: one scale per 16 x 16 tile (the four lanes of a group), and one
// quantisation per element with the row-wise random stream, written in both
// layouts.
template <bool STATS, bool DO_ROW, bool TWO_D>
__global__ void __launch_bounds__(kRcThreads, 3) quantize_tile4_kernel(
    const uint16_t* __restrict__ in, int64_t R, int64_t C, int fmt,
    const float* __restrict__ tscale, uint64_t seed, uint8_t* __restrict__ pay_row,
    uint8_t* __restrict__ sc_row, uint8_t* __restrict__ pay_col, uint8_t* __restrict__ sc_col,
    StatsDev* stats, float* amax_out, int* status) {
  __shared__ ScaleTab tab;
  __shared__ ColStage stage;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int own = lane & 3;                                         // rows r with r % 4 == own
  // one CTA per tile, tiles numbered row-major (a 1-D grid: no 65535 limit
  // on the number of tile rows)
  const uint32_t tiles_x = (uint32_t)((C + kRcCols - 1) / kRcCols);   // tile counts fit in 32 bits
  const uint32_t ty = blockIdx.x / tiles_x, tx = blockIdx.x - ty * tiles_x;
  const int64_t r0 = (int64_t)ty * kRcRows + warp * 16;
  const int64_t c0 = (int64_t)tx * kRcCols + lane * 4;
  // sizes are multiples of 16, so a 16-column block is either wholly inside
  // or wholly outside, and so is each 16 x 4 piece
  const bool ok = r0 < R && c0 < C;
  uint32_t r_sat = 0, r_uflow = 0, r_clamp = 0, r_flush = 0;
  uint32_t c_sat = 0, c_uflow = 0, c_clamp = 0, c_flush = 0;

  uint2 v[16];
  const uint16_t* src = in + r0 * C + c0;
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    if (ok) {
      asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                   : "=r"(v[rr].x), "=r"(v[rr].y) : "l"(src + rr * C));
    } else {
      v[rr] = make_uint2(0, 0);
    }
  }
  build_scale_tab(&tab, __ldg(tscale), fmt);   // while the piece is in flight
  const ScaleRegs kr = scale_regs(tab);

  // ---- magnitudes: cmx0 = columns 0 (low), 1 (high); cmx1 = columns 2, 3;
  // rpx[i] = rows 2i (low), 2i + 1 (high)
  uint32_t cmx0 = 0u, cmx1 = 0u, rpx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t rm[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t a = v[2 * i + k].x, b = v[2 * i + k].y;
      cmx0 = absmax_bf16x2(cmx0, a);
      cmx1 = absmax_bf16x2(cmx1, b);
      rm[k] = absmax_bf16x2(a, b);
    }
    rpx[i] = absmax_bf16x2(__byte_perm(rm[0], rm[1], 0x5410), __byte_perm(rm[0], rm[1], 0x7632)) & 0x7FFF7FFFu;
  }
  cmx0 &= 0x7FFF7FFFu;
  cmx1 &= 0x7FFF7FFFu;
  uint32_t tmax = __vmaxu2(cmx0, cmx1);
  tmax = max(tmax & 0xFFFFu, tmax >> 16);

  BlockScale ts;   // the 16 x 16 tile's scale (TWO_D)
  if (TWO_D) {
    uint32_t m = max(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    ts = block_scale<STATS>(m, tab, kr);
    if (STATS && ok && own == 0) {
      r_sat += ts.sat ? 1u : 0u;
      r_uflow += (m != 0u && ts.code == 0u) ? 1u : 0u;
    }
  }

  // ---- column scales (whole blocks in the lane)
  float rc[4];
#pragma unroll
  for (int j = 0; j < 4 && TWO_D; ++j) {
    rc[j] = ts.r;
    stage.sc[8 * (4 * lane + j) + warp] = (uint8_t)ts.code;
  }
#pragma unroll
  for (int j = 0; j < 4 && !TWO_D; ++j) {
    const uint32_t w = j < 2 ? cmx0 : cmx1;
    const uint32_t cm = (j & 1) ? (w >> 16) : (w & 0xFFFFu);
    const BlockScale bs = block_scale<STATS>(cm, tab, kr);
    rc[j] = bs.r;
    stage.sc[8 * (4 * lane + j) + warp] = (uint8_t)bs.code;
    if (ok) {
      if (STATS) {
        c_sat += bs.sat ? 1u : 0u;
        c_uflow += (cm != 0u && bs.code == 0u) ? 1u : 0u;
      }
    }
  }

  // ---- row scales: this lane computes rows own, own + 4, own + 8, own + 12
  // (codes through a base pointer advanced by four rows)
  float rown[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  uint8_t* srow = sc_row + (((r0 + own) * C + (c0 & ~(int64_t)15)) >> 4);
  const int64_t sstep = C >> 2;
  if (DO_ROW && TWO_D) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (ok) srow[k * sstep] = (uint8_t)ts.code;
  } else if (DO_ROW) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      rpx[i] = __vmaxu2(rpx[i], __shfl_xor_sync(0xFFFFFFFFu, rpx[i], 1));
      rpx[i] = __vmaxu2(rpx[i], __shfl_xor_sync(0xFFFFFFFFu, rpx[i], 2));
    }
    const uint32_t pick = (own & 1) ? 0x4432u : 0x4410u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // row 4k + own sits in word 2k + own / 2, half own % 2
      const uint32_t w = (own >> 1) ? rpx[2 * k + 1] : rpx[2 * k];
      const uint32_t m = __byte_perm(w, 0u, pick);
      const BlockScale bs = block_scale<STATS>(m, tab, kr);
      rown[k] = bs.r;
      if (ok) {
        srow[k * sstep] = (uint8_t)bs.code;
        if (STATS) {
          r_sat += bs.sat ? 1u : 0u;
          r_uflow += (m != 0u && bs.code == 0u) ? 1u : 0u;
        }
      }
    }
  }

  // ---- conversion, one row pair at a time
  uint2 pcol[4] = {make_uint2(0, 0), make_uint2(0, 0), make_uint2(0, 0), make_uint2(0, 0)};
  const int grp = lane & ~3;
  // Philox counter (element index / 4) of row r0 and the row payload pointer,
  // both advanced row by row
  const int64_t e0 = (r0 * C + c0) >> 2, estep = C >> 2;
  uint8_t* prow = pay_row + ((r0 * C + c0) >> 1);
  const int64_t pstep = C >> 1;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int64_t ea = e0 + (2 * p) * estep, eb = ea + estep;
    float re = 0.0f, ro = 0.0f;
    uint32_t wra[4], wrb[4], wca[4], wcb[4];
    if (DO_ROW) {
      if (TWO_D) {
        re = ro = ts.r;
      } else {
        // rows 2p and 2p + 1 belong to lanes grp + (2p) % 4 and grp + (2p + 1) % 4
        re = __shfl_sync(0xFFFFFFFFu, rown[p >> 1], grp + ((2 * p) & 3));
        ro = __shfl_sync(0xFFFFFFFFu, rown[p >> 1], grp + ((2 * p + 1) & 3));
      }
    }
    // one Philox block per row and four elements serves both layouts: the
    // row-wise rounding takes the low halves of the words, the column-wise
    // the high halves (16 x 16 scaling: one quantisation, the low halves)
    {
      const uint4 ra = sr_words4((uint64_t)ea, seed), rb = sr_words4((uint64_t)eb, seed);
      wra[0] = ra.x; wra[1] = ra.y; wra[2] = ra.z; wra[3] = ra.w;
      wrb[0] = rb.x; wrb[1] = rb.y; wrb[2] = rb.z; wrb[3] = rb.w;
#pragma unroll
      for (int k = 0; k < 4; ++k) { wca[k] = wra[k]; wcb[k] = wrb[k]; }
    }
    uint32_t rowa = 0u, rowb = 0u;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t wa = q ? v[2 * p].y : v[2 * p].x, wb = q ? v[2 * p + 1].y : v[2 * p + 1].x;
      const float a0 = bf16_lo(wa), a1 = bf16_hi(wa), b0 = bf16_lo(wb), b1 = bf16_hi(wb);
      if (DO_ROW) {
        float x0, x1, y0, y1;
        mul2f(a0, a1, re, x0, x1);
        mul2f(b0, b1, ro, y0, y1);
        const uint32_t ba = sr_e2m1x2<false>(x0, x1, wra[2 * q], wra[2 * q + 1]);
        const uint32_t bb = sr_e2m1x2<false>(y0, y1, wrb[2 * q], wrb[2 * q + 1]);
        rowa |= ba << (8 * q);
        rowb |= bb << (8 * q);
        if (STATS && ok) {
          r_clamp += clamped2(x0, x1) + clamped2(y0, y1);
          r_flush += flushed2(a0, a1, ba) + flushed2(b0, b1, bb);
        }
      }
      // columns 2q (elements a0, b0) and 2q + 1 (a1, b1), rows 2p, 2p + 1
      const float y0 = __fmul_rn(a0, rc[2 * q]), y1 = __fmul_rn(b0, rc[2 * q]);
      const float z0 = __fmul_rn(a1, rc[2 * q + 1]), z1 = __fmul_rn(b1, rc[2 * q + 1]);
      const uint32_t by = sr_e2m1x2<!TWO_D>(y0, y1, wca[2 * q], wcb[2 * q]);
      const uint32_t bz = sr_e2m1x2<!TWO_D>(z0, z1, wca[2 * q + 1], wcb[2 * q + 1]);
      uint32_t& py = (p < 4) ? pcol[2 * q].x : pcol[2 * q].y;
      uint32_t& pz = (p < 4) ? pcol[2 * q + 1].x : pcol[2 * q + 1].y;
      py = put_byte(py, by, p & 3);
      pz = put_byte(pz, bz, p & 3);
      if (STATS && !TWO_D && ok) {
        c_clamp += clamped2(y0, y1) + clamped2(z0, z1);
        c_flush += flushed2(a0, b0, by) + flushed2(a1, b1, bz);
      }
    }
    if (DO_ROW && ok) {
      *reinterpret_cast<uint16_t*>(prow + (2 * p) * pstep) = (uint16_t)rowa;
      *reinterpret_cast<uint16_t*>(prow + (2 * p + 1) * pstep) = (uint16_t)rowb;
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint2*>(&stage.pay[stage_word(4 * lane + j, 2 * warp)]) = pcol[j];
  __syncthreads();
  write_col_stage(stage, R, C, (int64_t)ty * kRcRows, (int64_t)tx * kRcCols, pay_col, sc_col);
  if (STATS) {
    if (DO_ROW) flush_stats(stats, r_sat, r_uflow, r_clamp, r_flush);
    if (!TWO_D) flush_stats(stats + (DO_ROW ? 1 : 0), c_sat, c_uflow, c_clamp, c_flush);
  }
  flush_amax(amax_out, status, tmax);
}

// ---------------------------------------------------------------- dequantise
// v = (e * s) * T per element, one binary32 rounding each, then BF16 (RNE)
// or binary32.  One chunk = 8 elements = one payload word.  E2M1 -> FP16
// pairs by the hardware conversion (every E2M1 value is an FP16 value, so it
// is exact), then FP16 -> binary32 (exact); e * s is exact in binary32.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float v[8]) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
#pragma unroll
  for (int j = 0; j < 4; ++j)
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.f32.f16 %0, lo;\n\t"
        "cvt.f32.f16 %1, hi;\n\t}"
        : "=f"(v[2 * j]), "=f"(v[2 * j + 1]) : "r"(h[j]));
}

// Each warp walks groups of 32 * kDeqUnroll consecutive chunks (lane l takes
// chunks l, l + 32, ...): every load and store instruction of a warp covers
// one contiguous span, and kDeqUnroll payload words and scale bytes are in
// flight per thread before the first conversion.
constexpr int kDeqUnroll = 4;

template <bool F32>
__global__ void __launch_bounds__(256) dequantize_kernel(const uint32_t* __restrict__ payload,
                                                         const uint8_t* __restrict__ scales,
                                                         int64_t nchunks, int fmt,
                                                         const float* __restrict__ tscale,
                                                         void* __restrict__ out) {
  const float T = __ldg(tscale);
  const int lane = threadIdx.x & 31;
  const int64_t span = 32 * kDeqUnroll;
  const int64_t stride = (((int64_t)gridDim.x * blockDim.x) >> 5) * span;
  for (int64_t base = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * span + lane;
       base < nchunks; base += stride) {
    uint32_t p[kDeqUnroll], c[kDeqUnroll];
#pragma unroll
    for (int u = 0; u < kDeqUnroll; ++u) {
      const int64_t g = base + 32 * u;
      p[u] = g < nchunks ? __ldg(payload + g) : 0u;
      c[u] = g < nchunks ? __ldg(scales + (g >> 1)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kDeqUnroll; ++u) {
      const int64_t g = base + 32 * u;
      if (g >= nchunks) continue;
      const float s = decode_scale(c[u], fmt);
      float v[8];
      e2m1x8_to_f32(p[u], v);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(__fmul_rn(v[j], s), T);
      if (F32) {
        float4* o = reinterpret_cast<float4*>(out) + 2 * g;
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
      } else {
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h[j]) : "f"(v[2 * j + 1]), "f"(v[2 * j]));
        reinterpret_cast<uint4*>(out)[g] = make_uint4(h[0], h[1], h[2], h[3]);
      }
    }
  }
}

// ---------------------------------------------------------------- launchers
static int grid_for(int64_t work_items, int threads, int per_sm) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * per_sm;
  const int64_t g = need < cap ? need : cap;
  return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_amax(const void* in, int64_t n, float* out, int* status, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const int64_t nchunks = n / 8;
  const int ntail = (int)(n % 8);
  const uint16_t* tail = static_cast<const uint16_t*>(in) + nchunks * 8;
  amax_kernel<<<grid_for(nchunks > 0 ? nchunks : 1, 256, 8), 256, 0, st>>>(
      static_cast<const uint4*>(in), nchunks, tail, ntail, out, status);
  return cudaGetLastError();
}

cudaError_t launch_tensor_scale(const float* amax, float denom, float* out, cudaStream_t st) {
  tensor_scale_kernel<<<1, 1, 0, st>>>(amax, denom, out);
  return cudaGetLastError();
}

template <bool SR, bool STATS>
static void row_launch(const QuantArgs& a, cudaStream_t st) {
  const int64_t nchunks = a.rows * a.cols / 8;
  quantize_row_kernel<SR, STATS><<<grid_for(nchunks / 4, kRowThreads, 2), kRowThreads, 0, st>>>(
      static_cast<const uint4*>(a.in), nchunks, a.fmt, a.tscale, a.seed,
      reinterpret_cast<uint32_t*>(a.pay_row), a.sc_row, a.stats, a.amax_out, a.status);
}

template <bool SR, bool STATS, bool DO_ROW, bool TWO_D = false>
static cudaError_t tile_launch(const QuantArgs& a, cudaStream_t st) {
  const int64_t ntiles = ((a.cols + kRcCols - 1) / kRcCols) * ((a.rows + kRcRows - 1) / kRcRows);
  if (ntiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const uint16_t* in = static_cast<const uint16_t*>(a.in);
  uint32_t* pr = reinterpret_cast<uint32_t*>(a.pay_row);
  if constexpr (SR)
    quantize_tile4_kernel<STATS, DO_ROW, TWO_D><<<(unsigned)ntiles, kRcThreads, 0, st>>>(
        in, a.rows, a.cols, a.fmt, a.tscale, a.seed, a.pay_row, a.sc_row, a.pay_col, a.sc_col, a.stats,
        a.amax_out, a.status);
  else
    quantize_tile_kernel<STATS, DO_ROW, TWO_D><<<grid_for(ntiles * kRcThreads, kRcThreads, 2), kRcThreads, 0, st>>>(
        in, a.rows, a.cols, a.fmt, a.tscale, pr, a.sc_row, a.pay_col, a.sc_col, a.stats,
        a.amax_out, a.status);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st) {
  cudaError_t e;
  if (a.stats) {
    e = cudaMemsetAsync(a.stats, 0, sizeof(StatsDev) * (a.axis == 2 ? 2 : 1), st);
    if (e != cudaSuccess) return e;
  }
  if (a.amax_out) {
    e = cudaMemsetAsync(a.amax_out, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  if (a.rows == 0 || a.cols == 0) return cudaSuccess;
  const bool sr = a.sr, stats = a.stats != nullptr;
  if (a.axis == 0) {
    if (sr) stats ? row_launch<true, true>(a, st) : row_launch<true, false>(a, st);
    else stats ? row_launch<false, true>(a, st) : row_launch<false, false>(a, st);
    return cudaGetLastError();
  }
  if (a.axis == 1) {
    if (sr) return stats ? tile_launch<true, true, false>(a, st) : tile_launch<true, false, false>(a, st);
    return stats ? tile_launch<false, true, false>(a, st) : tile_launch<false, false, false>(a, st);
  }
  if (a.axis == 3) {   // one scale per 16 x 16 tile, both layouts
    if (sr) return stats ? tile_launch<true, true, true, true>(a, st) : tile_launch<true, false, true, true>(a, st);
    return stats ? tile_launch<false, true, true, true>(a, st) : tile_launch<false, false, true, true>(a, st);
  }
  if (sr) return stats ? tile_launch<true, true, true>(a, st) : tile_launch<true, false, true>(a, st);
  return stats ? tile_launch<false, true, true>(a, st) : tile_launch<false, false, true>(a, st);
}

cudaError_t launch_dequantize(const uint8_t* payload, const uint8_t* scales, int64_t rows,
                              int64_t cols, int fmt, const float* tscale, void* out, bool f32,
                              cudaStream_t st) {
  const int64_t nchunks = rows * cols / 8;
  if (nchunks == 0) return cudaSuccess;
  const int grid = grid_for((nchunks + kDeqUnroll - 1) / kDeqUnroll, 256, 8);
  if (f32)
    dequantize_kernel<true><<<grid, 256, 0, st>>>(reinterpret_cast<const uint32_t*>(payload), scales,
                                                  nchunks, fmt, tscale, out);
  else
    dequantize_kernel<false><<<grid, 256, 0, st>>>(reinterpret_cast<const uint32_t*>(payload), scales,
                                                   nchunks, fmt, tscale, out);
  return cudaGetLastError();
}

}  // namespace fp4q
