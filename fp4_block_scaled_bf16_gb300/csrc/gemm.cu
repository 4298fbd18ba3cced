// gemm.cu -- the emulated UE5M3 block-scaled GEMM of libfp4q.so on the
// sm_103a tensor cores (tcgen05 on SM pairs, TMEM accumulators, TMA, mbarrier
// pipeline).
//
// Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
// Abstract -- the FP4 matrix multiplications of every internal linear run on
// E2M1 payloads with UE5M3 block-16 scales, emulated in software because the
// tensor cores' native block-scale formats are E4M3/E8M0.
//
//   C[m, n] = (T_A T_B) * sum_k (e_a s_a)[m, k] * (e_b s_b)[n, k]
//
// Every product e * s has at most 6 significant bits and lies in
// [2^-18, 688128], so e * s * 2^-4 is exact in FP16; the contraction
// therefore runs as an FP16 x FP16 -> FP32 tcgen05 MMA (kind::f16) over
// operands expanded in shared memory, and differs from an exact sum only by
// FP32 accumulation rounding.
//
// Organisation.  A cluster of two CTAs (one per SM) computes a 256 x 512
// output tile with the two-SM MMA (cta_group::2, M256 N256 K16): CTA rank r
// holds A rows 128 r .. 128 r + 127 of the tile and, for each of the two
// N256 halves of the tile, B rows 128 r .. 128 r + 127 of that half; its TMEM
// holds its 128 rows of both 128 x 256 FP32 accumulators (all 512 columns).
// The expansion is the costly part, and the pair expands 384 rows per SM and
// K step for 128 x 512 outputs, a quarter fewer than one SM expanding the
// 512 rows of a 256 x 256 tile on its own.  Per CTA, K step 64:
//   warp 16     TMA producer: FP4 payload tiles (the CTA's 384 rows x 32 B)
//               into a 4-stage raw ring, and the scale codes (16 per row,
//               four K steps) into a 2-slot ring when K % 256 == 0.
//   warps 0..15 expand raw stages into a 3-stage FP16 ring laid out in the
//               128-byte-swizzled K-major form the MMA descriptors read; each
//               thread expands one 16-element block (one scale) at a time by
//               the E2M1 -> FP16 conversion and one exact FP16 multiply by
//               the block scale, then signal the rank-0 CTA's "full"
//               barrier; after the main loop they run the epilogue (TMEM ->
//               registers -> alpha -> BF16/FP32 -> global).
//   warp 17     allocates the pair's TMEM; in the rank-0 CTA one lane waits
//               until both CTAs have expanded a stage, issues its 8 MMAs
//               (2 x M256 N256 K16 per K16 step) and commits them to both
//               CTAs' "empty" barriers.
// Every wait is bounded: a wait that runs out latches FP4Q_ERR_TIMEOUT in the
// device status word and the CTA winds down instead of hanging; the loads
// and MMAs already issued are waited for (bounded) and both CTAs meet at a
// cluster barrier before either frees TMEM or exits, so that nothing still
// targets a CTA's shared memory or TMEM when it is released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "fp4q_device.cuh"
#include "fp4q_launch.h"
#include "fp4q_pipeline.cuh"
#include "fp4q_tcgen05.cuh"

namespace fp4q {
namespace gemm {

constexpr int PM = 256, PN = 512;              // output tile of a CTA pair
constexpr int AM = 128;                        // A rows per CTA = M of the MMA per CTA
constexpr int BH = 128;                        // B rows per CTA and N256 half
constexpr int UN = 256;                        // N of one MMA = TMEM columns of one accumulator
constexpr int ROWS = AM + 2 * BH;              // rows expanded per CTA and K step
constexpr int BK = 64;
constexpr int S_RAW = 4, S_BF = 3;
constexpr int RAW_STAGE = ROWS * BK / 2;       // 12288 B
constexpr int BF_PART = AM * BK * 2;           // 16384 B: A, then the two B parts
constexpr int BF_STAGE = ROWS * BK * 2;        // 49152 B
constexpr int kDeqWarps = 16;
constexpr int kDeqThreads = 32 * kDeqWarps;
constexpr int kProducerWarp = kDeqWarps, kMmaWarp = kDeqWarps + 1;
constexpr int kThreads = kDeqThreads + 64;
constexpr uint32_t kTmemCols = 512;            // two 128 x 256 FP32 accumulators
constexpr int kRowStride = kDeqThreads / 4;    // rows between a thread's rows
constexpr int kRowsPerThread = ROWS / kRowStride;
// epilogue: warps 4j .. 4j + 3 cover the 128 TMEM lanes (the CTA's rows);
// lane group j takes TMEM columns 128 j .. 128 j + 127
constexpr int kColGroups = kDeqWarps / 4;
constexpr int kColChunks = 2 * UN / kColGroups / 32;   // 32-column TMEM loads per warp
static_assert(kRowStride == AM && BH == AM && ROWS % kRowStride == 0, "row map: A, B0, B1 rows per thread");
static_assert(kDeqWarps % 4 == 0 && (2 * UN) % (32 * kColGroups) == 0, "epilogue map");

// Scale codes (when K is a multiple of 256): TMA boxes of 16 codes per row
// (four K steps) for the CTA's 384 rows, in a 2-slot ring.
constexpr int CODE_KB = 4;                     // K steps per code stage
constexpr int CODE_STAGE = ROWS * 16;          // 6144 B
constexpr int S_CODE = 2;

constexpr int OFF_BF = 0;
constexpr int OFF_RAW = OFF_BF + S_BF * BF_STAGE;
constexpr int OFF_CODE = OFF_RAW + S_RAW * RAW_STAGE;
constexpr int NBARS = 2 * S_RAW + 2 * S_BF + 1 + 2 * S_CODE;
static_assert(OFF_RAW % 1024 == 0 && OFF_CODE % 1024 == 0 && BF_PART % 1024 == 0, "alignment");
// Epilogue staging: the BF16 result (eight 128 x 64 boxes) in the idle FP16
// ring, the quantised result (two payload boxes 128 x 128 B, codes box
// 128 x 32 B) in the idle raw ring.
constexpr int OUT_BOX = AM * 128;              // one 128 x 64 BF16 box, or 128 x 128 B of payload
constexpr int QST_PAY = 2 * OUT_BOX, QST_BYTES = QST_PAY + AM * 32;
constexpr int OFF_QST = OFF_RAW;
static_assert(S_BF * BF_STAGE >= (2 * UN / 64) * OUT_BOX, "BF16 staging fits the FP16 ring");
static_assert(S_RAW * RAW_STAGE >= QST_BYTES && OFF_QST % 1024 == 0, "quantised staging fits the raw ring");
// Without the code ring the kernel leaves its 12 KB to L1, which then holds
// the scale codes it loads directly.
__host__ __device__ constexpr int off_bar(bool tma_codes) { return OFF_CODE + (tma_codes ? S_CODE * CODE_STAGE : 0); }
// after the barriers: TMEM address (8 B), abort flag (8 B), then the scale
// table of the epilogue quantisation
constexpr int TAB_BYTES = (int)((sizeof(ScaleTab) + 15) / 16 * 16);
__host__ __device__ constexpr int smem_bytes(bool tma_codes) {
  return off_bar(tma_codes) + 8 * NBARS + 16 + TAB_BYTES + 1024;   // + 1 KB alignment slack
}
static_assert(smem_bytes(true) <= 227 * 1024, "shared memory per CTA");

// ---------------------------------------------------------------- kind::f16 MMA
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// Instruction descriptor for kind::f16: FP32 accumulator, FP16 A and B (format
// code 0), both K-major, M = 256 (the pair), N = 256.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(UN >> 3) << 17) | ((uint32_t)((2 * AM) >> 4) << 24);

// ---------------------------------------------------------------- expansion
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Expansion of E2M1 x UE5M3 to FP16.  Every product e * s * 2^-4 is exact in
// FP16: e is a multiple of 1/2 with at most 2 significant bits, s * 2^-4 a
// multiple of 2^-21 with at most 4, so the product is a multiple of 2^-22
// (on the FP16 subnormal grid of 2^-24) with at most 6 significant bits, and
// at most 6 * 114688 / 16 = 43008 < 65504.  The nibbles become FP16 pairs by
// the hardware E2M1 -> FP16 conversion (exact), and one FP16 multiply by
// (s * 2^-4) applies the block scale; the 2^-8 of the two operands comes back
// in the epilogue's alpha.

// (s * 2^-4, s * 2^-4) as an FP16 pair.  The scale code shifted into a binary32
// exponent/mantissa field is s * 2^-(127 - bias), subnormal codes included.
__device__ __forceinline__ uint32_t scale_pair(uint32_t code, int fmt) {
  const float s = __fmul_rn(__uint_as_float(code << 20), fmt == kUE5M3 ? 0x1p112f : 0x1p120f);
  const float s4 = __fmul_rn(s, 0x1p-4f);
  uint32_t ss;
  asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(ss) : "f"(s4));   // exact: <= 4 significant bits
  return ss;
}

// Eight nibbles (byte j holds K elements 2j, 2j + 1) -> four FP16 pairs.  The
// pair order within a byte is whatever the conversion gives; it is the same
// for A and B, which leaves every dot product unchanged.
__device__ __forceinline__ uint4 expand8(uint32_t w, uint32_t ss) {
  uint4 o;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w) : "r"(w));
  o.x = hmul2(o.x, ss);
  o.y = hmul2(o.y, ss);
  o.z = hmul2(o.z, ss);
  o.w = hmul2(o.w, ss);
  return o;
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------- kernel
// QOUT: the epilogue also quantises the BF16 result row-wise (blocks of 16
// along N, round to nearest even, tensor scale TC) -- the input format of the
// next layer -- and records max |bf16(C)|; `out` may then be null.
// Launched in clusters of two along x: blockIdx.x / 2 indexes the 512-column
// tile, blockIdx.y the 256-row tile.
template <bool F32OUT, bool TMA_CODES, bool QOUT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const __grid_constant__ CUtensorMap mapAs, const __grid_constant__ CUtensorMap mapBs,
                const __grid_constant__ CUtensorMap mapC, int tma_store,
                const uint8_t* __restrict__ As, const uint8_t* __restrict__ Bs,
                const float* __restrict__ TA, const float* __restrict__ TB, int M, int N, int K,
                int fmt, void* __restrict__ out, int* status, long long budget, int skip_loads,
                const float* __restrict__ TC, uint8_t* __restrict__ qpay, uint8_t* __restrict__ qsc,
                float* qamax, const __grid_constant__ CUtensorMap mapQP,
                const __grid_constant__ CUtensorMap mapQS, int qstaged, const int* run_if) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  constexpr int OFF_BAR = off_bar(TMA_CODES);
  constexpr int OFF_TMEM = OFF_BAR + 8 * NBARS;
  constexpr int OFF_ABORT = OFF_TMEM + 8;
  constexpr int OFF_TAB = OFF_ABORT + 8;
  // conditional launch (fp4q_gemm_if): both CTAs return before any setup
  // unless the device flag is set
  if (run_if && !pair_read_flag(run_if, sb + OFF_ABORT + 4)) return;
  ScaleTab* tab = reinterpret_cast<ScaleTab*>(smem + OFF_TAB);
  const uint32_t bar_raw_full = sb + OFF_BAR;
  const uint32_t bar_raw_empty = bar_raw_full + 8 * S_RAW;
  const uint32_t bar_bf_full = bar_raw_empty + 8 * S_RAW;
  const uint32_t bar_bf_empty = bar_bf_full + 8 * S_BF;
  const uint32_t bar_acc = bar_bf_empty + 8 * S_BF;
  const uint32_t bar_code_full = bar_acc + 8;
  const uint32_t bar_code_empty = bar_code_full + 8 * S_CODE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int m0 = blockIdx.y * PM, n0 = (blockIdx.x >> 1) * PN;
  const int am0 = m0 + AM * (int)rank;                 // this CTA's A rows
  const int bn0 = n0 + BH * (int)rank;                 // its B rows of the first N256 half
  const int bn1 = bn0 + UN;                            // ... and of the second
  const int nk = K / BK;

  if (QOUT) build_scale_tab(tab, __ldg(TC), fmt);   // block-wide, before the roles split
  if (threadIdx.x == 0) {
    for (int i = 0; i < S_RAW; ++i) {
      mbar_init(bar_raw_full + 8 * i, 1);
      mbar_init(bar_raw_empty + 8 * i, kDeqWarps);
    }
    for (int i = 0; i < S_BF; ++i) {
      mbar_init(bar_bf_full + 8 * i, 2 * kDeqWarps);   // every expansion warp of both CTAs (used in rank 0)
      mbar_init(bar_bf_empty + 8 * i, 1);
    }
    mbar_init(bar_acc, 1);
    for (int i = 0; i < S_CODE; ++i) {
      mbar_init(bar_code_full + 8 * i, 1);
      mbar_init(bar_code_empty + 8 * i, kDeqWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc_pair(sb + OFF_TMEM, kTmemCols);
  tc_fence_before();
  cluster_sync();   // both CTAs' barriers initialised before either arrives on the other's
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);

  if (warp == kProducerWarp) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_kb = -1, last_g = -1;   // the last K step / code stage whose loads were issued
      for (int kb = 0; kb < nk; ++kb) {
        if (TMA_CODES && kb % CODE_KB == 0) {
          const int g = kb / CODE_KB, cs = g % S_CODE;
          if (!mbar_wait(bar_code_empty + 8 * cs, ((g / S_CODE) & 1) ^ 1, abort_flag, budget)) {
            fail(abort_flag, status);
            break;
          }
          if (!skip_loads) {
            const uint32_t cdst = sb + OFF_CODE + cs * CODE_STAGE;
            mbar_expect_tx(bar_code_full + 8 * cs, CODE_STAGE);
            tma_load_2d(cdst, &mapAs, g * 16, am0, bar_code_full + 8 * cs);
            tma_load_2d(cdst + AM * 16, &mapBs, g * 16, bn0, bar_code_full + 8 * cs);
            tma_load_2d(cdst + (AM + BH) * 16, &mapBs, g * 16, bn1, bar_code_full + 8 * cs);
            last_g = g;
          }
        }
        const int s = kb % S_RAW;
        if (!mbar_wait(bar_raw_empty + 8 * s, ((kb / S_RAW) & 1) ^ 1, abort_flag, budget)) {
          fail(abort_flag, status);
          break;
        }
        const uint32_t dst = sb + OFF_RAW + s * RAW_STAGE;
        if (skip_loads) continue;   // test hook: consumers' waits run out
        mbar_expect_tx(bar_raw_full + 8 * s, RAW_STAGE);
        tma_load_2d(dst, &mapA, kb * (BK / 2), am0, bar_raw_full + 8 * s);
        tma_load_2d(dst + AM * (BK / 2), &mapB, kb * (BK / 2), bn0, bar_raw_full + 8 * s);
        tma_load_2d(dst + (AM + BH) * (BK / 2), &mapB, kb * (BK / 2), bn1, bar_raw_full + 8 * s);
        last_kb = kb;
      }
      // Drain, also after an abort: a load already issued still lands in this
      // CTA's shared memory, so the CTA must not exit before it has.  A stage
      // is refilled only after its previous contents were consumed, so only
      // the last load into each stage can still be in flight; wait for each
      // of those (bounded, whatever the abort flag says).
      bool drained = true;
      for (int s = 0; s < S_RAW; ++s) {
        if (last_kb < s) continue;
        const int kb = s + (last_kb - s) / S_RAW * S_RAW;
        drained &= mbar_wait_bounded(bar_raw_full + 8 * s, (kb / S_RAW) & 1, kDrainCycles);
      }
      for (int cs = 0; TMA_CODES && cs < S_CODE; ++cs) {
        if (last_g < cs) continue;
        const int g = cs + (last_g - cs) / S_CODE * S_CODE;
        drained &= mbar_wait_bounded(bar_code_full + 8 * cs, (g / S_CODE) & 1, kDrainCycles);
      }
      if (!drained) atomicOr(status, kStatusTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0) {
      if (rank == 0) {
        for (int kb = 0; kb < nk; ++kb) {
          const int t = kb % S_BF;
          if (!mbar_wait_cluster(bar_bf_full + 8 * t, (kb / S_BF) & 1, abort_flag, budget)) {
            fail(abort_flag, status);
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sb + OFF_BF + t * BF_STAGE;
          const uint64_t ad = sw128_desc(a_addr);
          const uint64_t b0 = sw128_desc(a_addr + BF_PART), b1 = sw128_desc(a_addr + 2 * BF_PART);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
            mma_f16_pair(tmem, ad + 2 * k, b0 + 2 * k, kIdesc, acc);        // columns 0..255
            mma_f16_pair(tmem + UN, ad + 2 * k, b1 + 2 * k, kIdesc, acc);   // columns 256..511
          }
          mma_commit_pair(bar_bf_empty + 8 * t);
        }
        mma_commit_pair(bar_acc);
      }
      // Drain, also after an abort: bar_acc completes (in both CTAs) once
      // every MMA issued above has finished reading both CTAs' shared memory
      // and writing their TMEM, which must happen before TMEM is freed and
      // either CTA exits (bounded, whatever the abort flag says).
      if (!mbar_wait_bounded(bar_acc, 0, kDrainCycles)) atomicOr(status, kStatusTimeout);
    }
  } else {
    // ------------------------------------------------ expansion warps
    // Thread t expands block (t % 4) of the 64-wide K step for row t/4 of
    // the CTA's A rows, of its first B part and of its second B part.
    const int tid = threadIdx.x;
    const int blk = tid & 3;
    const int rbase = tid >> 2;
    const int64_t lds_k = K / 16;
    const uint8_t* srow[kRowsPerThread];
    bool rok[kRowsPerThread];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int gr = (i == 0 ? am0 : i == 1 ? bn0 : bn1) + rbase;
      rok[i] = (i == 0) ? (gr < M) : (gr < N);
      srow[i] = ((i == 0) ? As : Bs) + (int64_t)(rok[i] ? gr : 0) * lds_k + blk;
    }
    auto load_codes = [&](int kb, uint32_t (&c)[kRowsPerThread]) {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) c[i] = (rok[i] && kb < nk) ? __ldg(srow[i] + kb * 4) : 0u;
    };
    // scale codes are prefetched two K steps ahead (their L2 latency is
    // longer than one step of expansion)
    uint32_t c0[kRowsPerThread], c1[kRowsPerThread], c2[kRowsPerThread];
    if (!TMA_CODES) {
      load_codes(0, c0);
      load_codes(1, c1);
    }
    const uint32_t sw = rbase & 7;               // (rbase + kRowStride i) & 7
    const uint32_t c_lo = ((2 * blk) ^ sw) << 4, c_hi = ((2 * blk + 1) ^ sw) << 4;
    int s = 0, t = 0;
    uint32_t ph_s = 0, ph_t = 1;
    for (int kb = 0; kb < nk; ++kb) {
      const int g = kb / CODE_KB, cs = g % S_CODE;
      if (TMA_CODES) {
        if (kb % CODE_KB == 0 &&
            !mbar_wait(bar_code_full + 8 * cs, (g / S_CODE) & 1, abort_flag, budget)) {
          fail(abort_flag, status);
          break;
        }
        const uint32_t code = sb + OFF_CODE + cs * CODE_STAGE + rbase * 16 + (kb % CODE_KB) * 4 + blk;
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) c0[i] = lds_u8(code + i * kRowStride * 16);
      } else {
        load_codes(kb + 2, c2);
      }
      if (!mbar_wait(bar_raw_full + 8 * s, ph_s, abort_flag, budget) ||
          !mbar_wait(bar_bf_empty + 8 * t, ph_t, abort_flag, budget)) {
        fail(abort_flag, status);
        break;
      }
      const uint32_t raw = sb + OFF_RAW + s * RAW_STAGE + rbase * (BK / 2) + blk * 8;
      const uint32_t bf = sb + OFF_BF + t * BF_STAGE + rbase * 128;
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const uint2 w = lds64(raw + i * kRowStride * (BK / 2));
        const uint32_t ss = scale_pair(c0[i], fmt);
        const uint4 lo = expand8(w.x, ss);         // K 16*blk + 0..7
        const uint4 hi = expand8(w.y, ss);         // K 16*blk + 8..15
        const uint32_t row_addr = bf + i * kRowStride * 128;
        sts128(row_addr + c_lo, lo);
        sts128(row_addr + c_hi, hi);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_rank0(bar_bf_full + 8 * t);
        mbar_arrive(bar_raw_empty + 8 * s);
        if (TMA_CODES && (kb % CODE_KB == CODE_KB - 1 || kb == nk - 1)) mbar_arrive(bar_code_empty + 8 * cs);
      }
      if (!TMA_CODES) {
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) { c0[i] = c1[i]; c1[i] = c2[i]; }
      }
      if (++s == S_RAW) { s = 0; ph_s ^= 1; }
      if (++t == S_BF) { t = 0; ph_t ^= 1; }
    }

    // ------------------------------------------------ epilogue
    // warp w drains TMEM lanes 32 (w % 4) .. +31 (the CTA's rows), columns
    // 128 (w / 4) .. +127 (accumulator 0 holds output columns 0..255, 1 the
    // rest).  BF16 output with a tensor map: the CTA's 128 x 512 result is
    // staged in the idle FP16 ring as eight 128 x 64 boxes (128-byte
    // swizzled) and leaves by TMA stores, whole lines; otherwise every
    // thread stores its 32 values directly.
    const bool staged = !F32OUT && tma_store;
    // quantised result staged in the idle raw ring (two payload boxes
    // 128 x 128 B, 128-byte swizzled; codes box 128 x 32 B) and stored by TMA
    const bool qst = QOUT && qstaged;
    const bool drained = mbar_wait(bar_acc, 0, abort_flag, budget);
    if (drained) {
      tc_fence_after();
      const int q = warp & 3, grp = warp >> 2;
      // T_A T_B, times 2^8 for the 2^-4 on each operand (exact)
      const float alpha = __fmul_rn(__fmul_rn(__ldg(TA), __ldg(TB)), 256.0f);
      const int rt = 32 * q + lane;                       // row within the CTA's 128
      const int row = am0 + rt;
      const bool vec = F32OUT ? (N % 4 == 0) : (N % 8 == 0);
      uint32_t qmax = 0;
      ScaleRegs kr{};
      if (QOUT) kr = scale_regs(*tab);
#pragma unroll 1
      for (int c = 0; c < kColChunks; ++c) {
        const int ct = 32 * (kColChunks * grp + c);        // column within the 512
        const int col0 = n0 + ct;
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)ct, r);
        const bool live = row < M && col0 < N;
        if (!staged && !live) continue;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), alpha);
        if (F32OUT) {
          float* o = static_cast<float*>(out) + (int64_t)row * N + col0;
          if (vec && col0 + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              reinterpret_cast<float4*>(o)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            for (int j = 0; j < 32 && col0 + j < N; ++j) o[j] = v[j];
          }
        } else {
          uint32_t h[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h[j]) : "f"(v[2 * j + 1]), "f"(v[2 * j]));
          if (staged) {
            // box ct / 64, row rt, 16-byte chunks (ct % 64) / 8 + i, swizzled by row
            const uint32_t rowb = sb + OFF_BF + (uint32_t)(ct >> 6) * OUT_BOX + (uint32_t)rt * 128;
            const int ch0 = (ct & 63) >> 3;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              sts128(rowb + ((uint32_t)((ch0 + i) ^ (rt & 7)) << 4),
                     make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]));
          } else if (out != nullptr) {
            uint16_t* o = static_cast<uint16_t*>(out) + (int64_t)row * N + col0;
            if (vec && col0 + 32 <= N) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                reinterpret_cast<uint4*>(o)[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
            } else {
              for (int j = 0; j < 32 && col0 + j < N; ++j)
                o[j] = (uint16_t)((j & 1) ? (h[j >> 1] >> 16) : (h[j >> 1] & 0xFFFFu));
            }
          }
          if (QOUT && live) {
            // two blocks of 16 along N (N % 32 == 0: a chunk is wholly inside)
            uint32_t pw[4], codes = 0, cl = 0, fl = 0;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              const uint32_t a = max(absmax16(h + 8 * b), absmax16(h + 8 * b + 4));
              qmax = max(qmax, a);
              const BlockScale bs = block_scale<false>(a, *tab, kr);
              pw[2 * b] = quantize8<false, false>(h + 8 * b, bs.r, nullptr, &cl, &fl);
              pw[2 * b + 1] = quantize8<false, false>(h + 8 * b + 4, bs.r, nullptr, &cl, &fl);
              codes |= bs.code << (8 * b);
            }
            if (qst) {
              // payload box ct / 256, row rt, 16-byte chunk (ct % 256) / 32, swizzled by row
              sts128(sb + OFF_QST + (uint32_t)(ct >> 8) * OUT_BOX + (uint32_t)rt * 128 +
                         ((uint32_t)(((ct & 255) >> 5) ^ (rt & 7)) << 4),
                     make_uint4(pw[0], pw[1], pw[2], pw[3]));
              asm volatile("st.shared.u16 [%0], %1;" ::"r"(sb + OFF_QST + QST_PAY + (uint32_t)rt * 32 + (ct >> 4)),
                           "h"((unsigned short)codes) : "memory");
            } else {
              *reinterpret_cast<uint4*>(qpay + (int64_t)row * (N / 2) + col0 / 2) =
                  make_uint4(pw[0], pw[1], pw[2], pw[3]);
              *reinterpret_cast<uint16_t*>(qsc + (int64_t)row * (N / 16) + col0 / 16) = (uint16_t)codes;
            }
          }
        }
      }
      if (QOUT) {
        // max |bf16(C)| (a 16-bit pattern; inf/NaN compare above every finite)
        qmax = __reduce_max_sync(0xFFFFFFFFu, qmax);
        if (lane == 0) {
          if (qmax >= 0x7F80u) atomicOr(status, kStatusNonFinite);
          if (qamax && qmax) atomicMax(reinterpret_cast<unsigned int*>(qamax), qmax << 16);
        }
      }
    } else {
      fail(abort_flag, status);
    }
    if (staged || qst) {
      // every expansion warp passes here exactly once, drained or not
      fence_proxy_async();
      asm volatile("bar.sync 1, %0;" ::"n"(kDeqThreads) : "memory");
      // boxes that start inside the result only (a ragged edge is clipped by
      // the store itself)
      if (threadIdx.x == 0 && drained && !*abort_flag && am0 < M) {
        if (staged) {
          for (int j = 0; j < 2 * UN / 64 && n0 + 64 * j < N; ++j)
            tma_store_2d(&mapC, sb + OFF_BF + j * OUT_BOX, n0 + 64 * j, am0);
        }
        if (qst) {
          tma_store_2d(&mapQP, sb + OFF_QST, n0 / 2, am0);
          if (n0 + 256 < N) tma_store_2d(&mapQP, sb + OFF_QST + OUT_BOX, n0 / 2 + 128, am0);
          tma_store_2d(&mapQS, sb + OFF_QST + QST_PAY, n0 / 16, am0);
        }
        tma_store_commit_and_wait_read();
      }
    }
  }

  // Both CTAs meet here once their loads, MMAs and remote arrivals are done;
  // only then is the pair's TMEM freed.
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace gemm

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D uint8 tensor map over a [rows, K/2] payload, box (32 B, box_rows),
// out-of-range rows read as zero.
static bool make_payload_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K,
                             uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  const cuuint32_t box[2] = {(cuuint32_t)(gemm::BK / 2), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 tensor map over a [rows, K/16] scale array, box (16 codes,
// box_rows); needs a row stride that is a multiple of 16 bytes (K % 256 == 0).
static bool make_code_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K,
                          uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (!fn || (K / 16) % 16 != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 16), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 16)};
  const cuuint32_t box[2] = {16u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D BF16 tensor map over the [M, N] output, box (64 columns, 128 rows),
// 128-byte swizzle; needs a row stride that is a multiple of 16 bytes.
static bool make_out_map(CUtensorMap* map, void* base, int64_t M, int64_t N) {
  auto fn = get_encode_fn();
  if (!fn || N % 8 != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)(N * 2)};
  const cuuint32_t box[2] = {64u, (cuuint32_t)gemm::AM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 tensor maps over the row-wise quantised result: payload [M, N/2]
// with box (128 B, 128 rows) and 128-byte swizzle; codes [M, N/16] with box
// (32 B, 128 rows).  Need row strides that are multiples of 16 bytes.
static bool make_qout_maps(CUtensorMap* mp, CUtensorMap* ms, uint8_t* pay, uint8_t* sc, int64_t M, int64_t N) {
  auto fn = get_encode_fn();
  if (!fn || N % 256 != 0) return false;
  const cuuint32_t estr[2] = {1, 1};
  const cuuint64_t pd[2] = {(cuuint64_t)(N / 2), (cuuint64_t)M};
  const cuuint64_t ps[1] = {(cuuint64_t)(N / 2)};
  const cuuint32_t pb[2] = {128u, (cuuint32_t)gemm::AM};
  const cuuint64_t sd[2] = {(cuuint64_t)(N / 16), (cuuint64_t)M};
  const cuuint64_t ss[1] = {(cuuint64_t)(N / 16)};
  const cuuint32_t sbx[2] = {32u, (cuuint32_t)gemm::AM};
  return fn(mp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, pay, pd, ps, pb, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
         fn(ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, sc, sd, ss, sbx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool F32OUT, bool TMA_CODES, bool QOUT = false>
static cudaError_t launch_gemm_t(const GemmArgs& a, const CUtensorMap& mapA, const CUtensorMap& mapB,
                                 const CUtensorMap& mapAs, const CUtensorMap& mapBs,
                                 const CUtensorMap& mapC, bool tma_store, cudaStream_t st) {
  CUtensorMap mapQP, mapQS;
  const bool qstaged = QOUT && make_qout_maps(&mapQP, &mapQS, a.qpay, a.qsc, a.M, a.N);
  if (!qstaged) {
    memset(&mapQP, 0, sizeof(mapQP));
    memset(&mapQS, 0, sizeof(mapQS));
  }
  constexpr int smem = gemm::smem_bytes(TMA_CODES);
  auto kern = gemm::gemm_kernel<F32OUT, TMA_CODES, QOUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * (unsigned)((a.N + gemm::PN - 1) / gemm::PN), (unsigned)((a.M + gemm::PM - 1) / gemm::PM));
  cfg.blockDim = dim3(gemm::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mapA, mapB, mapAs, mapBs, mapC, tma_store ? 1 : 0, a.As, a.Bs, a.TA, a.TB,
                         (int)a.M, (int)a.N, (int)a.K, a.fmt, a.out, a.status, a.wait_cycles,
                         a.skip_loads ? 1 : 0, a.TC, a.qpay, a.qsc, a.qamax, mapQP, mapQS, qstaged ? 1 : 0, a.run_if);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t st) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  CUtensorMap mapA, mapB, mapAs, mapBs;
  if (!make_payload_map(&mapA, a.A, a.M, a.K, gemm::AM) || !make_payload_map(&mapB, a.B, a.N, a.K, gemm::BH))
    return cudaErrorNotSupported;
  const bool tma_codes = make_code_map(&mapAs, a.As, a.M, a.K, gemm::AM) &&
                         make_code_map(&mapBs, a.Bs, a.N, a.K, gemm::BH);
  if (!tma_codes) {
    memset(&mapAs, 0, sizeof(mapAs));   // unused by the direct-load instantiation
    memset(&mapBs, 0, sizeof(mapBs));
  }
  CUtensorMap mapC;
  const bool tma_store = !a.out_f32 && a.out != nullptr && make_out_map(&mapC, a.out, a.M, a.N);
  if (!tma_store) memset(&mapC, 0, sizeof(mapC));
  if (a.qpay) {   // epilogue quantisation (BF16 result)
    if (a.qamax && a.zero_qamax) {
      cudaError_t e = cudaMemsetAsync(a.qamax, 0, sizeof(float), st);
      if (e != cudaSuccess) return e;
    }
    return tma_codes ? launch_gemm_t<false, true, true>(a, mapA, mapB, mapAs, mapBs, mapC, tma_store, st)
                     : launch_gemm_t<false, false, true>(a, mapA, mapB, mapAs, mapBs, mapC, tma_store, st);
  }
  if (a.out_f32)
    return tma_codes ? launch_gemm_t<true, true>(a, mapA, mapB, mapAs, mapBs, mapC, false, st)
                     : launch_gemm_t<true, false>(a, mapA, mapB, mapAs, mapBs, mapC, false, st);
  return tma_codes ? launch_gemm_t<false, true>(a, mapA, mapB, mapAs, mapBs, mapC, tma_store, st)
                   : launch_gemm_t<false, false>(a, mapA, mapB, mapAs, mapBs, mapC, tma_store, st);
}

}  // namespace fp4q
