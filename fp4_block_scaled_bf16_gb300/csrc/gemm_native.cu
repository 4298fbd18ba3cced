// gemm_native.cu -- the native NVFP4 GEMM of libfp4q.so on sm_103a: E2M1
// operands with UE4M3 block-16 scales multiplied by the tensor cores' own
// block-scaled MMA (tcgen05.mma kind::mxf4nvf4, scale_vec::4X), TMEM
// accumulators, TMA, mbarrier pipeline.
//
// Method: "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
// Abstract -- the native NVFP4 execution the page ablates against (UE4M3
// block scales are what the tensor cores take; UE5M3 is emulated, see
// gemm.cu).  Same contraction and operand layout as fp4q_gemm with UE4M3
// scales:  C[m, n] = (T_A T_B) sum_k (e_a s_a)[m, k] (e_b s_b)[n, k].
//
// CTA organisation (one CTA per SM, 128 x 256 output tile, 256 K elements per
// stage = one 128-byte swizzled row of packed E2M1 per operand row):
//   warp 8      TMA producer: payload tiles of A (128 x 128 B) and B
//               (256 x 128 B), 128-byte swizzled as the MMA descriptors read
//               them, and the stage's scale codes (16 per row) into a
//               4-stage ring.
//   warps 0..3  copy the stage's scale codes into TMEM (tcgen05.st), warp q
//               into lane quadrant q, all four the same data: for each of the
//               stage's four K64 MMAs, the 32-bit word of row r (its four
//               block scales, the first K block in the low byte) goes to
//               lane r mod 32, column base + r / 32 -- B's 256 rows in eight
//               columns, A's 128 rows in four (the scale-factor layout of the
//               block-scaled MMA: every lane quadrant sees every row).
//   warp 9      allocates TMEM (accumulator in columns 0..255, the scale
//               ring in 256..511); one lane issues four MMAs
//               (M128 N256 K64) per stage and commits them to the stage's
//               "empty" barrier.
//   warps 0..7  epilogue: TMEM -> registers -> alpha -> BF16 staged in the
//               idle ring, stored by TMA (or FP32 stored directly).
// Every wait is bounded; a wait that runs out latches FP4Q_ERR_TIMEOUT and
// the CTA exits once the loads and MMAs it issued have completed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "fp4q_device.cuh"
#include "fp4q_launch.h"
#include "fp4q_pipeline.cuh"
#include "fp4q_tcgen05.cuh"

namespace fp4q {
namespace native {

constexpr int BM = 128, BN = 256, BK = 256;      // CTA tile, K elements per stage
constexpr int ROWB = BK / 2;                     // payload bytes per row per stage (128)
constexpr int S = 4;                             // ring stages
constexpr int A_BYTES = BM * ROWB;               // 16384
constexpr int B_BYTES = BN * ROWB;               // 32768
constexpr int SA_BYTES = BM * (BK / 16);         // 2048: 16 scale codes per row
constexpr int SB_BYTES = BN * (BK / 16);         // 4096
constexpr int OFF_A = 0, OFF_B = A_BYTES, OFF_SA = OFF_B + B_BYTES, OFF_SB = OFF_SA + SA_BYTES;
constexpr int STAGE = OFF_SB + SB_BYTES;         // 55296 = 54 KB
static_assert(STAGE % 1024 == 0 && OFF_B % 1024 == 0 && OFF_SA % 128 == 0 && OFF_SB % 128 == 0, "alignment");
constexpr int MMAS = BK / 64;                    // four K64 MMAs per stage
constexpr int kSfWarps = 4, kEpiWarps = 8;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 32 * 10;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;                // scale ring: stage s at 256 + 64 s
constexpr uint32_t kSfStageCols = 64;            // per MMA 16 columns: B (8) then A (4)
static_assert(kSfCol0 + S * kSfStageCols <= kTmemCols && BN <= (int)kSfCol0, "TMEM map");
constexpr int NBARS = 3 * S + 1;
constexpr int OFF_BAR = S * STAGE;
constexpr int OFF_TMEM = OFF_BAR + 8 * NBARS;
constexpr int OFF_ABORT = OFF_TMEM + 8;
constexpr int SMEM_BYTES = OFF_ABORT + 8 + 1024;   // + 1 KB alignment slack
// epilogue: the BF16 tile as four 128 x 64 boxes (128-byte swizzled) in the idle ring
static_assert(4 * BM * 128 <= S * STAGE, "BF16 staging fits the ring");

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1), both
// K-major, UE4M3 scales (bit 23 clear), scale-factor data IDs 0,
// N = 256 (bits 17..22: N / 8), M = 128 (bits 24..28: M / 16); dense.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_nvfp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t sfa,
                                          uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(sfa), "r"(sfb), "r"(accum)
      : "memory");
}

// Sixteen 32-bit columns of this warp's TMEM lane quadrant.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                      const __grid_constant__ CUtensorMap mapSA, const __grid_constant__ CUtensorMap mapSB,
                      const __grid_constant__ CUtensorMap mapC, int tma_store, const float* __restrict__ TA,
                      const float* __restrict__ TB, int M, int N, int K, void* __restrict__ out, int* status,
                      long long budget) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar_full = sb + OFF_BAR;            // TMA bytes of stage s landed
  const uint32_t bar_sf = bar_full + 8 * S;          // stage s scales written to TMEM
  const uint32_t bar_empty = bar_sf + 8 * S;         // stage s MMAs completed
  const uint32_t bar_acc = bar_empty + 8 * S;        // every MMA completed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nk = K / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_sf + 8 * i, kSfWarps);
      mbar_init(bar_empty + 8 * i, 1);
    }
    mbar_init(bar_acc, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) tmem_alloc(sb + OFF_TMEM, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);

  if (warp == kProducerWarp) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_kb = -1;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % S;
        if (!mbar_wait(bar_empty + 8 * s, ((kb / S) & 1) ^ 1, abort_flag, budget)) {
          fail(abort_flag, status);
          break;
        }
        const uint32_t st = sb + s * STAGE;
        mbar_expect_tx(bar_full + 8 * s, STAGE);
        tma_load_2d(st + OFF_A, &mapA, kb * ROWB, m0, bar_full + 8 * s);
        tma_load_2d(st + OFF_B, &mapB, kb * ROWB, n0, bar_full + 8 * s);
        tma_load_2d(st + OFF_SA, &mapSA, kb * (BK / 16), m0, bar_full + 8 * s);
        tma_load_2d(st + OFF_SB, &mapSB, kb * (BK / 16), n0, bar_full + 8 * s);
        last_kb = kb;
      }
      // Drain, also after an abort: only the last load into each stage can
      // still be in flight (a stage is refilled only after its MMAs read it).
      bool drained = true;
      for (int s = 0; s < S; ++s) {
        if (last_kb < s) continue;
        const int kb = s + (last_kb - s) / S * S;
        drained &= mbar_wait_bounded(bar_full + 8 * s, (kb / S) & 1, kDrainCycles);
      }
      if (!drained) atomicOr(status, kStatusTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % S;
        const uint32_t ph = (kb / S) & 1;
        if (!mbar_wait(bar_full + 8 * s, ph, abort_flag, budget) ||
            !mbar_wait(bar_sf + 8 * s, ph, abort_flag, budget)) {
          fail(abort_flag, status);
          break;
        }
        tc_fence_after();
        const uint32_t st = sb + s * STAGE;
        const uint64_t ad = sw128_desc(st + OFF_A), bd = sw128_desc(st + OFF_B);
#pragma unroll
        for (int i = 0; i < MMAS; ++i) {
          const uint32_t sf = tmem + kSfCol0 + kSfStageCols * s + 16 * i;
          mma_nvfp4(tmem, ad + 2 * i, bd + 2 * i, sf + 8, sf, (kb | i) != 0 ? 1u : 0u);
        }
        mma_commit(bar_empty + 8 * s);
      }
      mma_commit(bar_acc);
      // Drain, also after an abort: every MMA issued above completes before
      // TMEM is freed.
      if (!mbar_wait_bounded(bar_acc, 0, kDrainCycles)) atomicOr(status, kStatusTimeout);
    }
  } else {
    if (warp < kSfWarps) {
      // ------------------------------------------------ scale codes -> TMEM
      // lane r0 of warp q writes TMEM lane 32 q + r0: for MMA i, column
      // 16 i + j holds the word of B row r0 + 32 j (j < 8), column
      // 16 i + 8 + j the word of A row r0 + 32 j (j < 4).
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % S;
        if (!mbar_wait(bar_full + 8 * s, (kb / S) & 1, abort_flag, budget)) {
          fail(abort_flag, status);
          break;
        }
        const uint32_t st = sb + s * STAGE;
        uint4 a[4], b[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = lds128(st + OFF_SA + (uint32_t)(lane + 32 * j) * 16);
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = lds128(st + OFF_SB + (uint32_t)(lane + 32 * j) * 16);
        const uint32_t col = tmem + ((uint32_t)(32 * warp) << 16) + kSfCol0 + kSfStageCols * s;
#pragma unroll
        for (int i = 0; i < MMAS; ++i) {
          uint32_t v[16];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = word_of(b[j], i);
#pragma unroll
          for (int j = 0; j < 4; ++j) v[8 + j] = word_of(a[j], i);
#pragma unroll
          for (int j = 12; j < 16; ++j) v[j] = 0u;
          tmem_st16(col + 16 * i, v);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sf + 8 * s);
      }
    }
    // ------------------------------------------------ epilogue (warps 0..7)
    // warp w drains TMEM lanes 32 (w % 4) .. +31, columns 128 (w / 4) .. +127
    const bool staged = !F32OUT && tma_store;
    const bool drained = mbar_wait(bar_acc, 0, abort_flag, budget);
    if (drained) {
      tc_fence_after();
      const int q = warp & 3, h = warp >> 2;
      const float alpha = __fmul_rn(__ldg(TA), __ldg(TB));
      const int rt = 32 * q + lane;
      const int row = m0 + rt;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int ct = 128 * h + 32 * c;
        const int col0 = n0 + ct;
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)ct, r);
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), alpha);
        if (F32OUT) {
          if (row < M) {
            float* o = static_cast<float*>(out) + (int64_t)row * N + col0;
            if (N % 4 == 0 && col0 + 32 <= N) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                reinterpret_cast<float4*>(o)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            } else {
              for (int j = 0; j < 32 && col0 + j < N; ++j) o[j] = v[j];
            }
          }
        } else {
          uint32_t hh[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hh[j]) : "f"(v[2 * j + 1]), "f"(v[2 * j]));
          if (staged) {
            // box ct / 64, row rt, 16-byte chunks (ct % 64) / 8 + i, swizzled by row
            const uint32_t rowb = sb + (uint32_t)(ct >> 6) * (BM * 128) + (uint32_t)rt * 128;
            const int ch0 = (ct & 63) >> 3;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              sts128(rowb + ((uint32_t)((ch0 + i) ^ (rt & 7)) << 4),
                     make_uint4(hh[4 * i], hh[4 * i + 1], hh[4 * i + 2], hh[4 * i + 3]));
          } else if (row < M) {
            uint16_t* o = static_cast<uint16_t*>(out) + (int64_t)row * N + col0;
            if (N % 8 == 0 && col0 + 32 <= N) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                reinterpret_cast<uint4*>(o)[j] = make_uint4(hh[4 * j], hh[4 * j + 1], hh[4 * j + 2], hh[4 * j + 3]);
            } else {
              for (int j = 0; j < 32 && col0 + j < N; ++j)
                o[j] = (uint16_t)((j & 1) ? (hh[j >> 1] >> 16) : (hh[j >> 1] & 0xFFFFu));
            }
          }
        }
      }
    } else {
      fail(abort_flag, status);
    }
    if (staged) {
      // every epilogue warp passes here exactly once, drained or not
      fence_proxy_async();
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      if (threadIdx.x == 0 && drained && !*abort_flag) {
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) tma_store_2d(&mapC, sb + j * (BM * 128), n0 + 64 * j, m0);
        tma_store_commit_and_wait_read();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace native

// ---------------------------------------------------------------- host side
// 2-D uint8 tensor map, 128-byte swizzle: [rows, K/2] payload, box
// (128 B, box_rows) -- one stage of K for box_rows rows.
static bool make_swizzled_payload_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K,
                                      uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  const cuuint32_t box[2] = {(cuuint32_t)native::ROWB, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, K/16] scale codes, box (16 codes, box_rows); K % 256 == 0 keeps the
// row stride a multiple of 16 bytes.
static bool make_scale_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K, uint32_t box_rows) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 16), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 16)};
  const cuuint32_t box[2] = {(cuuint32_t)(native::BK / 16), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [M, N] BF16 output, box (64 columns, 128 rows), 128-byte swizzle.
static bool make_native_out_map(CUtensorMap* map, void* base, int64_t M, int64_t N) {
  auto fn = get_encode_fn();
  if (!fn || N % 8 != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)(N * 2)};
  const cuuint32_t box[2] = {64u, (cuuint32_t)native::BM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool F32OUT>
static cudaError_t launch_native_t(const GemmArgs& a, const CUtensorMap& mA, const CUtensorMap& mB,
                                   const CUtensorMap& mSA, const CUtensorMap& mSB, const CUtensorMap& mC,
                                   bool tma_store, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(native::gemm_nvfp4_kernel<F32OUT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, native::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.N + native::BN - 1) / native::BN), (unsigned)((a.M + native::BM - 1) / native::BM));
  native::gemm_nvfp4_kernel<F32OUT><<<grid, native::kThreads, native::SMEM_BYTES, st>>>(
      mA, mB, mSA, mSB, mC, tma_store ? 1 : 0, a.TA, a.TB, (int)a.M, (int)a.N, (int)a.K, a.out, a.status,
      a.wait_cycles);
  return cudaGetLastError();
}

cudaError_t launch_gemm_nvfp4(const GemmArgs& a, cudaStream_t st) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  CUtensorMap mA, mB, mSA, mSB, mC;
  if (!make_swizzled_payload_map(&mA, a.A, a.M, a.K, native::BM) ||
      !make_swizzled_payload_map(&mB, a.B, a.N, a.K, native::BN) ||
      !make_scale_map(&mSA, a.As, a.M, a.K, native::BM) || !make_scale_map(&mSB, a.Bs, a.N, a.K, native::BN))
    return cudaErrorNotSupported;
  const bool tma_store = !a.out_f32 && make_native_out_map(&mC, a.out, a.M, a.N);
  if (!tma_store) memset(&mC, 0, sizeof(mC));
  return a.out_f32 ? launch_native_t<true>(a, mA, mB, mSA, mSB, mC, false, st)
                   : launch_native_t<false>(a, mA, mB, mSA, mSB, mC, tma_store, st);
}

}  // namespace fp4q
