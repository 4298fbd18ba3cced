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
// Organisation: a cluster of two CTAs (one per SM) computes 256 x 256 output
// tiles with the two-SM block-scaled MMA (cta_group::2, M256 N256 K64): CTA
// rank r holds A rows 128 r .. 128 r + 127 of a tile and B rows
// 128 r .. 128 r + 127, so a stage moves 38 KB per SM instead of the 54 KB
// of one SM computing a 128 x 256 tile alone; its TMEM holds its 128 rows of
// the accumulator.  Persistent: each cluster walks tiles c, c + clusters, ...
// A tile's main loop is short at the FP4 rate (a few microseconds at the
// 8B-class sizes), so the fill and drain of a tile are hidden behind the
// next one: the epilogue warps release TMEM to the next tile's MMAs as soon
// as they have read it, and convert and store from registers.  Per CTA, 256 K elements per stage (one 128-byte swizzled row of
// packed E2M1 per operand row):
//   warp 12     TMA producer: the CTA's payload tiles of A (128 x 128 B) and
//               B (128 x 128 B), 128-byte swizzled as the MMA descriptors
//               read them, and the stage's scale codes (16 per row: the
//               CTA's 128 A rows, and all 256 B rows of the tile -- each CTA
//               loads its 128 and multicasts them to both) into a 5-stage
//               ring.
//   warps 0..3  copy the stage's scale codes into one of four TMEM slots
//               (tcgen05.st), warp q into lane quadrant q, all four the same
//               data: for each of the stage's four K64 MMAs, the 32-bit word
//               of row r (its four block scales, the first K block in the
//               low byte) goes to lane r mod 32, column base + r / 32 -- B's
//               256 rows in eight columns, A's 128 in four (the
//               scale-factor layout of the block-scaled MMA: every lane
//               quadrant sees every row) -- then signal rank 0.
//   warp 13     allocates the pair's TMEM (accumulator in columns 0..255,
//               the scale ring in 256..511); in rank 0 one lane waits until
//               both CTAs have a stage's scales in TMEM (and so its operands
//               in shared memory), issues four MMAs (M256 N256 K64) and
//               commits them to both CTAs' "empty" barriers; a tile's first
//               MMA waits until both CTAs' epilogues have read the last one.
//   warps 4..11 epilogue: TMEM -> registers (64 columns per lane at a time)
//               -> alpha -> BF16 or FP32 -> global: a BF16 result through a
//               4 KB staging box per warp and TMA stores when a tensor map
//               describes it, else 256-bit stores of each lane's row
//               segment where 32-byte aligned (both write whole L2 sectors).
// Rebiased mode (fp4q_gemm_nvfp4_rebiased): UE5M3 block scales re-expressed
// as UE4M3 codes times a power of two, per A row (fa) and for all of B (fb);
// the epilogue multiplies each row by T_A T_B fb fa[row], exact products of
// powers of two.  A device flag (skip_if) read once per pair makes the whole
// launch a no-op, so that the caller need not read it on the host.  With
// QOUT the epilogue also quantises the BF16 result row-wise for the next
// layer (RNE, blocks of 16 along N, tensor scale TC, the quantisers' own
// block-scale and conversion code): two blocks per 32-column chunk, payload
// and codes stored from registers, and max |bf16(C)| into qamax.
// Two-window mode (fp4q_gemm_nvfp4_two_windows, the TWO shape): A's UE5M3
// codes split per row into a high and a low 14-binade window of UE4M3 codes;
// 256 x 128 tiles whose two 128-column accumulators take the high- and the
// low-window MMA of each K64 step on the same operand tiles, and the
// epilogue forms alpha (high + 2^-14 low).  Geometry of both shapes: Geo.
// Every wait is bounded; a wait that runs out latches FP4Q_ERR_TIMEOUT and
// the CTA winds down once the loads and MMAs it issued have completed; both
// CTAs meet at a cluster barrier before the pair's TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "fp4q_device.cuh"
#include "fp4q_launch.h"
#include "fp4q_pipeline.cuh"
#include "fp4q_tcgen05.cuh"

namespace fp4q {
namespace native {

constexpr int PM = 256;                          // output rows of a pair's tile
constexpr int BM = 128;                          // A rows per CTA
constexpr int BK = 256;                          // K elements per stage
constexpr int ROWB = BK / 2;                     // payload bytes per row per stage (128)
constexpr int A_BYTES = BM * ROWB;               // 16384
constexpr int SA_BYTES = BM * (BK / 16);         // 2048: 16 scale codes per row
constexpr int MMAS = BK / 64;                    // four K64 MMAs per stage
constexpr int kSfWarps = 4, kEpiWarp0 = 4, kEpiWarps = 8;
constexpr int kProducerWarp = 12, kMmaWarp = 13;
constexpr int kThreads = 32 * 14;
static_assert(kEpiWarp0 % 4 == 0, "epilogue warp w drains TMEM lane quadrant w % 4");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256;                // scale ring from column 256; accumulators below

// The two shapes of the kernel.  One window (TWO = false): 256 x 256 tiles,
// one 256-column accumulator, five 38 KB stages; the scale ring holds four
// entries of one stage each (per K64 step a group of 16 columns: B's words in
// 8, A's in 4 from column 8).  Two windows (TWO = true, A's codes split in a
// high and a low window): 256 x 128 tiles, two 128-column accumulators (high
// in columns 0..127, low in 128..255), both fed by each K64 step from the same
// operand tiles, six 30 KB stages (the low-window A codes added; six rather
// than seven leave room for the result's staging boxes: 1 % faster); a K64 step
// takes two 16-column scale groups (the high MMA's -- B's words in 4, A's
// high-window words from column 8 -- among the entry's first 64 columns, the
// low MMA's the same way 64 columns on), so the ring holds two entries of one
// stage each.  (Entries of half a stage, each
// released as soon as its own MMAs completed, so that three entries' MMAs
// rather than one stage's cover the next copy into TMEM, ran 23 % slower:
// the extra barrier wait and commits sit on the one thread that issues the
// MMAs.)
template <bool TWO>
struct Geo {
  static constexpr int PN = TWO ? 128 : 256;     // output columns of a pair's tile = N of the MMA
  static constexpr int BH = PN / 2;              // B rows per CTA
  static constexpr int S = TWO ? 6 : 5;          // shared-memory ring stages
  static constexpr int ESTEPS = 4;               // K64 steps per scale-ring entry (a stage)
  static constexpr int EPS = MMAS / ESTEPS;      // entries per stage
  static constexpr uint32_t kStepCols = 16;                       // a K64 step's scale group
  static constexpr uint32_t kEntryCols = (TWO ? 2 : 1) * ESTEPS * kStepCols;   // 64, TWO: 128
  static constexpr int NENT = (int)((kTmemCols - kSfCol0) / kEntryCols);   // ring entries (4, TWO: 2)
  static constexpr bool kEntryIsStage = EPS == 1;  // released with the stage (bar_empty)
  static constexpr int B_BYTES = BH * ROWB;      // this CTA's half of B
  static constexpr int SB_BYTES = PN * (BK / 16);   // every B row of the tile
  static constexpr int OFF_A = 0, OFF_B = A_BYTES, OFF_SA = OFF_B + B_BYTES;
  static constexpr int OFF_SA2 = OFF_SA + SA_BYTES;   // A's low-window codes (TWO)
  static constexpr int OFF_SB = OFF_SA2 + (TWO ? SA_BYTES : 0);
  static constexpr int STAGE = OFF_SB + SB_BYTES;     // 38912 or 30720
  static constexpr uint32_t kLoCol = 128;             // the low accumulator (TWO)
  static constexpr uint32_t kLoSf = ESTEPS * kStepCols;   // the low MMAs' scale groups, after the high ones (TWO)
  // full, empty per stage; sf (rank 0) and sfree per entry; acc full / empty, done
  static constexpr int NBARS = 2 * S + 2 * NENT + 3;
  static constexpr int OFF_BAR = S * STAGE;
  static constexpr int OFF_TMEM = OFF_BAR + 8 * NBARS;
  static constexpr int OFF_ABORT = OFF_TMEM + 8;
  static constexpr int OFF_TAB = OFF_ABORT + 8;  // the epilogue quantisation's scale table
  // BF16 result through TMA stores: a 32-row x 64-column box per epilogue
  // warp (4 KB, 128-byte swizzle, 1 KB aligned)
  static constexpr int OUT_BOX = 32 * 128;
  static constexpr int OFF_OUT = (OFF_TAB + (int)sizeof(ScaleTab) + 1023) / 1024 * 1024;
  static constexpr int OUT_BYTES = kEpiWarps * OUT_BOX;
  static constexpr int SMEM_BYTES = OFF_OUT + OUT_BYTES + 1024;   // + 1 KB alignment slack
  // Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1), both
  // K-major, UE4M3 scales (bit 23 clear), scale-factor data IDs 0,
  // N (bits 17..22: N / 8), M = 256 for the pair (bits 24..28: M / 16); dense.
  static constexpr uint32_t kIdesc =
      (1u << 7) | (1u << 10) | ((uint32_t)(PN >> 3) << 17) | ((uint32_t)(PM >> 4) << 24);
  static_assert(STAGE % 1024 == 0 && OFF_B % 1024 == 0 && OFF_SA % 128 == 0 && OFF_SA2 % 128 == 0 &&
                    OFF_SB % 128 == 0,
                "alignment");
  static_assert(MMAS % ESTEPS == 0 && kSfCol0 + NENT * kEntryCols <= kTmemCols &&
                    (TWO ? 2 * PN : PN) <= (int)kSfCol0 && NENT >= 2 && (!kEntryIsStage || NENT < S),
                "TMEM map");
  static_assert(PN % 32 == 0 && PN / 32 <= 8, "B's scale words fill at most 8 columns per MMA");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ void mma_nvfp4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t sfa, uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accum)
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

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// bulk-group bookkeeping of this thread's TMA stores
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Epilogue helpers (lane-local: one output row, 32 consecutive columns from
// col0; columns at or past N are not written).  A lane's row segment is
// written with 256-bit stores when its address is 32-byte aligned (whole L2
// sectors: 7 % on fprop's 268 MB result against 128-bit stores, which write
// each sector in two halves), else with 128-bit or scalar stores.  (The
// one-window BF16 result goes through TMA stores instead when a tensor map
// describes it: another 9 % on fprop, 1 % on the two-window wgrad.)
__device__ __forceinline__ bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void pack_bf16x32(const uint32_t (&r)[64], int off, float alpha, uint32_t (&hh)[16]) {
#pragma unroll
  for (int jj = 0; jj < 16; ++jj)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hh[jj])
        : "f"(__fmul_rn(__uint_as_float(r[off + 2 * jj + 1]), alpha)), "f"(__fmul_rn(__uint_as_float(r[off + 2 * jj]), alpha)));
}
__device__ __forceinline__ void store_bf16x32(void* out, int row, int col0, int N, const uint32_t (&hh)[16]) {
  if (col0 >= N) return;
  uint16_t* o = static_cast<uint16_t*>(out) + (int64_t)row * N + col0;
  if (col0 + 32 <= N && aligned32(o)) {
    st_global_v8(o, hh);
    st_global_v8(o + 16, hh + 8);
  } else if (N % 8 == 0 && col0 + 32 <= N) {
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      reinterpret_cast<uint4*>(o)[jj] = make_uint4(hh[4 * jj], hh[4 * jj + 1], hh[4 * jj + 2], hh[4 * jj + 3]);
  } else {
#pragma unroll
    for (int jj = 0; jj < 32; ++jj)
      if (col0 + jj < N) o[jj] = (uint16_t)((jj & 1) ? (hh[jj >> 1] >> 16) : (hh[jj >> 1] & 0xFFFFu));
  }
}
__device__ __forceinline__ void store_f32x32(void* out, int row, int col0, int N, const uint32_t (&r)[64], int off,
                                             float alpha) {
  if (col0 >= N) return;
  float* o = static_cast<float*>(out) + (int64_t)row * N + col0;
  if (col0 + 32 <= N && aligned32(o)) {
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint32_t w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__fmul_rn(__uint_as_float(r[off + 8 * jj + k]), alpha));
      st_global_v8(o + 8 * jj, w);
    }
  } else if (N % 4 == 0 && col0 + 32 <= N) {
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
      reinterpret_cast<float4*>(o)[jj] = make_float4(__fmul_rn(__uint_as_float(r[off + 4 * jj]), alpha),
                                                     __fmul_rn(__uint_as_float(r[off + 4 * jj + 1]), alpha),
                                                     __fmul_rn(__uint_as_float(r[off + 4 * jj + 2]), alpha),
                                                     __fmul_rn(__uint_as_float(r[off + 4 * jj + 3]), alpha));
  } else {
#pragma unroll
    for (int jj = 0; jj < 32; ++jj)
      if (col0 + jj < N) o[jj] = __fmul_rn(__uint_as_float(r[off + jj]), alpha);
  }
}

// The epilogue quantisation of one 32-column chunk of a BF16 result row
// (hh: 16 words, element 2j in the low half of word j): two blocks of 16,
// each scaled and converted as the quantisers do (RNE), stored as 16 payload
// bytes and two scale codes; qmax collects max |bf16| as a 16-bit pattern.
// N % 32 == 0, so the chunk is wholly inside a row.
__device__ __forceinline__ void quantize_chunk(const uint32_t (&hh)[16], const ScaleTab& tab, const ScaleRegs& kr,
                                               int row, int col0, int N, uint8_t* qpay, uint8_t* qsc,
                                               uint32_t& qmax) {
  uint32_t pw[4], codes = 0, cl = 0, fl = 0;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t a = max(absmax16(hh + 8 * b), absmax16(hh + 8 * b + 4));
    qmax = max(qmax, a);
    const BlockScale bs = block_scale<false>(a, tab, kr);
    pw[2 * b] = quantize8<false, false>(hh + 8 * b, bs.r, nullptr, &cl, &fl);
    pw[2 * b + 1] = quantize8<false, false>(hh + 8 * b + 4, bs.r, nullptr, &cl, &fl);
    codes |= bs.code << (8 * b);
  }
  *reinterpret_cast<uint4*>(qpay + (int64_t)row * (N / 2) + col0 / 2) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
  *reinterpret_cast<uint16_t*>(qsc + (int64_t)row * (N / 16) + col0 / 16) = (uint16_t)codes;
}

// BF16 store (out nullable) and quantisation of one chunk, if it starts
// inside the row.
__device__ __forceinline__ void store_quantize_chunk(const uint32_t (&hh)[16], void* out, const ScaleTab& tab,
                                                     const ScaleRegs& kr, int row, int col0, int N, uint8_t* qpay,
                                                     uint8_t* qsc, uint32_t& qmax) {
  if (col0 >= N) return;
  if (out) store_bf16x32(out, row, col0, N, hh);
  quantize_chunk(hh, tab, kr, row, col0, N, qpay, qsc, qmax);
}

// Persistent, launched in clusters of two along x: cluster c (= blockIdx.x / 2)
// takes tiles c, c + clusters, ... of the tiles_m x tiles_n grid of 256 x PN
// tiles (row-major: consecutive clusters share A rows).  With TWO, mapSA holds
// A's high-window codes and mapSA2 its low-window codes (unused otherwise).
template <bool F32OUT, bool QOUT, bool TWO>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                      const __grid_constant__ CUtensorMap mapSA, const __grid_constant__ CUtensorMap mapSB,
                      const __grid_constant__ CUtensorMap mapSA2, const __grid_constant__ CUtensorMap mapC,
                      int tma_out,
                      const float* __restrict__ TA, const float* __restrict__ TB, int M, int N, int K,
                      void* __restrict__ out, int* status, long long budget, int skip_loads,
                      const float* __restrict__ fa, const float* __restrict__ fb, const int* skip_if,
                      const float* __restrict__ TC, uint8_t* __restrict__ qpay, uint8_t* __restrict__ qsc,
                      float* qamax, int qfmt) {
  using G = Geo<TWO>;
  constexpr int PN = G::PN, BH = G::BH, S = G::S, STAGE = G::STAGE;
  constexpr int ESTEPS = G::ESTEPS, EPS = G::EPS, NENT = G::NENT;
  constexpr int OFF_A = G::OFF_A, OFF_B = G::OFF_B, OFF_SA = G::OFF_SA, OFF_SA2 = G::OFF_SA2, OFF_SB = G::OFF_SB;
  constexpr int OFF_BAR = G::OFF_BAR, OFF_TMEM = G::OFF_TMEM, OFF_ABORT = G::OFF_ABORT, OFF_TAB = G::OFF_TAB;
  constexpr uint32_t kStepCols = G::kStepCols, kEntryCols = G::kEntryCols, kLoCol = G::kLoCol, kLoSf = G::kLoSf;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  if (skip_if && pair_read_flag(skip_if, sb + OFF_ABORT + 4)) return;   // both CTAs, before any setup
  const uint32_t bar_full = sb + OFF_BAR;            // TMA bytes of stage s landed (this CTA)
  const uint32_t bar_empty = bar_full + 8 * S;       // stage s MMAs completed
  const uint32_t bar_sf = bar_empty + 8 * S;         // entry t's scales in both CTAs' TMEM (rank 0)
  const uint32_t bar_sfree = bar_sf + 8 * NENT;      // entry t's MMAs completed (unused when an entry is a stage)
  const uint32_t bar_acc_full = bar_sfree + 8 * NENT;   // a tile's MMAs completed
  const uint32_t bar_acc_empty = bar_acc_full + 8;   // both CTAs' epilogues read TMEM (rank 0)
  const uint32_t bar_done = bar_acc_empty + 8;       // every MMA issued completed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  ScaleTab* tab = reinterpret_cast<ScaleTab*>(smem + OFF_TAB);
  if (QOUT) build_scale_tab(tab, __ldg(TC), qfmt);   // block-wide, before the roles split

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int tiles_n = (N + PN - 1) / PN;
  const int ntiles = tiles_n * ((M + PM - 1) / PM);
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int nk = K / BK;
  // this CTA's rows of tile `tile`: A from am0, B from bn0; output columns from n0
  auto tile_rows = [&](int tile, int& am0, int& bn0, int& n0) {
    const int tm = tile / tiles_n, tn = tile - tm * tiles_n;
    n0 = tn * PN;
    am0 = tm * PM + BM * (int)rank;
    bn0 = n0 + BH * (int)rank;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, 1);
    }
    for (int i = 0; i < NENT; ++i) {
      mbar_init(bar_sf + 8 * i, 2 * kSfWarps);   // the scale warps of both CTAs
      mbar_init(bar_sfree + 8 * i, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 2 * kEpiWarps);          // the epilogue warps of both CTAs
    mbar_init(bar_done, 1);
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
      int64_t g = 0, last_g = -1;   // stages issued over all tiles; the last one loaded
      bool ok = true;
      for (int tile = cid; tile < ntiles && ok; tile += ncl) {
        int am0, bn0, n0;
        tile_rows(tile, am0, bn0, n0);
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = (int)(g % S);
          if (!mbar_wait(bar_empty + 8 * s, (uint32_t)((g / S) & 1) ^ 1, abort_flag, budget)) {
            fail(abort_flag, status);
            ok = false;
            break;
          }
          if (skip_loads) continue;   // test hook: consumers' waits run out
          const uint32_t st = sb + s * STAGE;
          mbar_expect_tx(bar_full + 8 * s, STAGE);
          tma_load_2d(st + OFF_A, &mapA, kb * ROWB, am0, bar_full + 8 * s);
          tma_load_2d(st + OFF_B, &mapB, kb * ROWB, bn0, bar_full + 8 * s);
          tma_load_2d(st + OFF_SA, &mapSA, kb * (BK / 16), am0, bar_full + 8 * s);
          if (TWO) tma_load_2d(st + OFF_SA2, &mapSA2, kb * (BK / 16), am0, bar_full + 8 * s);
          // the tile's PN B rows of scale codes: this CTA loads its PN / 2 and
          // delivers them to both CTAs of the pair
          tma_load_2d_multicast(st + OFF_SB + (uint32_t)(BH * (BK / 16)) * rank, &mapSB, kb * (BK / 16), bn0,
                                bar_full + 8 * s, (uint16_t)0x3);
          last_g = g;
        }
      }
      // Drain, also after an abort: only the last load into each stage can
      // still be in flight (a stage is refilled only after its MMAs read it).
      bool drained = true;
      for (int s = 0; s < S; ++s) {
        if (last_g < s) continue;
        const int64_t gs = s + (last_g - s) / S * S;
        drained &= mbar_wait_bounded(bar_full + 8 * s, (uint32_t)((gs / S) & 1), kDrainCycles);
      }
      if (!drained) atomicOr(status, kStatusTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0) {
      if (rank == 0) {
        int64_t g = 0;
        int j = 0;   // tiles begun
        bool ok = true;
        for (int tile = cid; tile < ntiles && ok; tile += ncl, ++j) {
          // both CTAs' epilogues have copied the previous tile out of TMEM
          if (j > 0 && !mbar_wait_cluster(bar_acc_empty, (uint32_t)((j - 1) & 1), abort_flag, budget)) {
            fail(abort_flag, status);
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < nk && ok; ++kb, ++g) {
            const int s = (int)(g % S);
            const uint32_t st = sb + s * STAGE;
            const uint64_t ad = sw128_desc(st + OFF_A), bd = sw128_desc(st + OFF_B);
#pragma unroll
            for (int el = 0; el < EPS; ++el) {
              const int64_t e = g * EPS + el;   // ring entry, over all tiles
              const int t = (int)(e % NENT);
              // both CTAs' scale warps have seen the stage's bytes land and put
              // the entry's scales in TMEM
              if (!mbar_wait_cluster(bar_sf + 8 * t, (uint32_t)((e / NENT) & 1), abort_flag, budget)) {
                fail(abort_flag, status);
                ok = false;
                break;
              }
              tc_fence_after();
#pragma unroll
              for (int jj = 0; jj < ESTEPS; ++jj) {
                const int i = el * ESTEPS + jj;   // K64 step within the stage
                const uint32_t sf = tmem + kSfCol0 + kEntryCols * t + kStepCols * jj;
                const uint32_t acc = (kb | i) != 0 ? 1u : 0u;
                mma_nvfp4_pair(tmem, ad + 2 * i, bd + 2 * i, G::kIdesc, sf + 8, sf, acc);
                if (TWO)   // the low window: same operand tiles, its own scales and accumulator
                  mma_nvfp4_pair(tmem + kLoCol, ad + 2 * i, bd + 2 * i, G::kIdesc, sf + kLoSf + 8, sf + kLoSf, acc);
              }
              if (!G::kEntryIsStage) mma_commit_pair(bar_sfree + 8 * t);
            }
            if (ok) mma_commit_pair(bar_empty + 8 * s);
          }
          if (ok) mma_commit_pair(bar_acc_full);
        }
        mma_commit_pair(bar_done);
      }
      // Drain, also after an abort: every MMA issued above completes (in
      // both CTAs) before TMEM is freed and either CTA exits.  In rank 1 this
      // wait spans the whole kernel.
      if (!mbar_wait_bounded(bar_done, 0, kDrainCycles)) atomicOr(status, kStatusTimeout);
    }
  } else if (warp < kSfWarps) {
    // ------------------------------------------------ scale codes -> TMEM
    // lane r0 of warp q writes TMEM lane 32 q + r0 of ring entry t: for the
    // entry's K64 step j, column kStepCols j + c holds the word of B row
    // r0 + 32 c (c < PN / 32, the tile's PN B rows), column kStepCols j + 8 + c
    // the word of A row r0 + 32 c (c < 4, this CTA's 128 A rows); with TWO
    // these are the high-window words, and the same group kLoSf columns on
    // holds B's words and A's low-window words.  Entry t is rewritten once the
    // MMAs that last read it (NENT entries back) have completed.
    constexpr int NBW = PN / 32;   // B's words per lane and K64 step
    int64_t g = 0;
    bool ok = true;
    for (int tile = cid; tile < ntiles && ok; tile += ncl) {
      for (int kb = 0; kb < nk && ok; ++kb, ++g) {
        const int s = (int)(g % S);
        if (!mbar_wait(bar_full + 8 * s, (uint32_t)((g / S) & 1), abort_flag, budget)) {
          fail(abort_flag, status);
          ok = false;
          break;
        }
        const uint32_t st = sb + s * STAGE;
        uint4 a[4], b[NBW];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) a[jj] = lds128(st + OFF_SA + (uint32_t)(lane + 32 * jj) * 16);
#pragma unroll
        for (int jj = 0; jj < NBW; ++jj) b[jj] = lds128(st + OFF_SB + (uint32_t)(lane + 32 * jj) * 16);
#pragma unroll
        for (int el = 0; el < EPS; ++el) {
          const int64_t e = g * EPS + el, ep = e - NENT;   // ep: the entry that last used t
          const int t = (int)(e % NENT);
          if (ep >= 0) {
            const bool done = G::kEntryIsStage
                                  ? mbar_wait(bar_empty + 8 * (int)(ep % S), (uint32_t)((ep / S) & 1), abort_flag, budget)
                                  : mbar_wait(bar_sfree + 8 * t, (uint32_t)((ep / NENT) & 1), abort_flag, budget);
            if (!done) {
              fail(abort_flag, status);
              ok = false;
              break;
            }
          }
          const uint32_t col = tmem + ((uint32_t)(32 * warp) << 16) + kSfCol0 + kEntryCols * t;
#pragma unroll
          for (int jj = 0; jj < ESTEPS; ++jj) {
            const int i = el * ESTEPS + jj;
            uint32_t v[16];
#pragma unroll
            for (int c = 0; c < 8; ++c) v[c] = c < NBW ? word_of(b[c], i) : 0u;
#pragma unroll
            for (int c = 0; c < 4; ++c) v[8 + c] = word_of(a[c], i);
#pragma unroll
            for (int c = 12; c < 16; ++c) v[c] = 0u;
            tmem_st16(col + kStepCols * jj, v);
          }
          if (TWO) {   // the low-window groups, loaded once the high ones are written
            uint4 a2[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) a2[c] = lds128(st + OFF_SA2 + (uint32_t)(lane + 32 * c) * 16);
#pragma unroll
            for (int jj = 0; jj < ESTEPS; ++jj) {
              const int i = el * ESTEPS + jj;
              uint32_t v[16];
#pragma unroll
              for (int c = 0; c < 8; ++c) v[c] = c < NBW ? word_of(b[c], i) : 0u;
#pragma unroll
              for (int c = 0; c < 4; ++c) v[8 + c] = word_of(a2[c], i);
#pragma unroll
              for (int c = 12; c < 16; ++c) v[c] = 0u;
              tmem_st16(col + kStepCols * jj + kLoSf, v);
            }
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_rank0(bar_sf + 8 * t);
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 4..11)
    // warp w takes TMEM lanes 32 (w % 4) .. +31 (the CTA's rows), columns
    // (PN / 2) h .. (PN / 2) (h + 1) - 1 (h = (w - 4) / 4), 64 at a time; TMEM
    // is released to the next tile's MMAs as soon as the last 64 are in
    // registers.
    const int q = warp & 3, h = (warp - kEpiWarp0) >> 2;
    float alpha0 = __fmul_rn(__ldg(TA), __ldg(TB));
    if (fb) alpha0 = __fmul_rn(alpha0, __ldg(fb));   // a power of two: exact
    uint32_t qmax = 0;                                // max |bf16(C)| of this lane's chunks (a pattern)
    ScaleRegs kr{};
    if (QOUT) kr = scale_regs(*tab);
    int j = 0;
    for (int tile = cid; tile < ntiles; tile += ncl, ++j) {
      if (!mbar_wait(bar_acc_full, (uint32_t)(j & 1), abort_flag, budget)) {
        fail(abort_flag, status);
        break;
      }
      tc_fence_after();
      int am0, bn0, n0;
      tile_rows(tile, am0, bn0, n0);
      const int row = am0 + 32 * q + lane;
      const int cbase = n0 + (PN / 2) * h;
      const bool live = row < M && cbase < N;
      const float alpha = (fa && row < M) ? __fmul_rn(alpha0, __ldg(fa + row)) : alpha0;
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((PN / 2) * h);
      if (TWO && !F32OUT) {
        // 32 columns of each accumulator at a time: C = alpha (high + 2^-14
        // low) -- the low window's factor is the high one's times 2^-14, an
        // exact scaling, so the sum is rounded once, then alpha as below.
        // The first chunk is packed to BF16 before the second is loaded, TMEM
        // released, and only then are both stored: the next tile's MMAs wait
        // for the loads alone.
        uint32_t h0[16], h1[16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[64];
          tmem_ld32_nowait(taddr + 32 * c, r);
          tmem_ld32_nowait(taddr + kLoCol + 32 * c, r + 32);
          tmem_ld_wait(r, 64);
          if (c == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_rank0(bar_acc_empty);
          }
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            r[jj] = __float_as_uint(__fmaf_rn(__uint_as_float(r[32 + jj]), 0x1p-14f, __uint_as_float(r[jj])));
          if (c == 0)
            pack_bf16x32(r, 0, alpha, h0);
          else
            pack_bf16x32(r, 0, alpha, h1);
        }
        if (tma_out) {
          const uint32_t stg = sb + G::OFF_OUT + (uint32_t)(warp - kEpiWarp0) * G::OUT_BOX;
          const int y0 = am0 + 32 * q;
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sts128(stg + (uint32_t)lane * 128 + ((uint32_t)(i ^ (lane & 7)) << 4), h0[4 * i], h0[4 * i + 1],
                   h0[4 * i + 2], h0[4 * i + 3]);
            sts128(stg + (uint32_t)lane * 128 + ((uint32_t)((4 + i) ^ (lane & 7)) << 4), h1[4 * i], h1[4 * i + 1],
                   h1[4 * i + 2], h1[4 * i + 3]);
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0 && cbase < N && y0 < M) {
            tma_store_2d(&mapC, stg, cbase, y0);
            bulk_commit();
          }
        } else if (live) {
          store_bf16x32(out, row, cbase, N, h0);
          store_bf16x32(out, row, cbase + 32, N, h1);
        }
      } else if (TWO) {
        // the same with a binary32 result, stored chunk by chunk
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[64];
          tmem_ld32_nowait(taddr + 32 * c, r);
          tmem_ld32_nowait(taddr + kLoCol + 32 * c, r + 32);
          tmem_ld_wait(r, 64);
          if (c == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_rank0(bar_acc_empty);
          }
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            r[jj] = __float_as_uint(__fmaf_rn(__uint_as_float(r[32 + jj]), 0x1p-14f, __uint_as_float(r[jj])));
          if (live) store_f32x32(out, row, cbase + 32 * c, N, r, 0, alpha);
        }
      } else if (F32OUT) {
        // 64 columns at a time; TMEM released (the next tile's MMAs may
        // overwrite the accumulator) once the second load is complete
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[64];
          tmem_ld32_nowait(taddr + 64 * half, r);
          tmem_ld32_nowait(taddr + 64 * half + 32, r + 32);
          tmem_ld_wait(r, 64);
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_rank0(bar_acc_empty);
          }
          if (live) store_f32x32(out, row, cbase + 64 * half, N, r, 0, alpha);
          if (live) store_f32x32(out, row, cbase + 64 * half + 32, N, r, 32, alpha);
        }
      } else if (!QOUT && tma_out) {
        // BF16 through TMA stores: each 64-column half is packed into the
        // warp's staging box (row = lane, 16-byte chunk c at c ^ (lane % 8):
        // the 128-byte swizzle of the output map, no bank conflicts) once the
        // box's previous store has read it, and lane 0 stores the 32 x 64 box;
        // TMEM is released once the second half is loaded.  Boxes starting
        // outside the result are skipped; the store clips a ragged edge.
        const uint32_t stg = sb + G::OFF_OUT + (uint32_t)(warp - kEpiWarp0) * G::OUT_BOX;
        const int y0 = am0 + 32 * q;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[64];
          tmem_ld32_nowait(taddr + 64 * half, r);
          tmem_ld32_nowait(taddr + 64 * half + 32, r + 32);
          tmem_ld_wait(r, 64);
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_rank0(bar_acc_empty);
          }
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t hh[16];
            pack_bf16x32(r, 32 * c, alpha, hh);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              sts128(stg + (uint32_t)lane * 128 + ((uint32_t)((4 * c + i) ^ (lane & 7)) << 4), hh[4 * i],
                     hh[4 * i + 1], hh[4 * i + 2], hh[4 * i + 3]);
          }
          fence_proxy_async();
          __syncwarp();
          const int x0 = cbase + 64 * half;
          if (lane == 0 && x0 < N && y0 < M) {
            tma_store_2d(&mapC, stg, x0, y0);
            bulk_commit();
          }
        }
      } else if (!QOUT) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[64];
          tmem_ld32_nowait(taddr + 64 * half, r);
          tmem_ld32_nowait(taddr + 64 * half + 32, r + 32);
          tmem_ld_wait(r, 64);
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_rank0(bar_acc_empty);
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t hh[16];
            pack_bf16x32(r, 32 * c, alpha, hh);
            if (live) store_bf16x32(out, row, cbase + 64 * half + 32 * c, N, hh);
          }
        }
      } else {
        // 64 columns at a time: loaded, packed to BF16 and quantised (the
        // payload and codes stored from registers); the BF16 result through
        // the warp's staging box and a TMA store as above when tma_out, else
        // stored with its chunk; TMEM released once the second load is
        // complete.  (Holding all 128 packed columns until the release, so
        // that the first 64's work follows it, needs more than the 128
        // registers a thread has here.)
        const uint32_t stg = sb + G::OFF_OUT + (uint32_t)(warp - kEpiWarp0) * G::OUT_BOX;
        const int y0 = am0 + 32 * q;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[64];
          tmem_ld32_nowait(taddr + 64 * half, r);
          tmem_ld32_nowait(taddr + 64 * half + 32, r + 32);
          tmem_ld_wait(r, 64);
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_rank0(bar_acc_empty);
          }
          if (tma_out) {
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t hh[16];
            pack_bf16x32(r, 32 * c, alpha, hh);
            if (tma_out) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                sts128(stg + (uint32_t)lane * 128 + ((uint32_t)((4 * c + i) ^ (lane & 7)) << 4), hh[4 * i],
                       hh[4 * i + 1], hh[4 * i + 2], hh[4 * i + 3]);
            }
            if (live)
              store_quantize_chunk(hh, tma_out ? nullptr : out, *tab, kr, row, cbase + 64 * half + 32 * c, N, qpay,
                                   qsc, qmax);
          }
          if (tma_out) {
            fence_proxy_async();
            __syncwarp();
            const int x0 = cbase + 64 * half;
            if (lane == 0 && x0 < N && y0 < M) {
              tma_store_2d(&mapC, stg, x0, y0);
              bulk_commit();
            }
          }
        }
      }
    }
    if (tma_out && lane == 0) bulk_wait0();   // this warp's TMA stores complete
    if (QOUT) {
      // max |bf16(C)| (a 16-bit pattern; inf/NaN compare above every finite)
      qmax = __reduce_max_sync(0xFFFFFFFFu, qmax);
      if (lane == 0) {
        if (qmax >= 0x7F80u) atomicOr(status, kStatusNonFinite);
        if (qamax && qmax) atomicMax(reinterpret_cast<unsigned int*>(qamax), qmax << 16);
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

// 2-D BF16 tensor map over the [M, N] result, box (64 columns, 32 rows),
// 128-byte swizzle; needs a row stride that is a multiple of 16 bytes.
static bool make_out_map(CUtensorMap* map, void* base, int64_t M, int64_t N) {
  auto fn = get_encode_fn();
  if (!fn || N % 8 != 0 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)(N * 2)};
  const cuuint32_t box[2] = {64u, 32u};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool F32OUT, bool QOUT, bool TWO>
static cudaError_t launch_native_t(const GemmArgs& a, const CUtensorMap& mA, const CUtensorMap& mB,
                                   const CUtensorMap& mSA, const CUtensorMap& mSB, const CUtensorMap& mSA2,
                                   cudaStream_t st) {
  using G = native::Geo<TWO>;
  auto kern = native::gemm_nvfp4_kernel<F32OUT, QOUT, TWO>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(native::kThreads);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = st;
  // one cluster per SM pair that can hold one (asked once per device and
  // output type; the tiles are then walked by the resident clusters)
  static int clusters[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (clusters[dev] == 0) {
    cfg.gridDim = dim3(2);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorNotSupported;
    clusters[dev] = n;
  }
  const int64_t ntiles = ((a.N + G::PN - 1) / G::PN) * ((a.M + native::PM - 1) / native::PM);
  const int ncl = (int)(ntiles < clusters[dev] ? ntiles : clusters[dev]);
  cfg.gridDim = dim3(2u * (unsigned)ncl);
  // the BF16 result through TMA stores when a map describes it
  CUtensorMap mC;
  const bool tma_out = !F32OUT && a.out != nullptr && make_out_map(&mC, a.out, a.M, a.N);
  if (!tma_out) memset(&mC, 0, sizeof(mC));
  e = cudaLaunchKernelEx(&cfg, kern, mA, mB, mSA, mSB, mSA2, mC, tma_out ? 1 : 0, a.TA, a.TB, (int)a.M, (int)a.N, (int)a.K, a.out, a.status,
                         a.wait_cycles, a.skip_loads ? 1 : 0, a.fa, a.fb, a.skip_if, a.TC, a.qpay, a.qsc, a.qamax,
                         a.fmt_out);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm_nvfp4(const GemmArgs& a, cudaStream_t st) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  const bool two = a.As_lo != nullptr;
  const uint32_t bh = two ? native::Geo<true>::BH : native::Geo<false>::BH;
  CUtensorMap mA, mB, mSA, mSB, mSA2;
  if (!make_swizzled_payload_map(&mA, a.A, a.M, a.K, native::BM) ||
      !make_swizzled_payload_map(&mB, a.B, a.N, a.K, bh) || !make_scale_map(&mSA, a.As, a.M, a.K, native::BM) ||
      !make_scale_map(&mSB, a.Bs, a.N, a.K, bh) ||
      !make_scale_map(&mSA2, two ? a.As_lo : a.As, a.M, a.K, native::BM))
    return cudaErrorNotSupported;
  if (two)   // A's codes in two windows: BF16 or binary32 result, no epilogue quantisation
    return a.out_f32 ? launch_native_t<true, false, true>(a, mA, mB, mSA, mSB, mSA2, st)
                     : launch_native_t<false, false, true>(a, mA, mB, mSA, mSB, mSA2, st);
  if (a.qpay)   // BF16 result (nullable) + its quantisation
    return launch_native_t<false, true, false>(a, mA, mB, mSA, mSB, mSA2, st);
  return a.out_f32 ? launch_native_t<true, false, false>(a, mA, mB, mSA, mSB, mSA2, st)
                   : launch_native_t<false, false, false>(a, mA, mB, mSA, mSB, mSA2, st);
}

}  // namespace fp4q
