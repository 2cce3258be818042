// gemm.cu -- block-scaled 4-bit GEMM D = alpha_g * A B^T on GB300 tcgen05
// tensor cores (sm_103a), for the three training GEMMs of a linear layer
// (HTX article on arXiv 2605.09825, "Experimento de diagnostico": Fprop
// Y = X W^T, Dgrad dX = dY W, Wgrad dW = dY^T X, every operand stored K-major
// by the quantizer so that each is A B^T).
//
//   E2M1 + MX (E8M0, block 32)   -> tcgen05.mma kind::mxf4, scale_vec::2X
//   E2M1 + NV (E4M3, block 16)   -> kind::mxf4nvf4, scale_vec::4X, alpha_g = S_t(A) S_t(B)
//   E1M2 + MX                    -> kind::mxf8f6f4 on the E4M3 byte copies
//                                   (every E1M2 level k/4 is exact in E4M3)
//
// Structure.  Persistent clusters of two CTAs on two SMs (a cta_group::2
// pair) own 256 x 256 output tiles; CTA r of a pair holds accumulator rows
// 128r..128r+127 of each tile in its TMEM, loads those rows of A and rows
// 128r..128r+127 of B, and the pair's MMAs, issued by rank 0 (the leader),
// read both CTAs' shared memory.  Each SM so pulls 32 KB of operands per
// 128-byte K-span (256 FP4 elements of every row) out of L2 for 128 x 256 x
// 256 of MMA work, which L2 sustains; a lone CTA on the same tile width would
// need 48 KB.  A stage holds two K-spans (kKT) for kind::mxf4 and
// mxf8f6f4: eight MMAs per stage barrier, because every stage boundary is a
// pipe bubble.  Roles (per CTA):
//   warp 0      producer: A rows and this CTA's half of B by
//               cp.async.bulk.tensor (.cta_group::2, 128-byte swizzled
//               K-major rows, one box per operand and K-span) into a ring of
//               kStages slots, the bytes completing on the leader's full
//               barrier of the slot (issuing TMA instructions is not free, so
//               the scale chunks have a loader of their own).
//   warp 1      owns the TMEM allocation (cta_group::2); on the leader one
//               lane waits for a stage (one barrier: both CTAs' operands and
//               both CTAs' scale writers), issues its MMAs back to back and
//               frees the stage with one tcgen05.commit (multicast to both
//               CTAs).  The tensor pipe queues only about one MMA ahead of
//               the lane, so the lane does nothing else between stages.
//   warps 6-9   scale writers, one per TMEM lane quarter.  The last warp
//               loads a stage's compact 512-byte scale chunks into the slot
//               beside its operands (cp.async.bulk, completing on a barrier of
//               this CTA); every writer copies its rows of the chunks into the
//               stage's TMEM scale slot with tcgen05.st and arrives on the
//               stage's barrier in the leader.
//   epilogue    (warps 2-5: columns 0-127, 10-13: columns 128-255) TMEM ->
//               registers (tcgen05.ld, 64 columns a load in the plain
//               kernels), alpha, fp32 / bf16, the accumulator is released to
//               the next tile's MMAs as soon as the last load has landed (the
//               one accumulator is single-buffered: the next tile's MMAs wait
//               for it), then the stores by TMA: through 32-row x 32-byte
//               boxes staged in 1 KB per warp in the plain kernels; through a
//               128-byte swizzled 32 x 128 slice per warp in the kernels that
//               quantize their output (TMA store, then the row-wise
//               quantization of the slice).
// Signals between the two CTAs are relaxed cluster-scope mbarrier arrivals:
// what they announce is already complete when they are sent (TMEM writes
// waited for with tcgen05.wait::st, TMEM reads with tcgen05.wait::ld), and a
// release arrival would stall the sending warp for ~1000 cycles each time.
//
// Scale factors in TMEM.  Sub-partition q of the tensor core (accumulator
// rows 32q..32q+31) reads its scales from TMEM lane quarter q: for A, row
// 32q+i at lane 32q+i, column sfa + q; for B (N = 256), row n at lane
// 32q + (n % 32), column sfb + n / 32, in every quarter.  Row i of a compact
// chunk (16 bytes) holds rows i, 32+i, 64+i, 96+i of its 128-row group, one
// 32-bit cell each, so lane i of every quarter stores row i of two chunks as
// 8 consecutive columns: for B the two row groups of one K chunk (columns
// sfb + 0..7), for A two consecutive K chunks (chunk c at sfa + 4c + 0..3, of
// which quarter q reads cell q).
//
// Grouped launches (fp4q_gemm_group) run the same kernel over the tiles of
// several GEMMs of one recipe, each pair walking its own host-made tile list
// (longest tiles first, each to the least-loaded pair), so that GEMMs with
// different K keep every SM busy to the end of one launch.
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer); on expiry the
// CTA raises FP4Q_DEV_TIMEOUT, stops issuing work, waits (bounded) for its
// own tensor-core work to drain, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <type_traits>

#include "../../include/fp4q.h"
#include "fp4q_dev.cuh"
#include "fp4q_internal.h"
#include "quant_core.cuh"

namespace fp4q {
namespace {

enum { KIND_MXF4 = 0, KIND_NVF4 = 1, KIND_F8 = 2 };

constexpr int BM = 128;              // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;              // tile columns (MMA N)
constexpr int TM = 256;              // tile rows (the pair's two CTAs)
constexpr int KROW = 128;            // bytes of one operand row per K-tile (one 128B swizzle span)
constexpr int A_BYTES = BM * KROW;   // 16 KB: this CTA's rows of A
constexpr int B_BYTES = 128 * KROW;  // 16 KB: this CTA's half of B
constexpr int OP_STAGE = A_BYTES + B_BYTES;
static_assert(A_BYTES == B_BYTES, "one descriptor step per K-span for both operands");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;      // accumulator columns [0, 256); scale slots after it
constexpr int kSmemMax = 232448;     // dynamic shared memory per CTA
constexpr int kBarBytes = 512;       // barriers, TMEM address, abort flag

#ifndef FP4Q_GEMM_KT
#define FP4Q_GEMM_KT 2
#endif

template <int KIND, bool FUSED = false>
struct KindK {
  // K-spans per stage: a span is one 128-byte (128B-swizzle) piece of every
  // operand row.  Two spans (eight MMAs per stage barrier) halve the stage
  // boundaries, where the tensor pipe idles; NVF4's scale columns and the
  // fused kernels' shared-memory staging leave room for one only.
  static constexpr int kKT = (KIND == KIND_NVF4 || FUSED) ? 1 : FP4Q_GEMM_KT;
  // chunks = 512-byte groups of 4 consecutive scale bytes of one 128-row group
  static constexpr int kChunks = kKT * (KIND == KIND_MXF4 ? 2 : (KIND == KIND_NVF4 ? 4 : 1));   // per stage
  static constexpr int kElemsPerTile = kKT * (KIND == KIND_F8 ? 128 : 256);                     // K per stage
  static constexpr int kMmaK = KIND == KIND_F8 ? 32 : 64;
  static constexpr int kMmas = kElemsPerTile / kMmaK;                                          // per stage
  static constexpr int kBlock = KIND == KIND_NVF4 ? 16 : 32;
  // a stage's operands: kKT spans of A (A_BYTES each), then kKT spans of B
  static constexpr int kOpStage = kKT * OP_STAGE;
  // one stage's compact chunks: A (kChunks), B row group 0 (kChunks), B row
  // group 1 (kChunks), loaded with the stage's operands into its slot
  static constexpr int kSfBytes = 3 * kChunks * 512;
  static constexpr int kSlot = kOpStage + (kSfBytes + 1023) / 1024 * 1024;
  // TMEM scale columns of a stage: A 4 per chunk, B 8 per chunk, rounded up
  // to the stores that write them (x16, x32 or x32 + x16)
  static constexpr int kSfColsA = 4 * kChunks;
  static constexpr int kSfColsB = 8 * kChunks;
  static constexpr int kSfCols = (kSfColsA + kSfColsB + 15) / 16 * 16;
  static_assert(kSfCols == 16 || kSfCols == 32 || kSfCols == 48, "scale slot stores");
  // every stage has its TMEM scale slot beside the accumulator
  static constexpr int kStagesTmem = (int)(TMEM_COLS - 256) / kSfCols;
  // threads: producer, MMA, scale-writer warps, the epilogue warps (8, two
  // per TMEM lane quarter, each with half of the tile's columns) and the
  // scale-chunk loader (the last warp)
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = 32 * (7 + kEpiWarps);
  static constexpr int kChunkWarp = 6 + kEpiWarps;
  static constexpr int kEpiCols = 256 / (kEpiWarps / 4);   // accumulator columns per epilogue warp
  // shared-memory staging of an epilogue warp: one 32-row x 32-byte store box
  // (plain kernels), or the warp's whole 32 x 128 bf16 slice of the tile
  // (fused output quantization)
  static constexpr int kBoxBytes = FUSED ? 128 : 32;
  static constexpr int kStgWarp = FUSED ? 32 * 2 * kEpiCols : 32 * kBoxBytes;
  static constexpr int kFixed = kEpiWarps * kStgWarp + kBarBytes + 1024;
  static constexpr int kStagesFit = (kSmemMax - kFixed) / kSlot;
  static constexpr int kStagesCap = kStagesFit > kStagesTmem ? kStagesTmem : kStagesFit;
  static constexpr int kStages = kStagesCap > 8 ? 8 : kStagesCap;
  static constexpr int kStgOff = kStages * kSlot;
  static constexpr int kBarOff = kStgOff + kEpiWarps * kStgWarp;
  static constexpr int kSmem = kBarOff + kBarBytes + 1024;   // + alignment slack
  static_assert(kStages >= 3, "pipeline depth");
  static_assert(kSmem <= kSmemMax, "shared memory");
  static_assert(kSfColsA + kSfColsB <= kSfCols, "scale columns");
  static_assert(ACC_COL + BN + kStages * kSfCols <= TMEM_COLS, "tensor memory");
  static_assert((3 * kStages + 3) * 8 + 24 <= kBarBytes, "barrier area");
  static_assert(kSlot % 1024 == 0, "slots stay aligned for the 128-byte swizzle");
};

struct GemmParams {
  const uint8_t* sfa;     // MMA scale layout of A (M x K/b)
  const uint8_t* sfb;     // MMA scale layout of B (N x K/b)
  const float* ts_a;      // NV tensor scales (or null)
  const float* ts_b;
  uint32_t* status;
  int32_t want_bf16, want_f32;
  int32_t M, N, K;
  // fused output quantization (the kernels with QG >= 0): the row-wise copy of
  // bf16(D) as fp4q_rht_quantize would make it from the stored bf16 D
  uint8_t* q_codes;       // M x N/2
  uint8_t* q_scales;      // M x N/32 E8M0 bytes, plain or MMA layout
  uint8_t* q_e4m3;        // optional M x N E4M3 bytes
  uint64_t q_seed;        // stochastic rounding
  uint32_t q_keys[20];    // its Philox round keys
  int32_t q_nh, q_sf_mma;
  uint32_t q_sgn[32];     // sign words of a 32-element chunk (bit 31 = negate)
};

// Several GEMMs of one kind in one persistent launch (the plain kernels
// only): each pair walks its own list of global tile ids, made on the host so
// that the pairs' summed tile costs are balanced (tiles of a long-K GEMM cost
// more).  Passed by value as one kernel parameter.
constexpr int kGroupMax = 4;          // GEMMs per launch
constexpr int kGroupMaxUnits = 256;   // pairs
constexpr int kGroupMaxTiles = 8192;  // 256 x 256 tiles of all the GEMMs together
struct GroupArgs {
  CUtensorMap a[kGroupMax], b[kGroupMax], dh[kGroupMax], df[kGroupMax];
  const uint8_t* sfa[kGroupMax];
  const uint8_t* sfb[kGroupMax];
  const float* ts_a[kGroupMax];
  const float* ts_b[kGroupMax];
  int32_t want_bf16[kGroupMax], want_f32[kGroupMax];
  int32_t M[kGroupMax], N[kGroupMax], K[kGroupMax];
  int32_t tile0[kGroupMax + 1];       // first global tile id of each GEMM; tile0[np] = all tiles
  int32_t np;
  uint16_t unit_begin[kGroupMaxUnits + 1];   // pair u walks order[unit_begin[u] .. unit_begin[u + 1])
  uint16_t order[kGroupMaxTiles];
};
struct NoGroupArgs {
  int32_t unused;
};
template <bool G>
using GroupArg = std::conditional_t<G, GroupArgs, NoGroupArgs>;

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false after ~2 s without completion, or when another role
// of the CTA already gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > 2000000000ull) return false;
    }
  }
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, int32_t x, int32_t y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(tm), "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start >> 4 in bits 0-13, LBO >> 4
// in 16-29, SBO >> 4 in 32-45, version 1 in 46-47, layout type in 61-63.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
// K-major operand rows of 128 bytes, 128B swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t op_desc(uint32_t saddr) { return sdesc(saddr, 16, 1024, 2); }

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// This warp's TMEM lane quarter, 32 (16) consecutive 32-bit columns from taddr.
// 64 consecutive fp32 accumulator columns of this thread's TMEM lane, one
// load and one wait.  `dep` (the packed bf16 words of the previous 64
// columns, unused by the instruction) orders the load after their conversion,
// so that no more than one load's registers are live at a time.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64], const uint32_t* dep) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(dep[0]), "r"(dep[1]), "r"(dep[2]), "r"(dep[3]), "r"(dep[4]), "r"(dep[5]), "r"(dep[6]), "r"(dep[7]), "r"(dep[8]), "r"(dep[9]), "r"(dep[10]), "r"(dep[11]), "r"(dep[12]), "r"(dep[13]), "r"(dep[14]), "r"(dep[15]), "r"(dep[16]), "r"(dep[17]), "r"(dep[18]), "r"(dep[19]), "r"(dep[20]), "r"(dep[21]), "r"(dep[22]), "r"(dep[23]), "r"(dep[24]), "r"(dep[25]), "r"(dep[26]), "r"(dep[27]), "r"(dep[28]), "r"(dep[29]), "r"(dep[30]), "r"(dep[31]));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
        "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
        "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};"
      ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}
__device__ __forceinline__ void put4(uint32_t* w, uint4 v) {
  w[0] = v.x;
  w[1] = v.y;
  w[2] = v.z;
  w[3] = v.w;
}
// 16-byte row i of a compact chunk (rows 0..31 of the 512-byte chunk).
__device__ __forceinline__ uint4 chunk_row(uint32_t chunk, int i) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(chunk + 16u * (uint32_t)i));
  return v;
}
__device__ __forceinline__ void st_shared16(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Instruction descriptor of the block-scaled kinds: B scale id in bits 4-5,
// A/B element types in 7-9 / 10-12, K-major A and B, N >> 3 in 17-22, scale
// type in 23 (1 = E8M0, 0 = E4M3), M >> 4 in 24-28, A scale id in 29-30.
// The pair's MMAs have M = 256.
template <int KIND>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id) {
  constexpr uint32_t ty = KIND == KIND_F8 ? 0u : 1u;   // E4M3 (f8f6f4) or E2M1 (mxf4 kinds)
  constexpr uint32_t sfmt = KIND == KIND_NVF4 ? 0u : 1u;
  return (sf_id << 4) | (ty << 7) | (ty << 10) | ((uint32_t)(BN >> 3) << 17) | (sfmt << 23) |
         ((uint32_t)(TM >> 4) << 24) | (sf_id << 29);
}

// ------------------------------------------------------------ cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of `saddr` in the CTA of cluster rank `rank`
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrivals on a barrier of either CTA of the pair (a shared::cluster
// address).  Relaxed: the data the arrival announces is complete already.
__device__ __forceinline__ void cluster_expect_tx(uint32_t cluster_bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cluster_arrive(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// TMA load into this CTA's shared memory that signals the pair leader's mbarrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}
// Commit of the pair's tensor-core work, arriving on the barrier at this
// offset in both CTAs (an mbarrier arrival, not a data transfer).
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
template <int KIND>
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t acc) {
  if constexpr (KIND == KIND_MXF4) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p; }"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
  } else if constexpr (KIND == KIND_NVF4) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p; }"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
  } else {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p; }"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
  }
}
// ------------------------------------------------------------ the kernel
// Persistent clusters of two CTAs: pair c owns the 256 x 256 tiles c,
// c + G/2, ... (G = gridDim.x), tile id -> (m block = id / n_blocks,
// n block = id % n_blocks); or, for GROUP, the tiles of its list in `ga`
// (p then only supplies the status word).  QG >= 0: the kernel quantizes
// its bf16 output with grid QG and rounding QR instead of storing it plain.
template <int KIND, int QG = -1, int QR = FP4Q_RTNE, bool GROUP = false>
__global__ void __launch_bounds__(KindK<KIND, (QG >= 0)>::kThreads, 1)
    bs_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmDh, const __grid_constant__ CUtensorMap tmDf,
                   const GemmParams p, const __grid_constant__ GroupArg<GROUP> ga) {
  static_assert(!GROUP || QG < 0, "grouped launches use the plain kernel");
  constexpr bool FUSED = QG >= 0;
  using KK = KindK<KIND, FUSED>;
  constexpr int S = KK::kStages;
  constexpr int SLOT = KK::kSlot;
  constexpr uint32_t SF_COLS = KK::kSfCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t stg_base = sbase + KK::kStgOff;    // epilogue staging
  // S (leader): a stage's operands (both CTAs) and scales (both CTAs' writers) are in place
  const uint32_t bar_full = sbase + KK::kBarOff;
  const uint32_t bar_empty = bar_full + 8 * S;      // S: the stage's MMAs finished (operand and scale slots free)
  const uint32_t bar_sfd = bar_empty + 8 * S;       // S: this CTA's scale chunks of a stage landed
  const uint32_t bar_acc_full = bar_sfd + 8 * S;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  const uint32_t bar_drain = bar_acc_empty + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bar_drain + 8 - sbase));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + (bar_drain + 16 - sbase));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;                   // issues MMAs
  const int unit = (int)(blockIdx.x >> 1);         // pair index
  const int n_units = (int)(gridDim.x >> 1);
  const int n_blocks = (p.N + BN - 1) / BN;
  const int n_tiles = ((p.M + TM - 1) / TM) * n_blocks;

  // The tiles this pair walks, by work index w in [w_begin, w_end) step
  // w_step, and what a tile needs: its GEMM (gi), this CTA's corner, shape
  // and K-tile count.
  struct TileCtx {
    int gi, m0, n0, M, N, K, num_kt, nq;
  };
  int w_begin = unit, w_end = n_tiles, w_step = n_units;
  if constexpr (GROUP) {
    w_begin = ga.unit_begin[unit];
    w_end = ga.unit_begin[unit + 1];
    w_step = 1;
  }
  auto tile_ctx = [&](int w) -> TileCtx {
    TileCtx t;
    int tile = w, nb = n_blocks;
    if constexpr (GROUP) {
      const int g = ga.order[w];
      int gi = 0;
#pragma unroll
      for (int q = 1; q < kGroupMax; ++q) gi += (q < ga.np && g >= ga.tile0[q]) ? 1 : 0;
      t.gi = gi;
      t.M = ga.M[gi];
      t.N = ga.N[gi];
      t.K = ga.K[gi];
      tile = g - ga.tile0[gi];
      nb = (t.N + BN - 1) / BN;
    } else {
      t.gi = 0;
      t.M = p.M;
      t.N = p.N;
      t.K = p.K;
    }
    t.m0 = (tile / nb) * TM + BM * (int)rank;
    t.n0 = (tile % nb) * BN;
    t.num_kt = (t.K + KK::kElemsPerTile - 1) / KK::kElemsPerTile;
    t.nq = t.K / KK::kBlock / 4;   // scale chunks per 128-row group
    return t;
  };
  auto map_a = [&](int gi) -> const CUtensorMap* {
    if constexpr (GROUP) return &ga.a[gi];
    else return &tmA;
  };
  auto map_b = [&](int gi) -> const CUtensorMap* {
    if constexpr (GROUP) return &ga.b[gi];
    else return &tmB;
  };
  auto map_dh = [&](int gi) -> const CUtensorMap* {
    if constexpr (GROUP) return &ga.dh[gi];
    else return &tmDh;
  };
  auto map_df = [&](int gi) -> const CUtensorMap* {
    if constexpr (GROUP) return &ga.df[gi];
    else return &tmDf;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full + 8 * s, 10);     // both producers' expect_tx and the 8 scale-writer warps
      mbar_init(bar_empty + 8 * s, 1);     // the leader's commit
      mbar_init(bar_sfd + 8 * s, 1);       // this CTA's chunk loader
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 2 * KK::kEpiWarps);   // one arrival per epilogue warp of both CTAs
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the operand maps are kernel parameters: fetch them before the wait below
    if constexpr (GROUP) {
      for (int q = 0; q < ga.np; ++q) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&ga.a[q]) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&ga.b[q]) : "memory");
      }
    } else {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  // Launched as a programmatic dependent of the stream's previous kernel: the
  // setup above touched only this CTA's shared and tensor memory; wait for
  // that grid to finish (its writes visible) before any global memory
  // access, then let the next kernel's launch begin.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  // barriers the leader owns, as seen from this CTA
  const uint32_t lead_full = mapa(bar_full, 0);
  const uint32_t lead_acc_empty = mapa(bar_acc_empty, 0);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- operand producer
      uint32_t it = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; w += w_step) {
        const TileCtx t = tile_ctx(w);
        const CUtensorMap* mA = map_a(t.gi);
        const CUtensorMap* mB = map_b(t.gi);
        for (int kt = 0; kt < t.num_kt; ++kt, ++it) {
          const int s = (int)(it % S);
          if (!mbar_wait(bar_empty + 8 * s, ((it / S) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + (uint32_t)s * SLOT;
          const uint32_t fb = lead_full + 8 * s;
          cluster_expect_tx(fb, KK::kOpStage);
          // rows past M or N (a 128-row tail) and spans past K are zero-filled and still counted
#pragma unroll
          for (int j = 0; j < KK::kKT; ++j) {
            const int x = (kt * KK::kKT + j) * KROW;
            tma_load_2d_pair(st + j * A_BYTES, mA, x, t.m0, fb);
            tma_load_2d_pair(st + KK::kKT * A_BYTES + j * B_BYTES, mB, x, t.n0 + 128 * (int)rank, fb);
          }
        }
      }
      // The leader's commits arrive on this CTA's empty barriers: wait for the
      // last use of every slot, so that none lands after exit.
      for (int i = 0; i < S && ok; ++i, ++it) {
        const int s = (int)(it % S);
        ok = mbar_wait(bar_empty + 8 * s, ((it / S) & 1u) ^ 1u, abort_flag);
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, FP4Q_DEV_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issue (lane 0 of the leader)
    // Per stage one wait (operands and scales in place), the MMAs back to
    // back and one commit: the tensor pipe queues about one MMA ahead, so
    // any further work here between stages leaves it idle.
    if (lane == 0 && leader) {
      uint32_t tl = 0, it = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; w += w_step, ++tl) {
        const TileCtx t = tile_ctx(w);
        ok = mbar_wait(bar_acc_empty, (tl & 1u) ^ 1u, abort_flag);
        for (int kt = 0; kt < t.num_kt && ok; ++kt, ++it) {
          const uint32_t s = it % S;
          ok = mbar_wait(bar_full + 8 * s, (it / S) & 1u, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = sbase + s * SLOT;
          const uint32_t sfa_col = tmem + ACC_COL + BN + SF_COLS * s;
          const uint32_t sfb_col = sfa_col + KK::kSfColsA;
          const int rem = t.K - kt * KK::kElemsPerTile;
          const int n_mma = min(KK::kMmas, rem / KK::kMmaK);
          // MMA k reads span k / 4 (its own 128-byte swizzle span of every
          // row); inside the span the descriptors' start address advances by
          // 32 bytes (2 units of 16) per MMA
          const uint64_t da = op_desc(st), db = op_desc(st + KK::kKT * A_BYTES);
          const uint32_t acc0 = kt > 0 ? 1u : 0u;
          auto issue = [&](int k) {
            // the 4-byte scale chunk of MMA k and the scale bytes inside it
            uint32_t sfa = sfa_col, sfb = sfb_col, sf_id = 0;
            if constexpr (KIND == KIND_MXF4) {
              sfa += 4 * (k >> 1);
              sfb += 8 * (k >> 1);
              sf_id = 2u * (uint32_t)(k & 1);
            } else if constexpr (KIND == KIND_NVF4) {
              sfa += 4 * k;
              sfb += 8 * k;
            } else {
              sfa += 4 * (k >> 2);
              sfb += 8 * (k >> 2);
              sf_id = (uint32_t)(k & 3);
            }
            const uint32_t acc = k > 0 ? 1u : acc0;
            const uint64_t off = (uint64_t)((A_BYTES >> 4) * (k >> 2) + 2 * (k & 3));   // A_BYTES == B_BYTES
            tc_mma_pair<KIND>(tmem + ACC_COL, da + off, db + off, make_idesc<KIND>(sf_id), sfa, sfb, acc);
          };
          if (n_mma == KK::kMmas) {
#pragma unroll
            for (int k = 0; k < KK::kMmas; ++k) issue(k);
          } else {
            for (int k = 0; k < n_mma; ++k) issue(k);
          }
          tc_commit_pair(bar_empty + 8 * s);
        }
        if (!ok) break;
        tc_commit_pair(bar_acc_full);
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, FP4Q_DEV_TIMEOUT);
      }
      // wait (bounded) until every tensor-core operation this lane issued finished
      asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar_drain)
                   : "memory");
      const uint64_t t0 = globaltimer();
      while (!mbar_try(bar_drain, 0) && globaltimer() - t0 < 2000000000ull) {
      }
    }
    __syncwarp();
  } else if (warp == KK::kChunkWarp) {
    if (lane == 0) {
      // ---------------- scale-chunk loader: a stage's compact chunks of this
      // CTA into its slot, once the slot's previous MMAs finished
      uint32_t it = 0;
      bool ok = true;
      for (int w = w_begin; w < w_end && ok; w += w_step) {
        const TileCtx t = tile_ctx(w);
        const bool rows = t.m0 < t.M;          // false only for the second CTA of a 128-row tail
        const bool rg1 = (t.n0 + 128) < t.N;   // the tile's second 128-row group of B exists
        const uint8_t* sfa_g;
        const uint8_t* sfb_g;
        if constexpr (GROUP) {
          sfa_g = ga.sfa[t.gi];
          sfb_g = ga.sfb[t.gi];
        } else {
          sfa_g = p.sfa;
          sfb_g = p.sfb;
        }
        const uint8_t* sfa_t = sfa_g + (size_t)(t.m0 / 128) * t.nq * 512;
        const uint8_t* sfb_t = sfb_g + (size_t)(t.n0 / 128) * t.nq * 512;
        for (int kt = 0; kt < t.num_kt; ++kt, ++it) {
          const int s = (int)(it % S);
          if (!mbar_wait(bar_empty + 8 * s, ((it / S) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const int q0 = kt * KK::kChunks;
          const uint32_t sf_bytes = (uint32_t)min(KK::kChunks, t.nq - q0) * 512u;
          const uint32_t sb = bar_sfd + 8 * s, ca = sbase + (uint32_t)s * SLOT + KK::kOpStage;
          mbar_expect_tx(sb, sf_bytes * ((rows ? 1u : 0u) + (rg1 ? 2u : 1u)));
          if (rows) bulk_load(ca, sfa_t + (size_t)q0 * 512, sf_bytes, sb);
          bulk_load(ca + KK::kChunks * 512, sfb_t + (size_t)q0 * 512, sf_bytes, sb);
          if (rg1) bulk_load(ca + 2 * KK::kChunks * 512, sfb_t + ((size_t)t.nq + q0) * 512, sf_bytes, sb);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, FP4Q_DEV_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp >= 6 && warp < 10) {
    // ---------------- scale writers: lane i of quarter q stores row i of the compact chunks
    // A stage's chunks land in its slot once the slot's previous MMAs have
    // finished (the producer waited for them), so the TMEM scale slot of the
    // stage is free too, and the full barrier of the slot is in this stage's
    // phase; one wait per stage.
    const uint32_t qbase = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    uint32_t it = 0;
    bool ok = true;
    for (int w = w_begin; w < w_end && ok; w += w_step) {
      const int num_kt = tile_ctx(w).num_kt;
      for (int kt = 0; kt < num_kt; ++kt, ++it) {
        const uint32_t s = it % S;
        ok = mbar_wait(bar_sfd + 8 * s, (it / S) & 1u, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ca = sbase + s * SLOT + KK::kOpStage, cb0 = ca + KK::kChunks * 512, cb1 = cb0 + KK::kChunks * 512;
        const uint32_t sfa_col = qbase + ACC_COL + BN + SF_COLS * s;
        // the slot's columns in order: A chunks (4 each), then per B chunk its two row groups
        uint32_t wv[KK::kSfCols];
#pragma unroll
        for (int c = 0; c < KK::kChunks; ++c) put4(wv + 4 * c, chunk_row(ca + 512u * c, lane));
#pragma unroll
        for (int c = 0; c < KK::kChunks; ++c) {
          put4(wv + KK::kSfColsA + 8 * c, chunk_row(cb0 + 512u * c, lane));
          put4(wv + KK::kSfColsA + 8 * c + 4, chunk_row(cb1 + 512u * c, lane));
        }
#pragma unroll
        for (int c = KK::kSfColsA + KK::kSfColsB; c < KK::kSfCols; ++c) wv[c] = 0u;
        if constexpr (KK::kSfCols == 16) {
          tmem_st16(sfa_col, wv);
        } else if constexpr (KK::kSfCols == 48) {
          tmem_st32(sfa_col, wv);
          tmem_st16(sfa_col + 32, wv + 32);
        } else {
          tmem_st32(sfa_col, wv);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) cluster_arrive(lead_full + 8 * s);
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      raise_status(p.status, FP4Q_DEV_TIMEOUT);
    }
  } else {
    // ---------------- epilogue (warps 2..5 and 10..13 -> TMEM lane quarters 2, 3, 0, 1)
    const int sp = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * sp) << 16) + ACC_COL;
    const int grp = warp < 6 ? 0 : 1;                              // warps 2-5: columns 0-127, 10-13: 128-255
    const int cbase = grp * KK::kEpiCols;                          // this warp's accumulator columns
    const int epi = grp * 4 + ((warp - 2) & 3);
    const uint32_t stg = stg_base + (uint32_t)epi * KK::kStgWarp;
    // swizzled 32-row boxes: 16-byte unit u of row `lane` sits at unit
    // u ^ (lane & 7) with 128-byte rows (fused kernels), u ^ ((lane >> 2) & 1)
    // with 32-byte rows (plain kernels)
    constexpr uint32_t BOXB = KK::kBoxBytes;
    static_assert(BOXB == 128 || BOXB == 32, "box row size");
    const uint32_t row_off = BOXB * (uint32_t)lane;
    const uint32_t swz = BOXB == 128 ? (uint32_t)(lane & 7) : (uint32_t)((lane >> 2) & 1);
    float alpha = 1.0f;
    if constexpr (KIND == KIND_NVF4 && !GROUP) alpha = __fmul_rn(*p.ts_a, *p.ts_b);
    uint32_t tl = 0;
    for (int w = w_begin; w < w_end; w += w_step, ++tl) {
      const TileCtx t = tile_ctx(w);
      const int m0 = t.m0, n0 = t.n0;
      const int y = m0 + 32 * sp;                // first row of this warp's slice
      const bool live = m0 < t.M;                // false only for the second CTA of a 128-row tail tile
      const CUtensorMap* mDh = map_dh(t.gi);
      const CUtensorMap* mDf = map_df(t.gi);
      bool want_bf16 = p.want_bf16, want_f32 = p.want_f32;
      if constexpr (GROUP) {
        want_bf16 = ga.want_bf16[t.gi];
        want_f32 = ga.want_f32[t.gi];
        if constexpr (KIND == KIND_NVF4) alpha = __fmul_rn(*ga.ts_a[t.gi], *ga.ts_b[t.gi]);
      }
      bool ok = mbar_wait(bar_acc_full, tl & 1u, abort_flag);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) {
        if (lane == 0) {
          *abort_flag = 1;
          raise_status(p.status, FP4Q_DEV_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const int ncols = min(BN, t.N - n0);   // 128 or 256
      if constexpr (FUSED) {
        // Fused output quantization.  The warp's 32 x 128 bf16 slice goes to
        // shared memory as two swizzled 32 x 64 boxes (the previous tile's
        // stores must have read them), the accumulator is released, the boxes
        // are stored by TMA when D is wanted, and each thread quantizes its
        // row from them, 32 values at a time.  Box rows are 128 bytes: 16-byte
        // unit u of row `lane` sits at unit u ^ (lane & 7).
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
#pragma unroll
        for (int c0 = 0; c0 < KK::kEpiCols; c0 += 32) {
          if (cbase + c0 < ncols) {
            uint32_t r[32];
            tmem_ld32(lane_base + (uint32_t)(cbase + c0), r);
            uint32_t hw[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
              if constexpr (KIND == KIND_NVF4) {
                a = __fmul_rn(a, alpha);
                b = __fmul_rn(b, alpha);
              }
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(a, b);
              hw[j] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            const uint32_t box = stg + 4096u * (uint32_t)(c0 / 64), u0 = 4u * (uint32_t)((c0 / 32) & 1);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              st_shared16(box + row_off + 16u * ((u0 + j) ^ swz),
                          make_uint4(hw[4 * j], hw[4 * j + 1], hw[4 * j + 2], hw[4 * j + 3]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) cluster_arrive(lead_acc_empty);
        if (!live) continue;
        if (want_bf16) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            for (int b = 0; 64 * b < KK::kEpiCols && cbase + 64 * b < ncols; ++b)
              tma_store_2d(&tmDh, n0 + cbase + 64 * b, y, stg + 4096u * (uint32_t)b);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
        const int64_t row = (int64_t)y + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < KK::kEpiCols && cbase + c0 < ncols; c0 += 32) {
          const uint32_t box = stg + 4096u * (uint32_t)(c0 / 64), u0 = 4u * (uint32_t)((c0 / 32) & 1);
          uint32_t wq[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) put4(wq + 4 * j, chunk_row(box + row_off + 16u * ((u0 + j) ^ swz), 0));
          float2 P[16];
          chunk_from_bf16_words(wq, p.q_sgn, P);
          // MX output scales: H16's 1/4 goes into the power-of-two block scale
          if (p.q_nh == 16) rotate_chunk<16, false>(P);
          else if (p.q_nh == 32) rotate_chunk<32>(P);
          ChunkOut o;
          const int64_t col = (int64_t)n0 + cbase + c0;
          quantize_chunk<(QG >= 0 ? QG : 0), FP4Q_SCALE_MX, QR>(P, 0.0f, (uint64_t)(row * p.N + col), 0u, p.q_keys,
                                                                 p.q_e4m3 != nullptr, p.status, o,
                                                                 p.q_nh == 16 ? 2 : 0);
          *reinterpret_cast<uint4*>(p.q_codes + row * (p.N / 2) + col / 2) = make_uint4(o.w[0], o.w[1], o.w[2], o.w[3]);
          const int64_t nkb = p.N / 32, k = col / 32;
          p.q_scales[p.q_sf_mma ? sf_mma_offset(row, k, nkb) : row * nkb + k] = (uint8_t)o.sbytes;
          if (p.q_e4m3) {
            uint4* ep = reinterpret_cast<uint4*>(p.q_e4m3 + row * p.N + col);
            ep[0] = make_uint4(o.e4[0], o.e4[1], o.e4[2], o.e4[3]);
            ep[1] = make_uint4(o.e4[4], o.e4[5], o.e4[6], o.e4[7]);
          }
        }
      } else {
        // Plain output through a 32-row x 32-byte swizzled box per warp, stored
        // by TMA: fp32 columns as they leave TMEM, the bf16 row slice once the
        // accumulator is released.  The accumulator is released as soon as the
        // last load has landed in registers; that chunk is converted after.
        constexpr int ECOLS = KK::kEpiCols, UNITS = (int)BOXB / 16;   // 16-byte units per box row
        constexpr int FCOLS = (int)BOXB / 4, HCOLS = (int)BOXB / 2;   // columns of an fp32 / bf16 box
        constexpr int LCOLS = 64;                                     // columns per TMEM load
        constexpr int NLOADS = ECOLS / LCOLS;
        static_assert(ECOLS % LCOLS == 0 && ECOLS / 2 >= 32, "epilogue columns");
        uint32_t h[ECOLS / 2];   // this warp's columns of the row as packed bf16
        // alpha, the fp32 stores and the bf16 words of the chunk at column c0
        auto consume = [&](int c0, uint32_t (&r)[LCOLS]) {
          if constexpr (KIND == KIND_NVF4) {
#pragma unroll
            for (int j = 0; j < LCOLS; ++j) r[j] = __float_as_uint(__fmul_rn(__uint_as_float(r[j]), alpha));
          }
          if (want_f32 && live) {
#pragma unroll
            for (int hh = 0; hh < LCOLS / FCOLS; ++hh) {
              if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
              __syncwarp();
#pragma unroll
              for (int u = 0; u < UNITS; ++u)
                st_shared16(stg + row_off + 16u * ((uint32_t)u ^ swz),
                            make_uint4(r[FCOLS * hh + 4 * u], r[FCOLS * hh + 4 * u + 1], r[FCOLS * hh + 4 * u + 2],
                                       r[FCOLS * hh + 4 * u + 3]));
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(mDf, n0 + cbase + c0 + FCOLS * hh, y, stg);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
              }
            }
          }
#pragma unroll
          for (int j = 0; j < LCOLS / 2; ++j) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            h[c0 / 2 + j] = *reinterpret_cast<const uint32_t*>(&b2);
          }
        };
        auto release = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) cluster_arrive(lead_acc_empty);
        };
        // ncols is 128 or 256 and a warp's columns start at 0 or 128, so a
        // warp loads all of its columns or none
        if (cbase < ncols) {
          const uint32_t zero[32] = {};
          uint32_t r[LCOLS];
#pragma unroll
          for (int k = 0; k < NLOADS; ++k) {
            tmem_ld64(lane_base + (uint32_t)(cbase + k * LCOLS), r, k > 0 ? h + (k * LCOLS / 2 - 32) : zero);
            if (k + 1 < NLOADS) consume(k * LCOLS, r);
          }
          // accumulator read out: let the next tile's MMAs start, then convert the last chunk
          release();
          consume(ECOLS - LCOLS, r);
        } else {
          release();
        }
        if (want_bf16 && live) {
#pragma unroll
          for (int b = 0; b < ECOLS / HCOLS; ++b) {
            if (cbase + HCOLS * b < ncols) {
              if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
              __syncwarp();
#pragma unroll
              for (int u = 0; u < UNITS; ++u)
                st_shared16(stg + row_off + 16u * ((uint32_t)u ^ swz),
                            make_uint4(h[(HCOLS / 2) * b + 4 * u], h[(HCOLS / 2) * b + 4 * u + 1],
                                       h[(HCOLS / 2) * b + 4 * u + 2], h[(HCOLS / 2) * b + 4 * u + 3]));
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(mDh, n0 + cbase + HCOLS * b, y, stg);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
              }
            }
          }
        }
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }
  tc_fence_before();
  // no CTA of a pair may leave while its peer can still use its shared or tensor memory
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ------------------------------------------------------------ host side
// 2-D byte tensor [rows][row_bytes], box = 128 bytes x 128 rows, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, row_bytes, rows, row_bytes, (uint32_t)KROW, 128u,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}
// Output [M][N] of bf16 or fp32, boxes of 32 rows x box_bytes with the
// swizzle of that row size (32 bytes for the plain kernels, 128 for the fused
// ones); the kernels' staging uses the same box.
bool make_out_map(CUtensorMap* m, const void* base, uint64_t N, uint64_t M, bool f32, uint32_t box_bytes) {
  return encode_tmap_2d(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, N, M,
                        N * (f32 ? 4u : 2u), box_bytes / (f32 ? 4u : 2u), 32u,
                        box_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B);
}
constexpr uint32_t kPlainBox = KindK<KIND_MXF4, false>::kBoxBytes;
constexpr uint32_t kFusedBox = KindK<KIND_MXF4, true>::kBoxBytes;
static_assert(kPlainBox == 32 && kFusedBox == 128, "output maps");

// Opt a kernel into its dynamic shared memory and find how many pairs can be
// resident at once, once per device (cached).  Returns 0 on error.
template <class Kern>
int resident_pairs(Kern kern, int smem, int threads, unsigned& done, int (&max_pairs)[32]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const unsigned bit = dev < 32 ? (1u << dev) : 0u;
  if (bit && (done & bit)) return max_pairs[dev];
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_sms() & ~1u, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return 0;
  if (bit) {
    max_pairs[dev] = n;
    done |= bit;
  }
  return n;
}

template <class Kern, class... Args>
cudaError_t launch_pairs(Kern kern, int pairs, int smem, int threads, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the kernel waits (griddepcontrol.wait)
  // for the previous grid before touching global memory
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int KIND, int QG = -1, int QR = FP4Q_RTNE>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& dh, const CUtensorMap& df,
                        const GemmParams& p, cudaStream_t s) {
  using KK = KindK<KIND, (QG >= 0)>;
  static unsigned done = 0;   // one bit per device ordinal < 32
  static int max_pairs[32] = {};
  auto kern = bs_gemm_kernel<KIND, QG, QR, false>;
  int pairs = resident_pairs(kern, KK::kSmem, KK::kThreads, done, max_pairs);
  if (pairs <= 0) return cudaErrorInvalidConfiguration;
  const int tiles = ((p.M + TM - 1) / TM) * ((p.N + BN - 1) / BN);
  if (tiles < pairs) pairs = tiles;
  return launch_pairs(kern, pairs, KK::kSmem, KK::kThreads, s, a, b, dh, df, p, NoGroupArgs{});
}

// Static schedule of a grouped launch: tiles taken longest first (a tile
// costs 4 per K-tile of 256 plus 10 for its epilogue, in about a quarter of a
// stage's time), each given to the pair with the least work so far (a binary
// heap of pair loads); every pair's tiles are then stored together, in the
// order it received them.  The last schedule is kept per host thread and
// reused while the shapes and the pair count repeat.  Returns the pair count.
int group_schedule(GroupArgs& ga, int units) {
  const int total = ga.tile0[ga.np];
  if (units > total) units = total;
  if (units > kGroupMaxUnits) units = kGroupMaxUnits;
  struct Cache {
    int np = 0, units = 0;
    int32_t M[kGroupMax], N[kGroupMax], K[kGroupMax];
    uint16_t unit_begin[kGroupMaxUnits + 1];
    uint16_t order[kGroupMaxTiles];
  };
  static thread_local Cache cache;
  bool hit = cache.np == ga.np && cache.units == units;
  for (int i = 0; hit && i < ga.np; ++i)
    hit = cache.M[i] == ga.M[i] && cache.N[i] == ga.N[i] && cache.K[i] == ga.K[i];
  if (!hit) {
    int gorder[kGroupMax];
    for (int i = 0; i < ga.np; ++i) gorder[i] = i;
    auto cost = [&](int gi) { return (int64_t)4 * ((ga.K[gi] + 255) / 256) + 10; };
    for (int i = 1; i < ga.np; ++i)   // GEMMs by decreasing tile cost (insertion sort, np <= 4)
      for (int j = i; j > 0 && cost(gorder[j]) > cost(gorder[j - 1]); --j) {
        const int t = gorder[j];
        gorder[j] = gorder[j - 1];
        gorder[j - 1] = t;
      }
    // min-heap of (load, unit); ties go to the lower unit
    static thread_local int64_t hload[kGroupMaxUnits];
    static thread_local int hunit[kGroupMaxUnits];
    static thread_local uint16_t owner[kGroupMaxTiles], by_seq[kGroupMaxTiles];
    static thread_local int count[kGroupMaxUnits + 1];
    auto less = [&](int x, int y) { return hload[x] < hload[y] || (hload[x] == hload[y] && hunit[x] < hunit[y]); };
    for (int u = 0; u < units; ++u) {
      hload[u] = 0;
      hunit[u] = u;
    }
    int seq = 0;
    for (int i = 0; i < ga.np; ++i) {
      const int gi = gorder[i];
      for (int g = ga.tile0[gi]; g < ga.tile0[gi + 1]; ++g) {
        owner[seq] = (uint16_t)hunit[0];
        by_seq[seq++] = (uint16_t)g;
        hload[0] += cost(gi);
        for (int x = 0;;) {   // sift the root down
          const int l = 2 * x + 1, r = l + 1;
          int m = x;
          if (l < units && less(l, m)) m = l;
          if (r < units && less(r, m)) m = r;
          if (m == x) break;
          const int64_t tl = hload[x];
          const int tu = hunit[x];
          hload[x] = hload[m];
          hunit[x] = hunit[m];
          hload[m] = tl;
          hunit[m] = tu;
          x = m;
        }
      }
    }
    for (int u = 0; u <= units; ++u) count[u] = 0;
    for (int k = 0; k < seq; ++k) ++count[owner[k] + 1];
    for (int u = 0; u < units; ++u) count[u + 1] += count[u];
    for (int u = 0; u <= units; ++u) cache.unit_begin[u] = (uint16_t)count[u];
    for (int k = 0; k < seq; ++k) cache.order[count[owner[k]]++] = by_seq[k];
    cache.np = ga.np;
    cache.units = units;
    for (int i = 0; i < ga.np; ++i) {
      cache.M[i] = ga.M[i];
      cache.N[i] = ga.N[i];
      cache.K[i] = ga.K[i];
    }
  }
  memcpy(ga.unit_begin, cache.unit_begin, sizeof(uint16_t) * (units + 1));
  memcpy(ga.order, cache.order, sizeof(uint16_t) * total);
  return units;
}

// One launch over the GEMMs of ga; p supplies the status word only.
template <int KIND>
cudaError_t launch_gemm_group(GroupArgs& ga, const GemmParams& p, cudaStream_t s) {
  using KK = KindK<KIND, false>;
  static unsigned done = 0;
  static int max_pairs[32] = {};
  auto kern = bs_gemm_kernel<KIND, -1, FP4Q_RTNE, true>;
  const int pairs = resident_pairs(kern, KK::kSmem, KK::kThreads, done, max_pairs);
  if (pairs <= 0) return cudaErrorInvalidConfiguration;
  const int units = group_schedule(ga, pairs);
  return launch_pairs(kern, units, KK::kSmem, KK::kThreads, s, ga.a[0], ga.b[0], ga.dh[0], ga.df[0], p, ga);
}

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks shared by the entry points, the kernel parameters and the operand /
// output tensor maps.  Returns FP4Q_OK or the error status.
int32_t prepare_gemm(const fp4q_operand* A, const fp4q_operand* B, int64_t M, int64_t N, int64_t K, int32_t grid,
                     int32_t scale, void* D_bf16, float* D_f32, uint32_t* d_status, bool fused, int& kind,
                     GemmParams& p, CUtensorMap& ta, CUtensorMap& tb, CUtensorMap& tdh, CUtensorMap& tdf) {
  if (!A || !B) return FP4Q_ERR_INVALID_ARG;
  if (grid != FP4Q_GRID_E2M1 && grid != FP4Q_GRID_E1M2 && grid != FP4Q_GRID_E2M1_R4) return FP4Q_ERR_INVALID_ARG;
  if (scale != FP4Q_SCALE_MX && scale != FP4Q_SCALE_NV) return FP4Q_ERR_INVALID_ARG;
  if (grid == FP4Q_GRID_E1M2 && scale == FP4Q_SCALE_NV) return FP4Q_ERR_UNSUPPORTED;
  if (M <= 0 || N <= 0 || K <= 0) return FP4Q_ERR_INVALID_ARG;
  if (M % 128 || N % 128) return FP4Q_ERR_INVALID_ARG;
  if (K % (scale == FP4Q_SCALE_NV ? 64 : 128)) return FP4Q_ERR_INVALID_ARG;
  if (M / 128 > 65535 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return FP4Q_ERR_INVALID_ARG;
  kind = grid == FP4Q_GRID_E1M2 ? KIND_F8 : (scale == FP4Q_SCALE_NV ? KIND_NVF4 : KIND_MXF4);
  const void* a_data = kind == KIND_F8 ? (const void*)A->e4m3 : (const void*)A->codes;
  const void* b_data = kind == KIND_F8 ? (const void*)B->e4m3 : (const void*)B->codes;
  if (!a_data || !b_data || !A->scales || !B->scales) return FP4Q_ERR_INVALID_ARG;
  if (kind == KIND_NVF4 && (!A->tensor_scale || !B->tensor_scale)) return FP4Q_ERR_INVALID_ARG;
  if (!al(a_data, 16) || !al(b_data, 16) || !al(A->scales, 16) || !al(B->scales, 16)) return FP4Q_ERR_ALIGNMENT;
  if ((D_bf16 && !al(D_bf16, 16)) || (D_f32 && !al(D_f32, 16))) return FP4Q_ERR_ALIGNMENT;
  const uint64_t row_bytes = kind == KIND_F8 ? (uint64_t)K : (uint64_t)K / 2;
  memset(&p, 0, sizeof p);
  p.sfa = A->scales;
  p.sfb = B->scales;
  p.ts_a = A->tensor_scale;
  p.ts_b = B->tensor_scale;
  p.status = d_status;
  p.want_bf16 = D_bf16 != nullptr;
  p.want_f32 = D_f32 != nullptr;
  p.M = (int32_t)M;
  p.N = (int32_t)N;
  p.K = (int32_t)K;
  memset(&tdh, 0, sizeof(tdh));
  memset(&tdf, 0, sizeof(tdf));
  if (!make_map(&ta, a_data, row_bytes, (uint64_t)M) || !make_map(&tb, b_data, row_bytes, (uint64_t)N))
    return FP4Q_ERR_CUDA;
  if (D_bf16 && !make_out_map(&tdh, D_bf16, (uint64_t)N, (uint64_t)M, false, fused ? kFusedBox : kPlainBox))
    return FP4Q_ERR_CUDA;
  if (D_f32 && !make_out_map(&tdf, D_f32, (uint64_t)N, (uint64_t)M, true, kPlainBox)) return FP4Q_ERR_CUDA;
  return FP4Q_OK;
}

template <int QG, int QR>
cudaError_t launch_kind(int kind, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tdh,
                        const CUtensorMap& tdf, const GemmParams& p, cudaStream_t s) {
  if (kind == KIND_MXF4) return launch_gemm<KIND_MXF4, QG, QR>(ta, tb, tdh, tdf, p, s);
  if (kind == KIND_NVF4) return launch_gemm<KIND_NVF4, QG, QR>(ta, tb, tdh, tdf, p, s);
  return launch_gemm<KIND_F8, QG, QR>(ta, tb, tdh, tdf, p, s);
}

}  // namespace
}  // namespace fp4q

extern "C" int32_t fp4q_gemm(const fp4q_operand* A, const fp4q_operand* B, int64_t M, int64_t N, int64_t K,
                             int32_t grid, int32_t scale, void* D_bf16, float* D_f32, uint32_t* d_status,
                             void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_gemm");
  using namespace fp4q;
  if (!D_bf16 && !D_f32) return FP4Q_ERR_INVALID_ARG;
  int kind = 0;
  GemmParams p;
  CUtensorMap ta, tb, tdh, tdf;
  const int32_t st =
      prepare_gemm(A, B, M, N, K, grid, scale, D_bf16, D_f32, d_status, false, kind, p, ta, tb, tdh, tdf);
  if (st != FP4Q_OK) return st;
  const cudaError_t e = launch_kind<-1, FP4Q_RTNE>(kind, ta, tb, tdh, tdf, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

extern "C" int32_t fp4q_gemm_group(const fp4q_gemm_problem* problems, int32_t count, int32_t grid, int32_t scale,
                                   uint32_t* d_status, void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_gemm_group");
  using namespace fp4q;
  if (!problems || count < 1 || count > kGroupMax) return FP4Q_ERR_INVALID_ARG;
  static thread_local GroupArgs ga;   // ~19 KB: copied into the launch, reused by the next call
  memset(&ga, 0, sizeof(GroupArgs));
  ga.np = count;
  ga.tile0[0] = 0;
  int kind = KIND_MXF4;
  GemmParams p0;
  for (int i = 0; i < count; ++i) {
    const fp4q_gemm_problem& q = problems[i];
    if (!q.D_bf16 && !q.D_f32) return FP4Q_ERR_INVALID_ARG;
    GemmParams pi;
    const int32_t st = prepare_gemm(q.A, q.B, q.M, q.N, q.K, grid, scale, q.D_bf16, q.D_f32, d_status, false, kind,
                                    pi, ga.a[i], ga.b[i], ga.dh[i], ga.df[i]);
    if (st != FP4Q_OK) return st;
    if (i == 0) p0 = pi;
    ga.sfa[i] = pi.sfa;
    ga.sfb[i] = pi.sfb;
    ga.ts_a[i] = pi.ts_a;
    ga.ts_b[i] = pi.ts_b;
    ga.want_bf16[i] = pi.want_bf16;
    ga.want_f32[i] = pi.want_f32;
    ga.M[i] = pi.M;
    ga.N[i] = pi.N;
    ga.K[i] = pi.K;
    const int64_t tiles = ((q.M + TM - 1) / TM) * ((q.N + BN - 1) / BN);
    if (ga.tile0[i] + tiles > kGroupMaxTiles) return FP4Q_ERR_UNSUPPORTED;
    ga.tile0[i + 1] = ga.tile0[i] + (int32_t)tiles;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (kind == KIND_MXF4) e = launch_gemm_group<KIND_MXF4>(ga, p0, s);
  else if (kind == KIND_NVF4) e = launch_gemm_group<KIND_NVF4>(ga, p0, s);
  else e = launch_gemm_group<KIND_F8>(ga, p0, s);
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

extern "C" int32_t fp4q_gemm_quantize(const fp4q_operand* A, const fp4q_operand* B, int64_t M, int64_t N, int64_t K,
                                      int32_t grid, int32_t scale, void* D_bf16, const fp4q_config* out_cfg,
                                      fp4q_operand* out, uint32_t* d_status, void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_gemm_quantize");
  using namespace fp4q;
  if (!out_cfg || !out || !out->codes || !out->scales) return FP4Q_ERR_INVALID_ARG;
  const fp4q_config& c = *out_cfg;
  if (c.grid != FP4Q_GRID_E2M1 && c.grid != FP4Q_GRID_E1M2 && c.grid != FP4Q_GRID_E2M1_R4) return FP4Q_ERR_INVALID_ARG;
  if (c.rot != FP4Q_ROT_NONE && c.rot != FP4Q_ROT_H16 && c.rot != FP4Q_ROT_H32) return FP4Q_ERR_INVALID_ARG;
  if (c.round != FP4Q_RTNE && c.round != FP4Q_SR) return FP4Q_ERR_INVALID_ARG;
  if (c.sf_layout != FP4Q_SF_PLAIN && c.sf_layout != FP4Q_SF_MMA) return FP4Q_ERR_INVALID_ARG;
  // one pass over D: MX scales only (NV needs the global amax of the whole rotated output first),
  // and only the row-wise copy (the column-wise blocks would span 32 tiles' rows)
  if (c.scale != FP4Q_SCALE_MX || !c.want_row || c.want_col) return FP4Q_ERR_UNSUPPORTED;
  if (c.emit_e4m3 && !out->e4m3) return FP4Q_ERR_INVALID_ARG;
  if (!al(out->codes, 16) || (c.emit_e4m3 && !al(out->e4m3, 16))) return FP4Q_ERR_ALIGNMENT;
  int kind = 0;
  GemmParams p;
  CUtensorMap ta, tb, tdh, tdf;
  const int32_t st =
      prepare_gemm(A, B, M, N, K, grid, scale, D_bf16, nullptr, d_status, true, kind, p, ta, tb, tdh, tdf);
  if (st != FP4Q_OK) return st;
  p.q_codes = out->codes;
  p.q_scales = out->scales;
  p.q_e4m3 = c.emit_e4m3 ? out->e4m3 : nullptr;
  p.q_seed = c.sr_seed;
  philox_round_keys(c.sr_seed, p.q_keys);
  p.q_nh = c.rot;
  p.q_sf_mma = c.sf_layout == FP4Q_SF_MMA;
  for (int t = 0; t < 32; ++t) p.q_sgn[t] = (c.rot && ((c.sign_mask_row >> (t % c.rot)) & 1u)) ? 0x80000000u : 0u;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (c.grid == FP4Q_GRID_E2M1)
    e = c.round == FP4Q_SR ? launch_kind<FP4Q_GRID_E2M1, FP4Q_SR>(kind, ta, tb, tdh, tdf, p, s)
                           : launch_kind<FP4Q_GRID_E2M1, FP4Q_RTNE>(kind, ta, tb, tdh, tdf, p, s);
  else if (c.grid == FP4Q_GRID_E1M2)
    e = c.round == FP4Q_SR ? launch_kind<FP4Q_GRID_E1M2, FP4Q_SR>(kind, ta, tb, tdh, tdf, p, s)
                           : launch_kind<FP4Q_GRID_E1M2, FP4Q_RTNE>(kind, ta, tb, tdh, tdf, p, s);
  else
    e = c.round == FP4Q_SR ? launch_kind<FP4Q_GRID_E2M1_R4, FP4Q_SR>(kind, ta, tb, tdh, tdf, p, s)
                           : launch_kind<FP4Q_GRID_E2M1_R4, FP4Q_RTNE>(kind, ta, tb, tdh, tdf, p, s);
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}
