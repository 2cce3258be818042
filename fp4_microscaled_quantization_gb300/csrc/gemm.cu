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
// Structure (persistent, one CTA per SM walking 128 x 256 output tiles, 192
// threads):
//   warp 0      TMA producer: A/B tiles (128-byte swizzled K-major rows) by
//               cp.async.bulk.tensor, scale-factor chunks by cp.async.bulk,
//               into a 4-stage ring guarded by full/empty mbarriers.
//   warp 1      owns the TMEM allocation; one lane copies each stage's scale
//               factors to TMEM (tcgen05.cp 32x128b.warpx4) and issues the
//               MMAs, then tcgen05.commit frees the stage.
//   warps 2-5   epilogue: TMEM -> registers (tcgen05.ld), alpha, bf16/fp32
//               stores; TMEM is released before the global stores so the
//               next tile's MMAs overlap them.
// Every mbarrier wait is bounded (about 2 s of %globaltimer); on expiry the
// CTA raises FP4Q_DEV_TIMEOUT, stops issuing work, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/fp4q.h"
#include "fp4q_dev.cuh"
#include "fp4q_internal.h"

#ifndef FP4Q_GEMM_PAIR
#define FP4Q_GEMM_PAIR 0
#endif

namespace fp4q {
namespace {

enum { KIND_MXF4 = 0, KIND_NVF4 = 1, KIND_F8 = 2 };

constexpr int BM = 128;              // tile rows (TMEM lanes)
constexpr int BN = 256;              // tile columns (MMA N)
constexpr int KROW = 128;            // bytes of one operand row per K-tile (one 128B swizzle span)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * KROW;   // 16 KB
constexpr int B_BYTES = BN * KROW;   // 32 KB
constexpr int SFA_OFF = A_BYTES + B_BYTES;
constexpr int SFB_OFF = SFA_OFF + 4 * 512;
constexpr int STAGE_BYTES = SFB_OFF + 8 * 512;   // 55296, a multiple of 1024
constexpr int BAR_OFF = STAGES * STAGE_BYTES;
constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;  // + barriers + alignment slack
constexpr int NTHREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;                   // accumulator columns [0, 256)
constexpr uint32_t SF_COL0 = 256;                 // 48 scale-factor columns per stage after it
constexpr uint32_t SF_COLS_PER_STAGE = 48;

template <int KIND>
struct KindK {
  // chunks = groups of 4 consecutive scale bytes of one 128-row group
  static constexpr int kChunksPerTile = KIND == KIND_MXF4 ? 2 : (KIND == KIND_NVF4 ? 4 : 1);
  static constexpr int kElemsPerTile = KIND == KIND_F8 ? 128 : 256;
  static constexpr int kMmaK = KIND == KIND_F8 ? 32 : 64;
  static constexpr int kBlock = KIND == KIND_NVF4 ? 16 : 32;
};

struct GemmParams {
  const uint8_t* sfa;     // MMA scale layout of A (M x K/b)
  const uint8_t* sfb;     // MMA scale layout of B (N x K/b)
  const float* ts_a;      // NV tensor scales (or null)
  const float* ts_b;
  uint16_t* d_bf16;
  float* d_f32;
  uint32_t* status;
  int32_t M, N, K;
};

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
    if ((i & 255u) == 255u) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > 2000000000ull) return false;
    }
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(tm), "r"(x), "r"(y), "r"(bar)
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
// A 32-row x 16-byte scale chunk (no swizzle, 8-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) { return sdesc(saddr, 16, 128, 0); }

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
template <int KIND>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
  if constexpr (KIND == KIND_MXF4) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p; }"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
  } else if constexpr (KIND == KIND_NVF4) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p; }"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
  } else {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p; }"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
  }
}

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

// Instruction descriptor of the block-scaled kinds: B scale id in bits 4-5,
// A/B element types in 7-9 / 10-12, K-major A and B, N >> 3 in 17-22, scale
// type in 23 (1 = E8M0, 0 = E4M3), M >> 4 in 24-28, A scale id in 29-30.
template <int KIND, int MM = BM>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id) {
  constexpr uint32_t ty = KIND == KIND_F8 ? 0u : 1u;   // E4M3 (f8f6f4) or E2M1 (mxf4 kinds)
  constexpr uint32_t sfmt = KIND == KIND_NVF4 ? 0u : 1u;
  return (sf_id << 4) | (ty << 7) | (ty << 10) | ((uint32_t)(BN >> 3) << 17) | (sfmt << 23) |
         ((uint32_t)(MM >> 4) << 24) | (sf_id << 29);
}

// ------------------------------------------------------------ the kernel
// Persistent: CTA b owns tiles b, b + G, b + 2G, ... (G = gridDim.x), tile id
// -> (m block = id / n_blocks, n block = id % n_blocks).  The producer and
// the MMA issuer stream through every (tile, K-tile) pair of the CTA without
// draining the ring between tiles.  The accumulator is single-buffered: the
// epilogue pulls a finished tile out of TMEM (as packed bf16 when only bf16 is
// wanted), releases TMEM through acc_empty, and only then writes global
// memory, so the next tile's MMAs overlap those stores.
template <int KIND>
__global__ void __launch_bounds__(NTHREADS, 1)
    bs_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  using KK = KindK<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + BAR_OFF;          // STAGES x 8 bytes
  const uint32_t bar_empty = bar_full + 8 * STAGES;   // STAGES x 8 bytes
  const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BAR_OFF + 16 * STAGES + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + BAR_OFF + 16 * STAGES + 24);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blocks = (p.N + BN - 1) / BN;
  const int n_tiles = (p.M / BM) * n_blocks;
  const int num_kt = (p.K + KK::kElemsPerTile - 1) / KK::kElemsPerTile;
  const int nq = p.K / KK::kBlock / 4;   // scale chunks per 128-row group

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 4);   // one arrival per epilogue warp
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
      uint32_t it = 0;
      for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
        const int m0 = (tile / n_blocks) * BM, n0 = (tile % n_blocks) * BN;
        const bool rg1 = (n0 + 128) < p.N;
        for (int kt = 0; kt < num_kt; ++kt, ++it) {
          const int s = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag)) {
            *abort_flag = 1;
            raise_status(p.status, FP4Q_DEV_TIMEOUT);
            break;
          }
          const int q0 = kt * KK::kChunksPerTile;
          const int nch = min(KK::kChunksPerTile, nq - q0);
          const uint32_t sf_bytes = (uint32_t)nch * 512u;
          const uint32_t tx = A_BYTES + B_BYTES + sf_bytes * (rg1 ? 3u : 2u);
          const uint32_t st = sbase + (uint32_t)s * STAGE_BYTES;
          mbar_expect_tx(bar_full + 8 * s, tx);
          tma_load_2d(st, &tmA, kt * KROW, m0, bar_full + 8 * s);
          tma_load_2d(st + A_BYTES, &tmB, kt * KROW, n0, bar_full + 8 * s);
          bulk_load(st + SFA_OFF, p.sfa + ((size_t)(m0 / 128) * nq + q0) * 512, sf_bytes, bar_full + 8 * s);
          bulk_load(st + SFB_OFF, p.sfb + ((size_t)(n0 / 128) * nq + q0) * 512, sf_bytes, bar_full + 8 * s);
          if (rg1)
            bulk_load(st + SFB_OFF + KK::kChunksPerTile * 512, p.sfb + ((size_t)(n0 / 128 + 1) * nq + q0) * 512,
                      sf_bytes, bar_full + 8 * s);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      uint32_t it = 0, tl = 0;
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tl) {
        if (!mbar_wait(bar_acc_empty, (tl & 1u) ^ 1u, abort_flag)) {
          *abort_flag = 1;
          raise_status(p.status, FP4Q_DEV_TIMEOUT);
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kt = 0; kt < num_kt; ++kt, ++it) {
          const int s = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar_full + 8 * s, ph, abort_flag)) {
            *abort_flag = 1;
            raise_status(p.status, FP4Q_DEV_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + (uint32_t)s * STAGE_BYTES;
          const uint32_t sfa_col = tmem + SF_COL0 + SF_COLS_PER_STAGE * (uint32_t)s;
          const uint32_t sfb_col = sfa_col + 16;
          const int q0 = kt * KK::kChunksPerTile;
          const int nch = min(KK::kChunksPerTile, nq - q0);
          for (int c = 0; c < nch; ++c) {
            tc_cp_sf(sfa_col + 4 * c, sf_desc(st + SFA_OFF + 512 * c));
            tc_cp_sf(sfb_col + 8 * c, sf_desc(st + SFB_OFF + 512 * c));
            tc_cp_sf(sfb_col + 8 * c + 4, sf_desc(st + SFB_OFF + KK::kChunksPerTile * 512 + 512 * c));
          }
          const int rem = p.K - kt * KK::kElemsPerTile;
          const int n_mma = min(4, rem / KK::kMmaK);
          for (int k = 0; k < n_mma; ++k) {
            uint32_t sfa = sfa_col, sfb = sfb_col, sf_id = 0;
            if constexpr (KIND == KIND_MXF4) {
              sfa += 4 * (k >> 1);
              sfb += 8 * (k >> 1);
              sf_id = 2u * (uint32_t)(k & 1);
            } else if constexpr (KIND == KIND_NVF4) {
              sfa += 4 * k;
              sfb += 8 * k;
            } else {
              sf_id = (uint32_t)k;
            }
            tc_mma<KIND>(tmem + ACC_COL, op_desc(st + 32 * k), op_desc(st + A_BYTES + 32 * k),
                         make_idesc<KIND>(sf_id), sfa, sfb, (kt > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(bar_empty + 8 * s);
        }
        if (!ok) break;
        tc_commit(bar_acc_full);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5 -> TMEM lane quarters 2, 3, 0, 1)
    const int sp = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * sp) << 16) + ACC_COL;
    float alpha = 1.0f;
    if constexpr (KIND == KIND_NVF4) alpha = __fmul_rn(*p.ts_a, *p.ts_b);
    uint32_t tl = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tl) {
      const int m0 = (tile / n_blocks) * BM, n0 = (tile % n_blocks) * BN;
      const int row = m0 + 32 * sp + lane;
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
      const int ncols = min(BN, p.N - n0);   // a multiple of 128
      if (p.d_f32 == nullptr) {
        // bf16 only: whole row to registers, release TMEM, then store
        uint32_t h[BN / 2];
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          if (c0 < ncols) {
            uint32_t r[32];
            tmem_ld32(lane_base + (uint32_t)c0, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
              if constexpr (KIND == KIND_NVF4) {
                a = __fmul_rn(a, alpha);
                b = __fmul_rn(b, alpha);
              }
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(a, b);
              h[c0 / 2 + j] = *reinterpret_cast<const uint32_t*>(&b2);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_acc_empty) : "memory");
        uint4* dst = reinterpret_cast<uint4*>(p.d_bf16 + (size_t)row * p.N + n0);
#pragma unroll
        for (int j = 0; j < BN / 8; ++j)
          if (8 * j < ncols) dst[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
      } else {
        // fp32 (and optional bf16): chunk by chunk, TMEM released at the end
        for (int c0 = 0; c0 < ncols; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(lane_base + (uint32_t)c0, r);
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = __uint_as_float(r[j]);
            if constexpr (KIND == KIND_NVF4) v[j] = __fmul_rn(v[j], alpha);
          }
          const size_t off = (size_t)row * p.N + n0 + c0;
          float4* df = reinterpret_cast<float4*>(p.d_f32 + off);
#pragma unroll
          for (int j = 0; j < 8; ++j) df[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          if (p.d_bf16) {
            uint32_t hb[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
              hb[j] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            uint4* db = reinterpret_cast<uint4*>(p.d_bf16 + off);
#pragma unroll
            for (int j = 0; j < 4; ++j) db[j] = make_uint4(hb[4 * j], hb[4 * j + 1], hb[4 * j + 2], hb[4 * j + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_acc_empty) : "memory");
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}


// ------------------------------------------------------------ CTA-pair kernel
// Two CTAs of a cluster share one 256 x 256 output tile through
// tcgen05.mma.cta_group::2 (M = 256 across the pair, N = 256): each CTA loads
// its own 128 rows of A and its own 128-row half of B (so each SM moves 32 KB
// of operands per K-tile instead of 48 KB), plus the scale chunks of its A rows
// and of both B row groups, and signals the leader CTA's full barrier
// (cp.async.bulk.tensor ... .cta_group::2).  The leader (cluster rank 0)
// copies scales to TMEM and issues the MMAs for both; commits are multicast to
// both CTAs' empty / accumulator barriers; each CTA's epilogue drains its own
// 128 accumulator rows and releases them with an arrive on the leader.
namespace pairk {

constexpr int A_BYTES = 128 * KROW;   // this CTA's 128 rows of A
constexpr int B_BYTES = 128 * KROW;   // this CTA's half of B

template <int KIND>
struct Layout {
  static constexpr int kSfChunk = KindK<KIND>::kChunksPerTile * 512;   // one row group, one K-tile
  static constexpr int SFA_OFF = A_BYTES + B_BYTES;
  static constexpr int SFB_OFF = SFA_OFF + kSfChunk;
  static constexpr int STAGE = ((SFB_OFF + 2 * kSfChunk) + 1023) / 1024 * 1024;
  static constexpr int STAGES = KIND == KIND_NVF4 ? 5 : 6;
  static constexpr int BAR_OFF = STAGES * STAGE;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;
  static constexpr uint32_t SF_COLS = 12u * KindK<KIND>::kChunksPerTile;   // SFA 4/chunk + SFB 8/chunk
  static constexpr uint32_t TX = A_BYTES + B_BYTES + 3 * kSfChunk;        // bytes one CTA lands per stage
  static_assert(BAR_OFF + 256 + 1024 <= 232448, "shared memory");
  static_assert(256 + STAGES * SF_COLS <= TMEM_COLS, "tensor memory");
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void remote_expect_tx(uint32_t cluster_bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void remote_arrive(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}
__device__ __forceinline__ void tc_cp_sf2(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
__device__ __forceinline__ void tc_commit2(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
template <int KIND>
__device__ __forceinline__ void tc_mma2(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
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

template <int KIND>
__global__ void __launch_bounds__(NTHREADS, 1)
    bs_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                        const GemmParams p) {
  using KK = KindK<KIND>;
  using L = Layout<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + L::BAR_OFF;
  const uint32_t bar_empty = bar_full + 8 * L::STAGES;
  const uint32_t bar_acc_full = bar_empty + 8 * L::STAGES;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR_OFF + 16 * L::STAGES + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 16 * L::STAGES + 24);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int n_blocks = (p.N + 255) / 256;
  const int n_tiles = ((p.M + 255) / 256) * n_blocks;
  const int num_kt = (p.K + KK::kElemsPerTile - 1) / KK::kElemsPerTile;
  const int nq = p.K / KK::kBlock / 4;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 2);    // one expect_tx arrival from each CTA's producer
      mbar_init(bar_empty + 8 * s, 1);   // the leader's multicast commit
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 8);         // every epilogue warp of both CTAs
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
  const uint32_t tmem = *tmem_slot;
  const uint32_t lead_full = mapa(bar_full, 0);
  const uint32_t lead_acc_empty = mapa(bar_acc_empty, 0);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer (both CTAs)
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
      uint32_t it = 0;
      for (int tile = pair; tile < n_tiles && !*abort_flag; tile += npairs) {
        const int m0 = (tile / n_blocks) * 256, n0 = (tile % n_blocks) * 256;
        for (int kt = 0; kt < num_kt; ++kt, ++it) {
          const int s = (int)(it % L::STAGES);
          const uint32_t ph = (it / L::STAGES) & 1u;
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag)) {
            *abort_flag = 1;
            raise_status(p.status, FP4Q_DEV_TIMEOUT);
            break;
          }
          const uint32_t st = sbase + (uint32_t)s * L::STAGE;
          const uint32_t fb = lead_full + 8 * s;
          const int q0 = kt * KK::kChunksPerTile;
          remote_expect_tx(fb, L::TX);
          tma_load_2d_pair(st, &tmA, kt * KROW, m0 + 128 * (int)rank, fb);
          tma_load_2d_pair(st + A_BYTES, &tmB, kt * KROW, n0 + 128 * (int)rank, fb);
          tma_load_2d_pair(st + L::SFA_OFF, &tmSA, 0, (m0 / 128 + (int)rank) * nq + q0, fb);
          tma_load_2d_pair(st + L::SFB_OFF, &tmSB, 0, (n0 / 128) * nq + q0, fb);
          tma_load_2d_pair(st + L::SFB_OFF + L::kSfChunk, &tmSB, 0, (n0 / 128 + 1) * nq + q0, fb);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader only)
      uint32_t it = 0, tl = 0;
      for (int tile = pair; tile < n_tiles; tile += npairs, ++tl) {
        if (!mbar_wait(bar_acc_empty, (tl & 1u) ^ 1u, abort_flag)) {
          *abort_flag = 1;
          raise_status(p.status, FP4Q_DEV_TIMEOUT);
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kt = 0; kt < num_kt; ++kt, ++it) {
          const int s = (int)(it % L::STAGES);
          const uint32_t ph = (it / L::STAGES) & 1u;
          if (!mbar_wait(bar_full + 8 * s, ph, abort_flag)) {
            *abort_flag = 1;
            raise_status(p.status, FP4Q_DEV_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + (uint32_t)s * L::STAGE;
          const uint32_t sfa_col = tmem + 256 + L::SF_COLS * (uint32_t)s;
          const uint32_t sfb_col = sfa_col + 4 * KK::kChunksPerTile;
          const int q0 = kt * KK::kChunksPerTile;
          const int nch = min(KK::kChunksPerTile, nq - q0);
          for (int c = 0; c < nch; ++c) {
            tc_cp_sf2(sfa_col + 4 * c, sf_desc(st + L::SFA_OFF + 512 * c));
            tc_cp_sf2(sfb_col + 8 * c, sf_desc(st + L::SFB_OFF + 512 * c));
            tc_cp_sf2(sfb_col + 8 * c + 4, sf_desc(st + L::SFB_OFF + L::kSfChunk + 512 * c));
          }
          const int rem = p.K - kt * KK::kElemsPerTile;
          const int n_mma = min(4, rem / KK::kMmaK);
          for (int k = 0; k < n_mma; ++k) {
            uint32_t sfa = sfa_col, sfb = sfb_col, sf_id = 0;
            if constexpr (KIND == KIND_MXF4) {
              sfa += 4 * (k >> 1);
              sfb += 8 * (k >> 1);
              sf_id = 2u * (uint32_t)(k & 1);
            } else if constexpr (KIND == KIND_NVF4) {
              sfa += 4 * k;
              sfb += 8 * k;
            } else {
              sf_id = (uint32_t)k;
            }
            tc_mma2<KIND>(tmem + ACC_COL, op_desc(st + 32 * k), op_desc(st + A_BYTES + 32 * k),
                          make_idesc<KIND, 256>(sf_id), sfa, sfb, (kt > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit2(bar_empty + 8 * s);
        }
        if (!ok) break;
        tc_commit2(bar_acc_full);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (both CTAs; warps 2..5 -> TMEM lane quarters 2, 3, 0, 1)
    const int sp = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * sp) << 16) + ACC_COL;
    float alpha = 1.0f;
    if constexpr (KIND == KIND_NVF4) alpha = __fmul_rn(*p.ts_a, *p.ts_b);
    uint32_t tl = 0;
    for (int tile = pair; tile < n_tiles; tile += npairs, ++tl) {
      const int m0 = (tile / n_blocks) * 256 + 128 * (int)rank, n0 = (tile % n_blocks) * 256;
      const int row = m0 + 32 * sp + lane;
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
      const int ncols = min(BN, p.N - n0);
      const bool live = m0 < p.M;   // the follower's rows of a 128-row tail tile lie outside the matrix
      if (p.d_f32 == nullptr) {
        uint32_t h[BN / 2];
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          if (c0 < ncols) {
            uint32_t r[32];
            tmem_ld32(lane_base + (uint32_t)c0, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
              if constexpr (KIND == KIND_NVF4) {
                a = __fmul_rn(a, alpha);
                b = __fmul_rn(b, alpha);
              }
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(a, b);
              h[c0 / 2 + j] = *reinterpret_cast<const uint32_t*>(&b2);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) remote_arrive(lead_acc_empty);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(p.d_bf16 + (size_t)row * p.N + n0);
#pragma unroll
          for (int j = 0; j < BN / 8; ++j)
            if (8 * j < ncols) dst[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
        }
      } else {
        for (int c0 = 0; c0 < ncols; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(lane_base + (uint32_t)c0, r);
          if (!live) continue;
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = __uint_as_float(r[j]);
            if constexpr (KIND == KIND_NVF4) v[j] = __fmul_rn(v[j], alpha);
          }
          const size_t off = (size_t)row * p.N + n0 + c0;
          float4* df = reinterpret_cast<float4*>(p.d_f32 + off);
#pragma unroll
          for (int j = 0; j < 8; ++j) df[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          if (p.d_bf16) {
            uint32_t hb[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
              hb[j] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            uint4* db = reinterpret_cast<uint4*>(p.d_bf16 + off);
#pragma unroll
            for (int j = 0; j < 4; ++j) db[j] = make_uint4(hb[4 * j], hb[4 * j + 1], hb[4 * j + 2], hb[4 * j + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) remote_arrive(lead_acc_empty);
      }
    }
  }
  // No CTA may leave while its peer can still read its shared memory or
  // tensor memory: meet, then free the pair's allocation together.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

}  // namespace pairk

// ------------------------------------------------------------ host side
// 2-D byte tensor [rows][row_bytes], box = 128 bytes x box_rows, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, row_bytes, rows, row_bytes, (uint32_t)KROW,
                        box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Scale factors in the MMA layout viewed as a 2-D u32 tensor: one row per
// 512-byte chunk (rows / 128 * blocks / 4 chunks), box = chunks of one K-tile.
bool make_sf_map(CUtensorMap* m, const void* base, uint64_t n_chunks, uint32_t box_chunks) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, base, 128u, n_chunks, 512u, 128u, box_chunks,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int KIND>
cudaError_t launch_gemm_pair(const fp4q_operand* A, const fp4q_operand* B, const void* a_data, const void* b_data,
                             uint64_t row_bytes, const GemmParams& p, cudaStream_t s) {
  using L = pairk::Layout<KIND>;
  CUtensorMap ta, tb, tsa, tsb;
  const uint64_t nq = (uint64_t)p.K / KindK<KIND>::kBlock / 4;
  if (!make_map(&ta, a_data, row_bytes, (uint64_t)p.M, 128) || !make_map(&tb, b_data, row_bytes, (uint64_t)p.N, 128) ||
      !make_sf_map(&tsa, A->scales, (uint64_t)p.M / 128 * nq, KindK<KIND>::kChunksPerTile) ||
      !make_sf_map(&tsb, B->scales, (uint64_t)p.N / 128 * nq, KindK<KIND>::kChunksPerTile))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(pairk::bs_gemm_pair_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int tiles = ((p.M + 255) / 256) * ((p.N + 255) / 256);
  int pairs = num_sms() / 2;
  if (tiles < pairs) pairs = tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pairk::bs_gemm_pair_kernel<KIND>, ta, tb, tsa, tsb, p);
}

template <int KIND>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bs_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int tiles = (p.M / BM) * ((p.N + BN - 1) / BN);
  const int g = tiles < num_sms() ? tiles : num_sms();
  bs_gemm_kernel<KIND><<<g, NTHREADS, SMEM_BYTES, s>>>(a, b, p);
  return cudaGetLastError();
}

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace fp4q

extern "C" int32_t fp4q_gemm(const fp4q_operand* A, const fp4q_operand* B, int64_t M, int64_t N, int64_t K,
                             int32_t grid, int32_t scale, void* D_bf16, float* D_f32, uint32_t* d_status,
                             void* stream) {
  using namespace fp4q;
  if (!A || !B || (!D_bf16 && !D_f32)) return FP4Q_ERR_INVALID_ARG;
  if (grid != FP4Q_GRID_E2M1 && grid != FP4Q_GRID_E1M2 && grid != FP4Q_GRID_E2M1_R4) return FP4Q_ERR_INVALID_ARG;
  if (scale != FP4Q_SCALE_MX && scale != FP4Q_SCALE_NV) return FP4Q_ERR_INVALID_ARG;
  if (grid == FP4Q_GRID_E1M2 && scale == FP4Q_SCALE_NV) return FP4Q_ERR_UNSUPPORTED;
  if (M <= 0 || N <= 0 || K <= 0) return FP4Q_ERR_INVALID_ARG;
  if (M % 128 || N % 128) return FP4Q_ERR_INVALID_ARG;
  if (K % (scale == FP4Q_SCALE_NV ? 64 : 128)) return FP4Q_ERR_INVALID_ARG;
  if (M / 128 > 65535 || M > (1LL << 31) || N > (1LL << 31) || K > (1LL << 31)) return FP4Q_ERR_INVALID_ARG;
  const int kind = grid == FP4Q_GRID_E1M2 ? KIND_F8 : (scale == FP4Q_SCALE_NV ? KIND_NVF4 : KIND_MXF4);
  const void* a_data = kind == KIND_F8 ? (const void*)A->e4m3 : (const void*)A->codes;
  const void* b_data = kind == KIND_F8 ? (const void*)B->e4m3 : (const void*)B->codes;
  if (!a_data || !b_data || !A->scales || !B->scales) return FP4Q_ERR_INVALID_ARG;
  if (kind == KIND_NVF4 && (!A->tensor_scale || !B->tensor_scale)) return FP4Q_ERR_INVALID_ARG;
  if (!al(a_data, 16) || !al(b_data, 16) || !al(A->scales, 16) || !al(B->scales, 16)) return FP4Q_ERR_ALIGNMENT;
  if ((D_bf16 && !al(D_bf16, 16)) || (D_f32 && !al(D_f32, 16))) return FP4Q_ERR_ALIGNMENT;
  const uint64_t row_bytes = kind == KIND_F8 ? (uint64_t)K : (uint64_t)K / 2;
  GemmParams p;
  p.sfa = A->scales;
  p.sfb = B->scales;
  p.ts_a = A->tensor_scale;
  p.ts_b = B->tensor_scale;
  p.d_bf16 = static_cast<uint16_t*>(D_bf16);
  p.d_f32 = D_f32;
  p.status = d_status;
  p.M = (int32_t)M;
  p.N = (int32_t)N;
  p.K = (int32_t)K;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
#if FP4Q_GEMM_PAIR
  if (kind == KIND_MXF4) e = launch_gemm_pair<KIND_MXF4>(A, B, a_data, b_data, row_bytes, p, s);
  else if (kind == KIND_NVF4) e = launch_gemm_pair<KIND_NVF4>(A, B, a_data, b_data, row_bytes, p, s);
  else e = launch_gemm_pair<KIND_F8>(A, B, a_data, b_data, row_bytes, p, s);
#else
  CUtensorMap ta, tb;
  if (!make_map(&ta, a_data, row_bytes, (uint64_t)M, BM) || !make_map(&tb, b_data, row_bytes, (uint64_t)N, BN))
    return FP4Q_ERR_CUDA;
  if (kind == KIND_MXF4) e = launch_gemm<KIND_MXF4>(ta, tb, p, s);
  else if (kind == KIND_NVF4) e = launch_gemm<KIND_NVF4>(ta, tb, p, s);
  else e = launch_gemm<KIND_F8>(ta, tb, p, s);
#endif
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}
