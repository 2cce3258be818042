// quant.cu -- fused blockwise Hadamard rotation + 4-bit microscaled quantizer
// for GB300 (sm_103a), and its companions: the rotated global-amax pass of the
// NVFP4-style recipe, the dequantizer and the unfused rotation arm.
//
// Method sources (web pages, by title and section):
//   [SB]  "Resumo Tecnico: Repensando o Vies de Encolhimento (Shrinkage Bias) no
//         Pre-treinamento de LLMs em FP4": Metodologia 1-2 (E2M1 vs uniform
//         E1M2 grid, RHT, SR on dY only), Eficiencia (RHT fused with FP4
//         quantization costs ~6-7% over quantization alone).
//   [MX]  "Resumo Tecnico: Pre-treinamento de ... com MXFP4": Metodologia 3
//         (deterministic H16/H32 rotations).
//   [HTX] HTX article on arXiv 2605.09825, "Que es MXFP4?" (32-element blocks,
//         E8M0 shared exponent, nearest 4-bit value).
//
// Design (GB300-first, HBM-bound):
//   * Persistent CTAs (three per SM for RTNE, two for stochastic rounding)
//     walk 32 x 256 bf16 tiles (16 KB).  Each tile is read once from HBM by
//     TMA into a shared-memory ring (128-byte swizzle) of two tiles (RTNE) or
//     three (SR): the depths measured fastest.  Every thread waits on the
//     tile's mbarrier itself and the CTA meets once per tile, before the
//     stage is refilled.  Both the row-wise copy (blocks along columns) and
//     the column-wise copy (blocks along rows, stored transposed) come from
//     that one read.
//   * A "chunk" is 32 consecutive elements of one row or one column.  A thread
//     holds a chunk as 16 fp32 pairs P[i] = (u[i], u[i+16]) so that every
//     butterfly stage of stride < 16 is one packed FADD2/FFMA2 over two
//     independent lanes; the two 16-element halves are also exactly the two
//     NV blocks.
//   * Scale, round and pack run in registers; codes leave as 16-byte stores.
//   * The butterfly order, the fp32 rounding of every step and the scale rules
//     are the library's definition of the method (they are what the tests hold
//     bit-exact against the CPU reference).
#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

#include "fp4q_dev.cuh"
#include "fp4q_internal.h"
#include "quant_core.cuh"

namespace fp4q {

#ifndef QUANT_STAGES
#define QUANT_STAGES 4       // tiles in flight per CTA (amax pass, rotation arm)
#endif
#ifndef QUANT_MIN_CTAS
#define QUANT_MIN_CTAS 3     // resident CTAs per SM the register budget is sized for
#endif
constexpr int kTR = 32;    // tile rows
constexpr int kTC = 256;   // tile columns
constexpr int kNT = 256;   // threads per CTA

// Store one quantized chunk of row `r` of a copy with `ncols` columns,
// starting at column c0 (multiple of 32).
template <int SCALE>
__device__ __forceinline__ void store_chunk(const CopyOut& d, int64_t r, int64_t c0, int64_t ncols,
                                            bool sf_mma, bool emit_e4m3, const ChunkOut& o) {
  uint4* cp = reinterpret_cast<uint4*>(d.codes + r * (ncols >> 1) + (c0 >> 1));
  *cp = make_uint4(o.w[0], o.w[1], o.w[2], o.w[3]);
  constexpr int B = (SCALE == FP4Q_SCALE_MX) ? 32 : 16;
  const int64_t nkb = ncols / B;
  const int64_t k = c0 / B;
  const int64_t off = sf_mma ? sf_mma_offset(r, k, nkb) : r * nkb + k;
  if constexpr (SCALE == FP4Q_SCALE_MX) {
    d.scales[off] = (uint8_t)o.sbytes;
  } else {
    *reinterpret_cast<uint16_t*>(d.scales + off) = (uint16_t)o.sbytes;
  }
  if (emit_e4m3) {
    uint4* ep = reinterpret_cast<uint4*>(d.e4m3 + r * ncols + c0);
    ep[0] = make_uint4(o.e4[0], o.e4[1], o.e4[2], o.e4[3]);
    ep[1] = make_uint4(o.e4[4], o.e4[5], o.e4[6], o.e4[7]);
  }
}

// ------------------------------------------------------------ tile pipeline
// Tiles of kTR x kTC bf16 arrive by TMA as four kTR-row x 64-column boxes
// with the 128-byte swizzle: within box b, logical row r occupies bytes
// [r*128, r*128+128) and its 16-byte unit c sits at unit c ^ (r & 7).  The
// thread <-> data mappings keep both access patterns conflict-free: eight
// threads of a quarter-warp read eight different rows of one row-wise chunk
// (distinct r & 7), and a warp reads 32 consecutive columns of one row.
constexpr int kStages = QUANT_STAGES;              // tiles in flight per CTA of the amax and rotation kernels
constexpr int kBoxBytes = kTR * 128;               // one 64-column box
constexpr int kTileBytes = kTR * kTC * 2;          // 16 KB
// tiles, alignment, barriers of a ring of `stages` tiles
constexpr int ring_smem(int stages) { return stages * kTileBytes + 1024 + 64; }
constexpr int kQuantSmem = ring_smem(kStages);

struct TileView {
  const uint8_t* t;
  // 16-byte unit u (0..31) of logical tile row r
  __device__ __forceinline__ uint4 unit(int r, int u) const {
    return *reinterpret_cast<const uint4*>(t + (u >> 3) * kBoxBytes + (r << 7) + (((u & 7) ^ (r & 7)) << 4));
  }
  // word holding columns 2p, 2p+1 of tile row r (p = 0..127)
  __device__ __forceinline__ uint32_t word(int r, int p) const {
    return *reinterpret_cast<const uint32_t*>(t + (p >> 5) * kBoxBytes + (r << 7) +
                                              ((((p >> 2) & 7) ^ (r & 7)) << 4) + ((p & 3) << 2));
  }
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool mbar_done(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for a phase of an mbarrier, giving up after limit_ns (about 2 s by
// default).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_done(bar, parity)) return true;
    if ((i & 255u) == 255u) {
      uint64_t now;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
      if (t0 == 0) t0 = now;
      else if (now - t0 > limit_ns) return false;
    }
  }
}

// Persistent walk over the tiles of the matrix: CTA b takes tiles b, b + G,
// b + 2G, ... (G = gridDim.x, column tiles fastest).  Thread 0 keeps kStages
// TMA tile loads in flight; every thread waits on the tile's mbarrier itself,
// computes, and all meet at one barrier per tile before the stage is refilled.  Used inline in each
// kernel so that the kernel parameters stay constant-bank operands.
template <int kStages>
struct TileRing {
  uint8_t* smem;
  uint32_t bar0;
  int ntc, ntiles;
  const CUtensorMap* tm;
  int stall_tile;          // bounded-wait test: CTA 0's tile that waits on bar_never
  uint64_t stall_limit_ns;

  __device__ __forceinline__ void issue(int s, int tile) const {
    const int tr0 = (tile / ntc) * kTR, tc0 = (tile % ntc) * kTC;
    const uint32_t bar = bar0 + 8 * s;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kTileBytes) : "memory");
#pragma unroll
    for (int b = 0; b < 4; ++b)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
          ::"r"(smem_addr(smem + s * kTileBytes + b * kBoxBytes)), "l"(tm), "r"(tc0 + 64 * b), "r"(tr0), "r"(bar)
          : "memory");
  }

  // The ring's barriers and the tensor map's prefetch: no global data is
  // touched, so a programmatic dependent may run this before its wait.
  __device__ __forceinline__ void setup(const CUtensorMap* tmap, int64_t rows, int64_t cols,
                                       int stall = -1, uint32_t stall_ns = 0) {
    extern __shared__ uint8_t smem_raw[];
    smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    bar0 = smem_addr(smem + kStages * kTileBytes);
    ntc = (int)((cols + kTC - 1) / kTC);
    ntiles = ntc * (int)((rows + kTR - 1) / kTR);
    tm = tmap;
    stall_tile = blockIdx.x == 0 ? stall : -1;
    stall_limit_ns = stall_ns;
    if (threadIdx.x == 0) {
      // kStages tile barriers, then one that nothing ever arrives at
      for (int s = 0; s <= kStages; ++s)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8 * s) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
    }
    __syncthreads();
  }
  // The first kStages loads.
  __device__ __forceinline__ void start() const {
    if (threadIdx.x == 0) {
      for (int s = 0; s < kStages; ++s) {
        const int t = blockIdx.x + s * gridDim.x;
        if (t < ntiles) issue(s, t);
      }
    }
  }
  __device__ __forceinline__ void init(const CUtensorMap* tmap, int64_t rows, int64_t cols,
                                      int stall = -1, uint32_t stall_ns = 0) {
    setup(tmap, rows, cols, stall, stall_ns);
    start();
  }

  __device__ __forceinline__ TileView view(int k) const { return TileView{smem + (k % kStages) * kTileBytes}; }

  // This thread's bounded wait for the k-th tile of this CTA (no CTA
  // barrier: every thread waits on the tile's mbarrier itself).
  __device__ __forceinline__ bool wait(int k) const {
    const int s = k % kStages;
    return k == stall_tile ? mbar_wait_bounded(bar0 + 8 * kStages, 0u, stall_limit_ns)
                           : mbar_wait_bounded(bar0 + 8 * s, (uint32_t)(k / kStages) & 1u);
  }

  // All threads are done with the k-th tile (ok: this thread saw it arrive):
  // the one CTA barrier of a tile, then thread 0 refills its stage.  Returns
  // false, after raising FP4Q_DEV_TIMEOUT and draining this CTA's own loads,
  // when any thread's wait ran out; every thread then leaves together.
  __device__ __forceinline__ bool release(int k, int tile, bool ok, uint32_t* status) const {
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        raise_status(status, FP4Q_DEV_TIMEOUT);
        for (int j = 0; j < kStages; ++j) {
          const int kk = k + j, tt = blockIdx.x + kk * gridDim.x;
          if (tt < ntiles) (void)mbar_wait_bounded(bar0 + 8 * (kk % kStages), (uint32_t)(kk / kStages) & 1u);
        }
      }
      __syncthreads();
      return false;
    }
    if (threadIdx.x == 0) {
      const int nt = tile + kStages * gridDim.x;
      if (nt < ntiles) issue(k % kStages, nt);
    }
    return true;
  }
};

// Row-wise chunk q (0..7) of tile row r as pairs with the signs applied.
__device__ __forceinline__ void read_row_chunk(const TileView& tv, int r, int q, const uint32_t* sgn,
                                               float2 (&P)[16]) {
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = tv.unit(r, 4 * q + j);
    w[4 * j + 0] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
  }
  // word k holds elements 2k (low half) and 2k+1 (high half)
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    P[2 * k].x = __uint_as_float(w[k] * 65536u + sgn[2 * k]);
    P[2 * k + 1].x = __uint_as_float((w[k] & 0xFFFF0000u) ^ sgn[2 * k + 1]);
    P[2 * k].y = __uint_as_float(w[k + 8] * 65536u + sgn[2 * k + 16]);
    P[2 * k + 1].y = __uint_as_float((w[k + 8] & 0xFFFF0000u) ^ sgn[2 * k + 17]);
  }
}

// Column c (0..255) of the tile's 32 rows as pairs with the signs applied.
// A word holds columns 2p (low half) and 2p+1 (high half); an integer multiply
// (by 65536 for the low half, by 1 for the high half) brings this thread's
// half to the top and the mask clears the rest.
__device__ __forceinline__ void read_col_chunk(const TileView& tv, int c, const uint32_t* sgn, float2 (&P)[16]) {
  const uint32_t mul = (c & 1) ? 1u : 65536u;   // brings this thread's half of a word to the top
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t a = tv.word(i, c >> 1), b = tv.word(i + 16, c >> 1);
    P[i].x = __uint_as_float(((a * mul) & 0xFFFF0000u) ^ sgn[i]);
    P[i].y = __uint_as_float(((b * mul) & 0xFFFF0000u) ^ sgn[i + 16]);
  }
}

// Row-wise task t (0..255) of a tile -> (row, chunk): eight consecutive tasks
// are eight rows with distinct r & 7 of one chunk.
__device__ __forceinline__ void row_task(int t, int& r, int& q) {
  r = (t & 7) | ((t >> 6) << 3);
  q = (t >> 3) & 7;
}

// ------------------------------------------------------------ fused kernel
// Per tile each thread quantizes one column chunk (32 rows of one column, the
// column-wise copy) and one row chunk (32 columns of one row, the row-wise
// copy).  Signs are applied to the packed bf16 words with one XOR per word
// (the sign words sw_row / sw_col of the kernel parameters) before the words
// are widened to fp32.

// Column c (0..255) of the tile's 32 rows as P[i] = (row i, row i + 16) with
// the column copy's signs applied: one XOR per word (the sign word carries the
// row's sign in both halves), then a byte permute with this thread's selector
// brings its half of the word to the top and clears the rest.  SIGNS = false
// (no rotation, all sign words zero) leaves the XORs out.
template <bool SIGNS>
__device__ __forceinline__ void read_col_chunk_sw(const TileView& tv, int c, const uint32_t* sw, float2 (&P)[16]) {
  const uint32_t sel = (c & 1) ? 0x3244u : 0x1044u;   // high half / low half to bits 16..31, zeros below
  const uint8_t* b = tv.t + (c >> 6) * kBoxBytes + (((c >> 1) & 3) << 2);
  const int x = (c >> 3) & 7;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint8_t* u = b + ((x ^ (i & 7)) << 4);   // rows i and i + 16 share the swizzle unit
    const uint32_t a = *reinterpret_cast<const uint32_t*>(u + (i << 7)) ^ (SIGNS ? sw[i] : 0u);
    const uint32_t d = *reinterpret_cast<const uint32_t*>(u + ((i + 16) << 7)) ^ (SIGNS ? sw[i + 16] : 0u);
    P[i] = make_float2(__uint_as_float(__byte_perm(a, 0u, sel)), __uint_as_float(__byte_perm(d, 0u, sel)));
  }
}

// Row-wise chunk q (0..7) of tile row r with the row copy's signs applied
// (none for SIGNS = false).
template <bool SIGNS>
__device__ __forceinline__ void read_row_chunk_sw(const TileView& tv, int r, int q, const uint32_t* sw,
                                                  float2 (&P)[16]) {
  const uint8_t* b = tv.t + (q >> 1) * kBoxBytes + (r << 7);
  const int y = ((q & 1) << 2) ^ (r & 7);
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = *reinterpret_cast<const uint4*>(b + ((y ^ j) << 4));
    w[4 * j + 0] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
  }
  // word k holds elements 2k (low half) and 2k+1 (high half)
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t a = w[k] ^ (SIGNS ? sw[k] : 0u), c = w[k + 8] ^ (SIGNS ? sw[k + 8] : 0u);
    P[2 * k] = make_float2(__uint_as_float(a << 16), __uint_as_float(c << 16));
    P[2 * k + 1] = make_float2(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(c & 0xFFFF0000u));
  }
}

// Resident CTAs per SM: stochastic rounding runs Philox and the exact
// round-up decision per element and does better with the register budget of
// two CTAs per SM; the other modes with three.
template <int ROUND>
constexpr int quant_ctas() { return ROUND == FP4Q_SR ? 2 : QUANT_MIN_CTAS; }
// Tiles in flight per CTA, measured on the linear-layer tensors (16384 x 4096
// both copies, CUDA events, L2 flushed): RTNE 60.1 / 61.1 / 62.1 us with
// 2 / 3 / 4 stages; SR on the E2M1 grid 133.8 / 131.7 / 133.8 us, on the E1M2
// and capped E2M1 grids 137.9 / 139.9 / 140.0 us.
template <int ROUND, int GRID>
constexpr int quant_stages() { return ROUND == FP4Q_SR && GRID == FP4Q_GRID_E2M1 ? 3 : 2; }

// Where one thread's chunks of a copy go: offsets that depend only on the
// thread (fixed over the tiles) plus, per tile, the tile's own.
struct ChunkDst {
  int64_t code, scale, e4;   // byte offsets of the thread's first chunk in the current tile
  int64_t code2, scale2, e42;   // the step to the thread's second chunk
};

// Scale, round, pack and store one chunk.
template <int GRID, int SCALE, int NH, int ROUND>
__device__ __forceinline__ void emit_chunk(float2 (&P)[16], const QuantParams& p, const CopyOut& d, float S_t,
                                           uint64_t idx0, uint32_t orient, int64_t code_off, int64_t scale_off,
                                           int64_t e4_off) {
  constexpr bool kMX = SCALE == FP4Q_SCALE_MX;
  ChunkOut o;
  if constexpr (kMX && ROUND == FP4Q_SR) {
    // the chunk's random words first: their chains overlap the rotation's
    Philox4 R[4];
    const uint64_t c = idx0 >> 3;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      R[q] = philox4x32_10_rk((uint32_t)(c + q), (uint32_t)((c + q) >> 32), orient, 0u, p.sr_keys);
    const float m = rotate_chunk_mx<NH>(P);
    quantize_chunk<GRID, SCALE, ROUND, true>(P, S_t, idx0, orient, p.sr_keys, p.emit_e4m3, p.status, o,
                                             NH == 16 ? 2 : 0, m, R);
  } else if constexpr (kMX) {
    // H16's 1/4 goes into the power-of-two block scale
    const float m = rotate_chunk_mx<NH>(P);
    quantize_chunk<GRID, SCALE, ROUND, true>(P, S_t, idx0, orient, p.sr_keys, p.emit_e4m3, p.status, o,
                                             NH == 16 ? 2 : 0, m);
  } else {
    rotate_chunk<NH>(P);
    quantize_chunk<GRID, SCALE, ROUND>(P, S_t, idx0, orient, p.sr_keys, p.emit_e4m3, p.status, o);
  }
  *reinterpret_cast<uint4*>(d.codes + code_off) = make_uint4(o.w[0], o.w[1], o.w[2], o.w[3]);
  if constexpr (kMX) d.scales[scale_off] = (uint8_t)o.sbytes;
  else *reinterpret_cast<uint16_t*>(d.scales + scale_off) = (uint16_t)o.sbytes;
  if (p.emit_e4m3) {
    uint4* ep = reinterpret_cast<uint4*>(d.e4m3 + e4_off);
    ep[0] = make_uint4(o.e4[0], o.e4[1], o.e4[2], o.e4[3]);
    ep[1] = make_uint4(o.e4[4], o.e4[5], o.e4[6], o.e4[7]);
  }
}

template <int GRID, int SCALE, int NH, int ROUND>
__global__ void __launch_bounds__(kNT, quant_ctas<ROUND>())
    rht_quant_kernel(const __grid_constant__ CUtensorMap tmx, const QuantParams p) {
  // Launched as a programmatic dependent of the stream's previous kernel: the
  // ring's setup touches only shared memory and the kernel parameters; then
  // wait for that grid to finish (its writes visible) before any global
  // memory access, and let the next kernel's launch begin.
  TileRing<quant_stages<ROUND, GRID>()> ring;
  ring.setup(&tmx, p.rows, p.cols, p.stall_tile, p.wait_limit_ns);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ring.start();
  constexpr float kDen = 448.0f * GridK<GRID>::kQmax;
  constexpr int B = SCALE == FP4Q_SCALE_MX ? 32 : 16;
  float S_row = 0.0f, S_col = 0.0f;
  if constexpr (SCALE == FP4Q_SCALE_NV) {
    if (p.want_row) S_row = __fdiv_rn(p.gamax[0], kDen);
    if (p.want_col) S_col = __fdiv_rn(p.gamax[1], kDen);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      if (p.want_row) *p.row.tensor_scale = S_row;
      if (p.want_col) *p.col.tensor_scale = S_col;
    }
  }

  // ---- offsets of this thread's chunks that do not change from tile to tile
  const int tid = threadIdx.x;
  int rr, rq;
  row_task(tid, rr, rq);
  int64_t c_code = 0, c_scale = 0, c_e4 = 0, r_code = 0, r_scale = 0, r_e4 = 0;
  if (p.want_col) {
    const int64_t nkb = p.rows / B;
    c_code = tid * (p.rows >> 1);
    c_e4 = tid * p.rows;
    c_scale = p.sf_mma ? (int64_t)(tid >> 7) * (nkb >> 2) * 512 + 16 * (tid & 31) + 4 * ((tid >> 5) & 3)
                       : tid * nkb;
  }
  if (p.want_row) {
    const int kq = rq * (32 / B);
    r_code = rr * (p.cols >> 1) + 16 * rq;
    r_e4 = rr * p.cols + 32 * rq;
    r_scale = p.sf_mma ? (int64_t)((kq >> 2) * 512 + 16 * rr + (kq & 3)) : rr * (p.cols / B) + kq;
  }

  // the tile's (row, column) position, stepped by the grid size without a division per tile
  int t_r = blockIdx.x / ring.ntc, t_c = blockIdx.x % ring.ntc;
  const int d_r = gridDim.x / ring.ntc, d_c = gridDim.x % ring.ntc;
  int k = 0;
  for (int tile = blockIdx.x; tile < ring.ntiles; tile += gridDim.x, ++k) {
    const bool arrived = ring.wait(k);
    const TileView tv = ring.view(k);
    const int64_t tr0 = (int64_t)t_r * kTR, tc0 = (int64_t)t_c * kTC;
    t_c += d_c;
    t_r += d_r;
    if (t_c >= ring.ntc) {
      t_c -= ring.ntc;
      ++t_r;
    }
    if (arrived && p.want_col) {
      const int64_t c = tc0 + tid;
      if (c < p.cols) {
        // column c is row c of the column copy; the chunk covers its elements tr0 .. tr0 + 31
        const int64_t nkb = p.rows / B, kb = tr0 / B;
        const int64_t code = tc0 * (p.rows >> 1) + (tr0 >> 1) + c_code;
        const int64_t e4 = tc0 * p.rows + tr0 + c_e4;
        const int64_t scale =
            (p.sf_mma ? (tc0 >> 7) * (nkb >> 2) * 512 + (kb >> 2) * 512 + (kb & 3) : tc0 * nkb + kb) + c_scale;
        float2 P[16];
        read_col_chunk_sw<(NH > 0)>(tv, tid, p.sw_col, P);
        emit_chunk<GRID, SCALE, NH, ROUND>(P, p, p.col, S_col, (uint64_t)(c * p.rows + tr0), 1u, code, scale, e4);
      }
    }
    if (arrived && p.want_row) {
      const int64_t gr = tr0 + rr, gc = tc0 + 32 * rq;
      if (gr < p.rows && gc < p.cols) {
        const int64_t nkb = p.cols / B, kb = tc0 / B;
        const int64_t code = tr0 * (p.cols >> 1) + (tc0 >> 1) + r_code;
        const int64_t e4 = tr0 * p.cols + tc0 + r_e4;
        const int64_t scale = (p.sf_mma ? ((tr0 >> 7) * (nkb >> 2) + (kb >> 2)) * 512 + 4 * ((tr0 >> 5) & 3)
                                        : tr0 * nkb + kb) + r_scale;
        float2 P[16];
        read_row_chunk_sw<(NH > 0)>(tv, rr, rq, p.sw_row, P);
        emit_chunk<GRID, SCALE, NH, ROUND>(P, p, p.row, S_row, (uint64_t)(gr * p.cols + gc), 0u, code, scale, e4);
      }
    }
    if (!ring.release(k, tile, arrived, p.status)) return;
  }
}

// ------------------------------------------------------------ amax pass
// G of the rotated row-wise and column-wise copies (NVFP4-style recipe):
// per-thread maxima over all tiles of the CTA, a CTA reduction, then one
// atomicMax on the float bits (non-negative floats order like their bit
// patterns).  amax[0..1] must hold 0 beforehand.
template <int NH>
__global__ void __launch_bounds__(kNT, QUANT_MIN_CTAS) rotated_amax_kernel(const __grid_constant__ CUtensorMap tmx,
                                                                           const QuantParams p, float* amax) {
  __shared__ float red[2][kNT / 32];
  float mrow = 0.0f, mcol = 0.0f;
  TileRing<kStages> ring;
  ring.init(&tmx, p.rows, p.cols);
  int k = 0;
  for (int tile = blockIdx.x; tile < ring.ntiles; tile += gridDim.x, ++k) {
    const bool arrived = ring.wait(k);
    const TileView tv = ring.view(k);
    // zero-filled padding contributes |0| and cannot raise the maximum
    if (arrived && p.want_col) {
      float2 P[16];
      read_col_chunk(tv, threadIdx.x, p.sgn_col, P);
      rotate_chunk<NH>(P);
#pragma unroll
      for (int i = 0; i < 16; ++i) mcol = absmax_nan(mcol, absmax_nan(P[i].x, P[i].y));
    }
    if (arrived && p.want_row) {
      int r, q;
      row_task(threadIdx.x, r, q);
      float2 P[16];
      read_row_chunk(tv, r, q, p.sgn_row, P);
      rotate_chunk<NH>(P);
#pragma unroll
      for (int i = 0; i < 16; ++i) mrow = absmax_nan(mrow, absmax_nan(P[i].x, P[i].y));
    }
    if (!ring.release(k, tile, arrived, p.status)) return;
  }
  mrow = fabsf(mrow);
  mcol = fabsf(mcol);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mrow = fabsf(absmax_nan(mrow, __shfl_xor_sync(0xFFFFFFFFu, mrow, o)));
    mcol = fabsf(absmax_nan(mcol, __shfl_xor_sync(0xFFFFFFFFu, mcol, o)));
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = mrow;
    red[1][threadIdx.x >> 5] = mcol;
  }
  __syncthreads();
  if (threadIdx.x < 2) {
    float m = 0.0f;
    for (int i = 0; i < kNT / 32; ++i) m = fabsf(absmax_nan(m, red[threadIdx.x][i]));
    if (__float_as_uint(m) >= 0x7F800000u) raise_status(p.status, FP4Q_DEV_NONFINITE);
    atomicMax(reinterpret_cast<unsigned int*>(amax) + threadIdx.x, __float_as_uint(m));
  }
}

// ------------------------------------------------------------ dequantize
// One thread per 32-element chunk of a stored copy (plain scale layout).
template <int GRID, int SCALE, int NH>
__global__ void __launch_bounds__(256) dequant_kernel(DequantParams d) {
  const int64_t nchunk_row = d.cols >> 5;
  const int64_t cid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (cid >= d.rows * nchunk_row) return;
  const int64_t r = cid / nchunk_row, c0 = (cid % nchunk_row) * 32;
  const uint4 cw = *reinterpret_cast<const uint4*>(d.codes + r * (d.cols >> 1) + (c0 >> 1));
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
  constexpr int B = (SCALE == FP4Q_SCALE_MX) ? 32 : 16;
  const int64_t nkb = d.cols / B;
  float step[2];
  if constexpr (SCALE == FP4Q_SCALE_MX) {
    const uint32_t sb = d.scales[r * nkb + c0 / B];
    // 2^(sb-127): normal for sb >= 1, 2^-127 (subnormal) at sb = 0
    const float s = sb ? __uint_as_float(sb << 23) : __uint_as_float(0x00400000u);
    step[0] = step[1] = s;
  } else {
    step[0] = e4m3_to_f32(d.scales[r * nkb + c0 / B]);
    step[1] = e4m3_to_f32(d.scales[r * nkb + c0 / B + 1]);
  }
  const float S_t = (SCALE == FP4Q_SCALE_NV) ? *d.tensor_scale : 1.0f;
  float v[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const uint32_t code = (w[t >> 3] >> (4 * (t & 7))) & 15u;
    const uint32_t k = code & 7u;
    float g;
    if constexpr (GRID == FP4Q_GRID_E1M2) {
      g = 0.25f * (float)k;
    } else {
      // E2M1 level k: 0, .5, 1, 1.5, 2, 3, 4, 6
      g = (k < 4) ? 0.5f * (float)k : (float)(1u << ((k >> 1) - 1)) * ((k & 1) ? 1.5f : 1.0f);
    }
    if (code & 8u) g = -g;
    float x = __fmul_rn(g, step[t >> 4 & (SCALE == FP4Q_SCALE_NV ? 1 : 0)]);
    if constexpr (SCALE == FP4Q_SCALE_NV) x = __fmul_rn(x, S_t);
    v[t] = x;
  }
  if constexpr (NH == 16 || NH == 32) {
    if (d.unrotate) {
      // inverse rotation: same butterfly and c_n, then the sign flips
#pragma unroll
      for (int b0 = 0; b0 < 32; b0 += NH) {
#pragma unroll
        for (int h = 1; h < NH; h <<= 1) {
#pragma unroll
          for (int i = 0; i < NH; ++i) {
            if (i & h) continue;
            const float a = v[b0 + i], b = v[b0 + i + h];
            v[b0 + i] = __fadd_rn(a, b);
            v[b0 + i + h] = __fsub_rn(a, b);
          }
        }
        const float c = (NH == 16) ? 0.25f : __uint_as_float(0x3E3504F3u);
#pragma unroll
        for (int i = 0; i < NH; ++i) v[b0 + i] = __fmul_rn(v[b0 + i], c);
      }
#pragma unroll
      for (int t = 0; t < 32; ++t)
        if ((d.sign_mask >> (t % NH)) & 1u) v[t] = -v[t];
    }
  }
  float4* out = reinterpret_cast<float4*>(d.out + r * d.cols + c0);
#pragma unroll
  for (int t = 0; t < 8; ++t) out[t] = make_float4(v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
}

// ------------------------------------------------------------ unfused arm
// Rotation only, written back in bf16 (RNE): the first kernel of the unfused
// rotate-then-quantize comparison.
template <int NH>
__global__ void __launch_bounds__(kNT, QUANT_MIN_CTAS) rotate_bf16_kernel(const __grid_constant__ CUtensorMap tmx,
                                                                          const QuantParams p, uint16_t* y_row,
                                                                          uint16_t* y_col) {
  TileRing<kStages> ring;
  ring.init(&tmx, p.rows, p.cols);
  int k = 0;
  for (int tile = blockIdx.x; tile < ring.ntiles; tile += gridDim.x, ++k) {
    const bool arrived = ring.wait(k);
    const TileView tv = ring.view(k);
    const int64_t tr0 = (int64_t)(tile / ring.ntc) * kTR, tc0 = (int64_t)(tile % ring.ntc) * kTC;
    if (arrived && y_col) {
      const int64_t c = tc0 + threadIdx.x;
      if (c < p.cols && tr0 < p.rows) {
        float2 P[16];
        read_col_chunk(tv, threadIdx.x, p.sgn_col, P);
        rotate_chunk<NH>(P);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          y_col[(tr0 + i) * p.cols + c] = (uint16_t)f32_to_bf16_rne(P[i].x);
          y_col[(tr0 + i + 16) * p.cols + c] = (uint16_t)f32_to_bf16_rne(P[i].y);
        }
      }
    }
    if (arrived && y_row) {
      int r, q;
      row_task(threadIdx.x, r, q);
      const int64_t gr = tr0 + r, gc = tc0 + 32 * q;
      if (gr < p.rows && gc < p.cols) {
        float2 P[16];
        read_row_chunk(tv, r, q, p.sgn_row, P);
        rotate_chunk<NH>(P);
        uint32_t o[16];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) {
          o[k2] = f32_to_bf16_rne(P[2 * k2].x) | (f32_to_bf16_rne(P[2 * k2 + 1].x) << 16);
          o[k2 + 8] = f32_to_bf16_rne(P[2 * k2].y) | (f32_to_bf16_rne(P[2 * k2 + 1].y) << 16);
        }
        uint4* dst = reinterpret_cast<uint4*>(y_row + gr * p.cols + gc);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
      }
    }
    if (!ring.release(k, tile, arrived, p.status)) return;
  }
}

// ------------------------------------------------------------ launchers
// The input's tensor map: bf16 [rows][cols] with row stride ld, boxes of kTR
// rows x 64 columns (kBoxBytes, one ring slot each), 128-byte swizzle, zero
// fill outside the matrix.
static bool input_map(const QuantParams& p, CUtensorMap* m) {
  static_assert(kTR * 64 * 2 == kBoxBytes, "a TMA box must fill exactly one ring slot");
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.x, (uint64_t)p.cols, (uint64_t)p.rows,
                        (uint64_t)p.ld * 2u, 64u, (uint32_t)kTR, CU_TENSOR_MAP_SWIZZLE_128B);
}

static unsigned persistent_grid(const QuantParams& p, int ctas_per_sm = QUANT_MIN_CTAS) {
  const int64_t ntiles = ((p.cols + kTC - 1) / kTC) * ((p.rows + kTR - 1) / kTR);
  const int64_t g = ctas_per_sm * (int64_t)num_sms();
  return (unsigned)(ntiles < g ? ntiles : g);
}

// Opt a kernel into the dynamic shared memory of the tile ring once.
template <class K>
static cudaError_t smem_attr(K kernel, bool& done, int smem = kQuantSmem) {
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) done = true;
  return e;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the stream's previous kernel finishes; it waits for that grid
// (griddepcontrol.wait) before touching global memory.
template <class K, class... Args>
static cudaError_t launch_dependent(K kernel, unsigned grid, int threads, int smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int GRID, int SCALE, int NH, int ROUND>
static cudaError_t launch_quant_inst(const CUtensorMap& m, const QuantParams& p, cudaStream_t s) {
  static bool attr = false;
  constexpr int smem = ring_smem(quant_stages<ROUND, GRID>());
  cudaError_t e = smem_attr(rht_quant_kernel<GRID, SCALE, NH, ROUND>, attr, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(rht_quant_kernel<GRID, SCALE, NH, ROUND>, persistent_grid(p, quant_ctas<ROUND>()), kNT,
                          smem, s, m, p);
}

template <int GRID, int SCALE, int NH>
static cudaError_t launch_quant_round(const CUtensorMap& m, const QuantParams& p, int round, cudaStream_t s) {
  return round == FP4Q_SR ? launch_quant_inst<GRID, SCALE, NH, FP4Q_SR>(m, p, s)
                          : launch_quant_inst<GRID, SCALE, NH, FP4Q_RTNE>(m, p, s);
}

template <int GRID, int SCALE>
static cudaError_t launch_quant_nh(const CUtensorMap& m, const QuantParams& p, int nh, int round, cudaStream_t s) {
  switch (nh) {
    case 16: return launch_quant_round<GRID, SCALE, 16>(m, p, round, s);
    case 32: return launch_quant_round<GRID, SCALE, 32>(m, p, round, s);
    default: return launch_quant_round<GRID, SCALE, 0>(m, p, round, s);
  }
}

cudaError_t launch_rht_quant(const QuantParams& p, int grid_kind, int scale, int nh, int round,
                             cudaStream_t s) {
  CUtensorMap m;
  if (!input_map(p, &m)) return cudaErrorInvalidValue;
  if (grid_kind == FP4Q_GRID_E2M1) {
    return scale == FP4Q_SCALE_NV ? launch_quant_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_NV>(m, p, nh, round, s)
                                  : launch_quant_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_MX>(m, p, nh, round, s);
  }
  if (grid_kind == FP4Q_GRID_E2M1_R4) {
    return scale == FP4Q_SCALE_NV ? launch_quant_nh<FP4Q_GRID_E2M1_R4, FP4Q_SCALE_NV>(m, p, nh, round, s)
                                  : launch_quant_nh<FP4Q_GRID_E2M1_R4, FP4Q_SCALE_MX>(m, p, nh, round, s);
  }
  return scale == FP4Q_SCALE_NV ? launch_quant_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_NV>(m, p, nh, round, s)
                                : launch_quant_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_MX>(m, p, nh, round, s);
}

template <int NH>
static cudaError_t launch_amax_inst(const CUtensorMap& m, const QuantParams& p, float* amax, cudaStream_t s) {
  static bool attr = false;
  cudaError_t e = smem_attr(rotated_amax_kernel<NH>, attr);
  if (e != cudaSuccess) return e;
  rotated_amax_kernel<NH><<<persistent_grid(p), kNT, kQuantSmem, s>>>(m, p, amax);
  return cudaGetLastError();
}

cudaError_t launch_rotated_amax(const QuantParams& p, int nh, float* amax, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax, 0, 2 * sizeof(float), s);
  if (e != cudaSuccess) return e;
  CUtensorMap m;
  if (!input_map(p, &m)) return cudaErrorInvalidValue;
  switch (nh) {
    case 16: return launch_amax_inst<16>(m, p, amax, s);
    case 32: return launch_amax_inst<32>(m, p, amax, s);
    default: return launch_amax_inst<0>(m, p, amax, s);
  }
}

template <int GRID, int SCALE>
static void launch_deq_nh(const DequantParams& d, int nh, unsigned nb, cudaStream_t s) {
  switch (nh) {
    case 16: dequant_kernel<GRID, SCALE, 16><<<nb, 256, 0, s>>>(d); break;
    case 32: dequant_kernel<GRID, SCALE, 32><<<nb, 256, 0, s>>>(d); break;
    default: dequant_kernel<GRID, SCALE, 0><<<nb, 256, 0, s>>>(d); break;
  }
}

cudaError_t launch_dequant(const DequantParams& d, int grid_kind, int scale, int nh, cudaStream_t s) {
  const int64_t nchunks = d.rows * (d.cols >> 5);
  const unsigned nb = (unsigned)((nchunks + 255) / 256);
  if (grid_kind != FP4Q_GRID_E1M2) {   // the capped grid decodes with the E2M1 table
    if (scale == FP4Q_SCALE_NV) launch_deq_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_NV>(d, nh, nb, s);
    else launch_deq_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_MX>(d, nh, nb, s);
  } else {
    if (scale == FP4Q_SCALE_NV) launch_deq_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_NV>(d, nh, nb, s);
    else launch_deq_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_MX>(d, nh, nb, s);
  }
  return cudaGetLastError();
}

template <int NH>
static cudaError_t launch_rot_inst(const CUtensorMap& m, const QuantParams& p, uint16_t* yr, uint16_t* yc,
                                   cudaStream_t s) {
  static bool attr = false;
  cudaError_t e = smem_attr(rotate_bf16_kernel<NH>, attr);
  if (e != cudaSuccess) return e;
  rotate_bf16_kernel<NH><<<persistent_grid(p), kNT, kQuantSmem, s>>>(m, p, yr, yc);
  return cudaGetLastError();
}

cudaError_t launch_rotate_bf16(const QuantParams& p, int nh, uint16_t* y_row, uint16_t* y_col, cudaStream_t s) {
  CUtensorMap m;
  if (!input_map(p, &m)) return cudaErrorInvalidValue;
  switch (nh) {
    case 16: return launch_rot_inst<16>(m, p, y_row, y_col, s);
    case 32: return launch_rot_inst<32>(m, p, y_row, y_col, s);
    default: return launch_rot_inst<0>(m, p, y_row, y_col, s);
  }
}

}  // namespace fp4q
