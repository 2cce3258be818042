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
//   * One CTA owns a 64 x 256 bf16 tile (32 KB), read once from HBM with
//     coalesced 16-byte loads into a bank-swizzled shared-memory tile.  Both
//     the row-wise copy (blocks along columns) and the column-wise copy (blocks
//     along rows, stored transposed) are produced from that one read.
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

namespace fp4q {

constexpr int kTR = 64;    // tile rows
constexpr int kTC = 256;   // tile columns
constexpr int kNT = 256;   // threads per CTA
constexpr int kUnitsPerRow = kTC * 2 / 16;  // 16-byte units per tile row (32)

// 16-byte unit u of a tile row is stored at u ^ ((u >> 3) & 3): row-wise chunk
// reads (8 threads on 8 chunks of one row) and column-pair reads (32 threads
// on one 128-byte span) are both free of bank conflicts.
__device__ __forceinline__ int swz(int u) { return u ^ ((u >> 3) & 3); }

template <int GRID>
struct GridK;
template <>
struct GridK<FP4Q_GRID_E2M1> {
  static constexpr float kQmax = 6.0f;
  static constexpr int kEmax = 2;
  static constexpr uint32_t kE4T0 = 0x3C383000u, kE4T1 = 0x4C484440u;  // E4M3 bytes of the 8 levels
};
template <>
struct GridK<FP4Q_GRID_E1M2> {
  static constexpr float kQmax = 1.75f;
  static constexpr int kEmax = 0;
  static constexpr uint32_t kE4T0 = 0x34302800u, kE4T1 = 0x3E3C3A38u;
};

// ------------------------------------------------------------ rounding
// RTNE onto {k/4}: clamp |v| to 1.75, then k = RNE(4|v|) read from the low
// mantissa bits of 4|v| + 2^23 (exact product, one rounding).
__device__ __forceinline__ uint32_t rtne_e1m2(float v) {
  const float a = fminf(fabsf(v), 1.75f);
  const float t = __fmaf_rn(a, 4.0f, 8388608.0f);
  return (__float_as_uint(t) & 7u) | ((__float_as_uint(v) >> 28) & 8u);
}

// SR onto {k/4}: s = 4|v| (exact), k0 = floor(s) by a round-down add of 2^23,
// frac = s - k0 (exact); up iff r16 < frac * 2^16.
__device__ __forceinline__ uint32_t sr_e1m2(float v, uint32_t r16) {
  const float s = fminf(fabsf(v), 1.75f) * 4.0f;
  float t;
  asm("add.rm.f32 %0, %1, %2;" : "=f"(t) : "f"(s), "f"(8388608.0f));
  const float fl = t - 8388608.0f;
  const float frac = s - fl;
  const uint32_t up = ((float)r16 < frac * 65536.0f) ? 1u : 0u;
  return ((__float_as_uint(t) & 7u) + up) | ((__float_as_uint(v) >> 28) & 8u);
}

// SR onto E2M1: with E = clamp(floor(log2 |v|), 0, 2) the levels around |v|
// are 2^(E-1) apart, s = |v| 2^(1-E) is exact, the lower level's code is
// 2E + floor(s) and frac(s) is the distance to it in gaps.
__device__ __forceinline__ uint32_t sr_e2m1(float v, uint32_t r16) {
  const float a = fminf(fabsf(v), 6.0f);
  int E = (int)(__float_as_uint(a) >> 23) - 127;
  E = E < 0 ? 0 : (E > 2 ? 2 : E);
  const float s = a * __uint_as_float((uint32_t)(128 - E) << 23);  // 2^(1-E)
  float t;
  asm("add.rm.f32 %0, %1, %2;" : "=f"(t) : "f"(s), "f"(8388608.0f));
  const float frac = s - (t - 8388608.0f);
  const uint32_t up = ((float)r16 < frac * 65536.0f) ? 1u : 0u;
  return ((uint32_t)(2 * E) + (__float_as_uint(t) & 3u) + up) | ((__float_as_uint(v) >> 28) & 8u);
}

// E4M3 bytes of eight packed codes (element 0 in the low nibble): magnitude by
// byte permutation of the level table, sign from bit 3 of each nibble.
template <int GRID>
__device__ __forceinline__ uint2 codes_to_e4m3(uint32_t w) {
  const uint32_t lo = __byte_perm(GridK<GRID>::kE4T0, GridK<GRID>::kE4T1, w & 0x7777u) |
                      __byte_perm(0u, 0x80808080u, (w >> 1) & 0x4444u);
  const uint32_t hw = w >> 16;
  const uint32_t hi = __byte_perm(GridK<GRID>::kE4T0, GridK<GRID>::kE4T1, hw & 0x7777u) |
                      __byte_perm(0u, 0x80808080u, (hw >> 1) & 0x4444u);
  return make_uint2(lo, hi);
}

// ------------------------------------------------------------ one chunk
// Rotation of a chunk held as P[i] = (u[i], u[i+16]) (signs already applied).
template <int NH>
__device__ __forceinline__ void rotate_chunk(float2 (&P)[16]) {
  if constexpr (NH == 16 || NH == 32) {
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i & h) continue;
        const float2 a = P[i], b = P[i + h];
        P[i] = add2(a, b);
        P[i + h] = sub2(a, b);
      }
    }
    if constexpr (NH == 32) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = P[i].x, b = P[i].y;
        P[i].x = __fadd_rn(a, b);
        P[i].y = __fsub_rn(a, b);
      }
    }
    const float c = (NH == 16) ? 0.25f : __uint_as_float(0x3E3504F3u);  // fl32(1/sqrt(32))
#pragma unroll
    for (int i = 0; i < 16; ++i) P[i] = mul2(P[i], make_float2(c, c));
  }
}

struct ChunkOut {
  uint32_t w[4];     // 32 packed codes
  uint32_t sbytes;   // MX: 1 byte; NV: 2 bytes (block of lanes .x, block of lanes .y)
  uint32_t e4[8];    // optional E4M3 bytes
};

// Scale, round and pack one rotated chunk.
//   S_t    NV tensor scale (ignored for MX)
//   idx0   index of element 0 in the stored copy (multiple of 32), for SR
template <int GRID, int SCALE, int ROUND>
__device__ __forceinline__ void quantize_chunk(float2 (&P)[16], float S_t, uint64_t idx0,
                                               uint32_t orient, uint32_t key0, uint32_t key1,
                                               bool emit_e4m3, uint32_t* status, ChunkOut& o) {
  constexpr float QMAX = GridK<GRID>::kQmax;
  // block amax (NaN-propagating)
  float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    m0 = absmax_nan(m0, P[i].x);
    m1 = absmax_nan(m1, P[i].y);
  }
  m0 = fabsf(m0);
  m1 = fabsf(m1);
  float2 vm;
  if constexpr (SCALE == FP4Q_SCALE_MX) {
    const float m = fabsf(absmax_nan(m0, m1));
    const uint32_t mb = __float_as_uint(m);
    if (mb >= 0x7F800000u) raise_status(status, FP4Q_DEV_NONFINITE);
    int sb = (int)(mb >> 23) - GridK<GRID>::kEmax;   // floor(log2 m) - e_max + 127, 0 for m = 0
    sb = sb < 0 ? 0 : (sb > 254 ? 254 : sb);
    // 2^-e = 2^(127 - sb): exponent field 254 - sb, or 2^-127 (subnormal) at sb = 254
    const float mul = (sb < 254) ? __uint_as_float((uint32_t)(254 - sb) << 23) : __uint_as_float(0x00400000u);
    vm = make_float2(mul, mul);
    o.sbytes = (uint32_t)sb;
  } else {
    if (__float_as_uint(m0) >= 0x7F800000u || __float_as_uint(m1) >= 0x7F800000u)
      raise_status(status, FP4Q_DEV_NONFINITE);
    uint32_t s0 = 0, s1 = 0;
    float r0 = 0.0f, r1 = 0.0f;
    if (S_t > 0.0f) {
      s0 = cvt_e4m3(__fdiv_rn(__fdiv_rn(m0, QMAX), S_t));
      s1 = cvt_e4m3(__fdiv_rn(__fdiv_rn(m1, QMAX), S_t));
      if (s0) {
        r0 = __frcp_rn(__fmul_rn(e4m3_to_f32(s0), S_t));
        if (isinf(r0)) r0 = FLT_MAX;
      }
      if (s1) {
        r1 = __frcp_rn(__fmul_rn(e4m3_to_f32(s1), S_t));
        if (isinf(r1)) r1 = FLT_MAX;
      }
    }
    vm = make_float2(r0, r1);   // a zero multiplier leaves sign|0 codes
    o.sbytes = s0 | (s1 << 8);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) P[i] = mul2(P[i], vm);

  if constexpr (ROUND == FP4Q_RTNE && GRID == FP4Q_GRID_E2M1) {
    o.w[0] = cvt_e2m1x8(P[0].x, P[1].x, P[2].x, P[3].x, P[4].x, P[5].x, P[6].x, P[7].x);
    o.w[1] = cvt_e2m1x8(P[8].x, P[9].x, P[10].x, P[11].x, P[12].x, P[13].x, P[14].x, P[15].x);
    o.w[2] = cvt_e2m1x8(P[0].y, P[1].y, P[2].y, P[3].y, P[4].y, P[5].y, P[6].y, P[7].y);
    o.w[3] = cvt_e2m1x8(P[8].y, P[9].y, P[10].y, P[11].y, P[12].y, P[13].y, P[14].y, P[15].y);
  } else if constexpr (ROUND == FP4Q_RTNE) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = (q & 1) * 8 + j;
        const float v = (q < 2) ? P[i].x : P[i].y;
        w |= rtne_e1m2(v) << (4 * j);
      }
      o.w[q] = w;
    }
  } else {
    // stochastic rounding: element t of the chunk takes half (t & 1) of word
    // (t >> 1) & 3 of Philox call t >> 3, counter (idx >> 3) of the copy.
    const uint64_t c = idx0 >> 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t cq = c + (uint64_t)q;
      const Philox4 r = philox4x32_10((uint32_t)cq, (uint32_t)(cq >> 32), orient, 0u, key0, key1);
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = q * 8 + j;
        const float v = (t < 16) ? P[t].x : P[t - 16].y;
        const uint32_t r16 = (j & 1) ? (r.v[j >> 1] >> 16) : (r.v[j >> 1] & 0xFFFFu);
        const uint32_t code = (GRID == FP4Q_GRID_E1M2) ? sr_e1m2(v, r16) : sr_e2m1(v, r16);
        w |= code << (4 * j);
      }
      o.w[q] = w;
    }
  }
  if (emit_e4m3) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint2 e = codes_to_e4m3<GRID>(o.w[q]);
      o.e4[2 * q] = e.x;
      o.e4[2 * q + 1] = e.y;
    }
  }
}

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

// ------------------------------------------------------------ tile loading
// Load the kTR x kTC tile at (tr0, tc0) into shared memory; rows or 8-column
// units outside the matrix read as zero.
__device__ __forceinline__ void load_tile(uint4* tile, const uint16_t* __restrict__ x, int64_t rows,
                                          int64_t cols, int64_t ld, int64_t tr0, int64_t tc0) {
#pragma unroll
  for (int k = 0; k < (kTR * kUnitsPerRow) / kNT; ++k) {
    const int id = threadIdx.x + kNT * k;
    const int r = id / kUnitsPerRow, u = id % kUnitsPerRow;
    const int64_t gr = tr0 + r, gc = tc0 + (int64_t)u * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (gr < rows && gc < cols) v = __ldcs(reinterpret_cast<const uint4*>(x + gr * ld + gc));
    tile[r * kUnitsPerRow + swz(u)] = v;
  }
}

// Chunk of tile row r, 32-column chunk q (0..7), as pairs with signs applied.
__device__ __forceinline__ void read_row_chunk(const uint4* tile, int r, int q, const uint32_t* sgn,
                                               float2 (&P)[16]) {
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = tile[r * kUnitsPerRow + swz(4 * q + j)];
    w[4 * j + 0] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
  }
  // word k holds elements 2k (low half) and 2k+1 (high half)
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    P[2 * k].x = __uint_as_float((w[k] << 16) ^ sgn[2 * k]);
    P[2 * k + 1].x = __uint_as_float((w[k] & 0xFFFF0000u) ^ sgn[2 * k + 1]);
    P[2 * k].y = __uint_as_float((w[k + 8] << 16) ^ sgn[2 * k + 16]);
    P[2 * k + 1].y = __uint_as_float((w[k + 8] & 0xFFFF0000u) ^ sgn[2 * k + 17]);
  }
}

// Word (bf16 pair of columns 2p, 2p+1) of tile row r.
__device__ __forceinline__ uint32_t tile_word(const uint4* tile, int r, int p) {
  const uint32_t* row = reinterpret_cast<const uint32_t*>(tile + r * kUnitsPerRow);
  return row[swz(p >> 2) * 4 + (p & 3)];
}

// ------------------------------------------------------------ fused kernel
template <int GRID, int SCALE, int NH, int ROUND>
__global__ void __launch_bounds__(kNT, 2) rht_quant_kernel(const QuantParams p) {
  __shared__ uint4 tile[kTR * kUnitsPerRow];
  const int64_t tr0 = (int64_t)blockIdx.y * kTR, tc0 = (int64_t)blockIdx.x * kTC;
  load_tile(tile, p.x, p.rows, p.cols, p.ld, tr0, tc0);
  __syncthreads();

  const uint32_t key0 = (uint32_t)p.sr_seed, key1 = (uint32_t)(p.sr_seed >> 32);
  constexpr float kDen = 448.0f * GridK<GRID>::kQmax;

  // column-wise copy: thread owns columns 2cp, 2cp+1 of rows 32h .. 32h+31
  if (p.want_col) {
    float S_t = 0.0f;
    if constexpr (SCALE == FP4Q_SCALE_NV) {
      S_t = __fdiv_rn(p.gamax[1], kDen);
      if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.col.tensor_scale = S_t;
    }
    const int cp = threadIdx.x & 127, h = threadIdx.x >> 7;
    const int64_t col = tc0 + 2 * cp, row0 = tr0 + 32 * h;
    if (col < p.cols && row0 < p.rows) {
      uint32_t w[32];
#pragma unroll
      for (int t = 0; t < 32; ++t) w[t] = tile_word(tile, 32 * h + t, cp);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float2 P[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t a = half ? (w[i] & 0xFFFF0000u) : (w[i] << 16);
          const uint32_t b = half ? (w[i + 16] & 0xFFFF0000u) : (w[i + 16] << 16);
          P[i].x = __uint_as_float(a ^ p.sgn_col[i]);
          P[i].y = __uint_as_float(b ^ p.sgn_col[i + 16]);
        }
        rotate_chunk<NH>(P);
        const int64_t c = col + half;
        ChunkOut o;
        quantize_chunk<GRID, SCALE, ROUND>(P, S_t, (uint64_t)(c * p.rows + row0), 1u, key0, key1,
                                           p.emit_e4m3, p.status, o);
        store_chunk<SCALE>(p.col, c, row0, p.rows, p.sf_mma, p.emit_e4m3, o);
      }
    }
  }

  // row-wise copy: tasks (row r, chunk q), 8 consecutive threads per row
  if (p.want_row) {
    float S_t = 0.0f;
    if constexpr (SCALE == FP4Q_SCALE_NV) {
      S_t = __fdiv_rn(p.gamax[0], kDen);
      if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.row.tensor_scale = S_t;
    }
#pragma unroll 1
    for (int k = 0; k < (kTR * (kTC / 32)) / kNT; ++k) {
      const int id = threadIdx.x + kNT * k;
      const int r = id >> 3, q = id & 7;
      const int64_t gr = tr0 + r, gc = tc0 + 32 * q;
      if (gr < p.rows && gc < p.cols) {
        float2 P[16];
        read_row_chunk(tile, r, q, p.sgn_row, P);
        rotate_chunk<NH>(P);
        ChunkOut o;
        quantize_chunk<GRID, SCALE, ROUND>(P, S_t, (uint64_t)(gr * p.cols + gc), 0u, key0, key1,
                                           p.emit_e4m3, p.status, o);
        store_chunk<SCALE>(p.row, gr, gc, p.cols, p.sf_mma, p.emit_e4m3, o);
      }
    }
  }
}

// ------------------------------------------------------------ amax pass
// G of the rotated row-wise and column-wise copies (NVFP4-style recipe):
// per-CTA maxima, then one atomicMax on the float bits (non-negative floats
// order like their bit patterns).  amax[0..1] must hold 0 beforehand.
template <int NH>
__global__ void __launch_bounds__(kNT) rotated_amax_kernel(const QuantParams p, float* amax) {
  __shared__ uint4 tile[kTR * kUnitsPerRow];
  __shared__ float red[2][kNT / 32];
  const int64_t tr0 = (int64_t)blockIdx.y * kTR, tc0 = (int64_t)blockIdx.x * kTC;
  load_tile(tile, p.x, p.rows, p.cols, p.ld, tr0, tc0);
  __syncthreads();
  float mrow = 0.0f, mcol = 0.0f;
  if (p.want_col) {
    const int cp = threadIdx.x & 127, h = threadIdx.x >> 7;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      float2 P[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t wa = tile_word(tile, 32 * h + i, cp), wb = tile_word(tile, 32 * h + i + 16, cp);
        P[i].x = __uint_as_float((half ? (wa & 0xFFFF0000u) : (wa << 16)) ^ p.sgn_col[i]);
        P[i].y = __uint_as_float((half ? (wb & 0xFFFF0000u) : (wb << 16)) ^ p.sgn_col[i + 16]);
      }
      rotate_chunk<NH>(P);
#pragma unroll
      for (int i = 0; i < 16; ++i) mcol = absmax_nan(mcol, absmax_nan(P[i].x, P[i].y));
    }
  }
  if (p.want_row) {
#pragma unroll 1
    for (int k = 0; k < (kTR * (kTC / 32)) / kNT; ++k) {
      const int id = threadIdx.x + kNT * k;
      float2 P[16];
      read_row_chunk(tile, id >> 3, id & 7, p.sgn_row, P);
      rotate_chunk<NH>(P);
#pragma unroll
      for (int i = 0; i < 16; ++i) mrow = absmax_nan(mrow, absmax_nan(P[i].x, P[i].y));
    }
  }
  // (zero-filled padding contributes |0| and cannot raise the maximum)
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
__global__ void __launch_bounds__(kNT) rotate_bf16_kernel(const QuantParams p, uint16_t* y_row, uint16_t* y_col) {
  __shared__ uint4 tile[kTR * kUnitsPerRow];
  const int64_t tr0 = (int64_t)blockIdx.y * kTR, tc0 = (int64_t)blockIdx.x * kTC;
  load_tile(tile, p.x, p.rows, p.cols, p.ld, tr0, tc0);
  __syncthreads();
  if (y_col) {
    const int cp = threadIdx.x & 127, h = threadIdx.x >> 7;
    const int64_t col = tc0 + 2 * cp, row0 = tr0 + 32 * h;
    if (col < p.cols && row0 < p.rows) {
      float2 Pa[16], Pb[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t wa = tile_word(tile, 32 * h + i, cp), wb = tile_word(tile, 32 * h + i + 16, cp);
        Pa[i].x = __uint_as_float((wa << 16) ^ p.sgn_col[i]);
        Pa[i].y = __uint_as_float((wb << 16) ^ p.sgn_col[i + 16]);
        Pb[i].x = __uint_as_float((wa & 0xFFFF0000u) ^ p.sgn_col[i]);
        Pb[i].y = __uint_as_float((wb & 0xFFFF0000u) ^ p.sgn_col[i + 16]);
      }
      rotate_chunk<NH>(Pa);
      rotate_chunk<NH>(Pb);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint32_t* o0 = reinterpret_cast<uint32_t*>(y_col + (row0 + i) * p.cols + col);
        uint32_t* o1 = reinterpret_cast<uint32_t*>(y_col + (row0 + i + 16) * p.cols + col);
        *o0 = f32_to_bf16_rne(Pa[i].x) | (f32_to_bf16_rne(Pb[i].x) << 16);
        *o1 = f32_to_bf16_rne(Pa[i].y) | (f32_to_bf16_rne(Pb[i].y) << 16);
      }
    }
  }
  if (y_row) {
#pragma unroll 1
    for (int k = 0; k < (kTR * (kTC / 32)) / kNT; ++k) {
      const int id = threadIdx.x + kNT * k;
      const int r = id >> 3, q = id & 7;
      const int64_t gr = tr0 + r, gc = tc0 + 32 * q;
      if (gr < p.rows && gc < p.cols) {
        float2 P[16];
        read_row_chunk(tile, r, q, p.sgn_row, P);
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
  }
}

// ------------------------------------------------------------ launchers
template <int GRID, int SCALE, int NH>
static cudaError_t launch_quant_round(const QuantParams& p, int round, dim3 grid, cudaStream_t s) {
  if (round == FP4Q_SR)
    rht_quant_kernel<GRID, SCALE, NH, FP4Q_SR><<<grid, kNT, 0, s>>>(p);
  else
    rht_quant_kernel<GRID, SCALE, NH, FP4Q_RTNE><<<grid, kNT, 0, s>>>(p);
  return cudaGetLastError();
}

template <int GRID, int SCALE>
static cudaError_t launch_quant_nh(const QuantParams& p, int nh, int round, dim3 grid, cudaStream_t s) {
  switch (nh) {
    case 16: return launch_quant_round<GRID, SCALE, 16>(p, round, grid, s);
    case 32: return launch_quant_round<GRID, SCALE, 32>(p, round, grid, s);
    default: return launch_quant_round<GRID, SCALE, 0>(p, round, grid, s);
  }
}

static dim3 tile_grid(int64_t rows, int64_t cols) {
  return dim3((unsigned)((cols + kTC - 1) / kTC), (unsigned)((rows + kTR - 1) / kTR), 1);
}

cudaError_t launch_rht_quant(const QuantParams& p, int grid_kind, int scale, int nh, int round,
                             cudaStream_t s) {
  const dim3 g = tile_grid(p.rows, p.cols);
  if (grid_kind == FP4Q_GRID_E2M1) {
    return scale == FP4Q_SCALE_NV ? launch_quant_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_NV>(p, nh, round, g, s)
                                  : launch_quant_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_MX>(p, nh, round, g, s);
  }
  return scale == FP4Q_SCALE_NV ? launch_quant_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_NV>(p, nh, round, g, s)
                                : launch_quant_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_MX>(p, nh, round, g, s);
}

cudaError_t launch_rotated_amax(const QuantParams& p, int nh, float* amax, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax, 0, 2 * sizeof(float), s);
  if (e != cudaSuccess) return e;
  const dim3 g = tile_grid(p.rows, p.cols);
  switch (nh) {
    case 16: rotated_amax_kernel<16><<<g, kNT, 0, s>>>(p, amax); break;
    case 32: rotated_amax_kernel<32><<<g, kNT, 0, s>>>(p, amax); break;
    default: rotated_amax_kernel<0><<<g, kNT, 0, s>>>(p, amax); break;
  }
  return cudaGetLastError();
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
  if (grid_kind == FP4Q_GRID_E2M1) {
    if (scale == FP4Q_SCALE_NV) launch_deq_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_NV>(d, nh, nb, s);
    else launch_deq_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_MX>(d, nh, nb, s);
  } else {
    if (scale == FP4Q_SCALE_NV) launch_deq_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_NV>(d, nh, nb, s);
    else launch_deq_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_MX>(d, nh, nb, s);
  }
  return cudaGetLastError();
}

cudaError_t launch_rotate_bf16(const QuantParams& p, int nh, uint16_t* y_row, uint16_t* y_col, cudaStream_t s) {
  const dim3 g = tile_grid(p.rows, p.cols);
  switch (nh) {
    case 16: rotate_bf16_kernel<16><<<g, kNT, 0, s>>>(p, y_row, y_col); break;
    case 32: rotate_bf16_kernel<32><<<g, kNT, 0, s>>>(p, y_row, y_col); break;
    default: rotate_bf16_kernel<0><<<g, kNT, 0, s>>>(p, y_row, y_col); break;
  }
  return cudaGetLastError();
}

}  // namespace fp4q
