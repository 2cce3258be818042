// diag.cu -- two diagnostics of a quantized copy, beside the bias statistics:
//
//  * the rounding error in grid units per level: for every element of a
//    row-wise copy, its position v = y * step^-1 on the grid (y the rotated
//    value, the step exactly as the quantizer takes it) and its code's level
//    g[k]; per level k the sum of g[k] - |v| and the count ("Repensando o Vies
//    de Encolhimento", Metodologia 1, "Origem Geometrica": elements rounded to
//    q_i err by (l_i - r_i)/2 on average, negative where the level's bin is
//    wider above it than below, the source of the magnitude shrinkage);
//  * the per-element mean signed relative error (|approx| - |ref|) / |ref|
//    over ref != 0, the per-element form of the shrinkage that the tiny
//    workload's report asks for beside the aggregate.
//
// Both are streaming reductions with fp64 sums: a grid of four CTAs per SM
// (at most kDiagMaxBlocks), a fixed-order reduction inside each CTA, per-CTA
// partials in a caller workspace and a final sum in CTA order by the last CTA
// to finish, so results are bit-reproducible on a given device.
#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>
#include <string.h>

#include "../../include/fp4q.h"
#include "fp4q_dev.cuh"
#include "fp4q_internal.h"
#include "quant_core.cuh"

namespace fp4q {
namespace {

constexpr int kDiagThreads = 256;
constexpr int kDiagMaxBlocks = 640;
constexpr int kDiagMaxVals = 16;   // values reduced per call (grid error: 8 sums + 8 counts)

size_t diag_workspace() { return (size_t)kDiagMaxBlocks * kDiagMaxVals * 8 + 256; }

__device__ __forceinline__ void put_words(uint32_t* w, uint4 v) {
  w[0] = v.x;
  w[1] = v.y;
  w[2] = v.z;
  w[3] = v.w;
}

// Magnitude of level k (0..7): E2M1 {0, .5, 1, 1.5, 2, 3, 4, 6}, E1M2 {k/4}.
template <int GRID>
__device__ __forceinline__ float grid_level(uint32_t k) {
  if constexpr (GRID == FP4Q_GRID_E1M2) return 0.25f * (float)k;
  else return k < 4 ? 0.5f * (float)k : (float)(1u << ((k >> 1) - 1)) * ((k & 1) ? 1.5f : 1.0f);
}

int diag_blocks(int64_t work_items) {
  const int64_t want = (work_items + kDiagThreads - 1) / kDiagThreads;
  int b = 4 * num_sms();
  if (b > kDiagMaxBlocks) b = kDiagMaxBlocks;
  if (want < b) b = (int)(want > 0 ? want : 1);
  return b;
}

// Deterministic reduction of NV per-thread doubles: warp butterfly, warps in
// order, per-CTA partials, and the last CTA sums the partials in CTA order
// into out[0 .. NV).  The arrival counter (after the partials) is zeroed by
// the host before the launch and again by the last CTA.
template <int NV>
__device__ void reduce_to(double (&v)[NV], void* workspace, double* out) {
  __shared__ double red[NV][kDiagThreads / 32];
  __shared__ bool last;
  double* part = reinterpret_cast<double*>(workspace);
  unsigned int* counter = reinterpret_cast<unsigned int*>(part + kDiagMaxBlocks * kDiagMaxVals);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    double s = v[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if ((threadIdx.x & 31) == 0) red[k][threadIdx.x >> 5] = s;
  }
  __syncthreads();
  if (threadIdx.x < NV) {
    double s = 0;
    for (int w = 0; w < kDiagThreads / 32; ++w) s += red[threadIdx.x][w];
    part[blockIdx.x * kDiagMaxVals + threadIdx.x] = s;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(counter, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x < NV) {
    double s = 0;
    for (int b = 0; b < (int)gridDim.x; ++b) s += ((volatile double*)part)[b * kDiagMaxVals + threadIdx.x];
    out[threadIdx.x] = s;
  }
  if (threadIdx.x == 0) *counter = 0u;
}

struct GridErrParams {
  const uint16_t* x;
  int64_t rows, cols, ld;
  const uint8_t* codes;
  const uint8_t* scales;
  const float* tensor_scale;
  int32_t sf_mma;
  uint32_t sgn[32];   // sign words of a 32-element chunk (bit 31 = negate)
  void* workspace;
  double* out;        // 8 sums, then 8 counts (as doubles; the host converts)
};

// One thread per 32-element chunk of the row-wise copy, grid-stride.
template <int GRID, int SCALE, int NH>
__global__ void __launch_bounds__(kDiagThreads) grid_error_kernel(const GridErrParams p) {
  double acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.0;
  const int64_t cpr = p.cols >> 5;   // chunks per row
  const int64_t nchunks = p.rows * cpr;
  for (int64_t ci = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; ci < nchunks;
       ci += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = ci / cpr, c0 = (ci % cpr) * 32;
    const uint4* src = reinterpret_cast<const uint4*>(p.x + r * p.ld + c0);
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) put_words(w + 4 * j, src[j]);
    float2 P[16];
    chunk_from_bf16_words(w, p.sgn, P);
    rotate_chunk<NH, true>(P);   // y, with the rotation's own final multiply
    const uint4 cw = *reinterpret_cast<const uint4*>(p.codes + r * (p.cols >> 1) + (c0 >> 1));
    const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
    float mul0, mul1;
    if constexpr (SCALE == FP4Q_SCALE_MX) {
      const int64_t nkb = p.cols >> 5, k = c0 >> 5;
      const uint32_t sb = p.scales[p.sf_mma ? sf_mma_offset(r, k, nkb) : r * nkb + k];
      // 2^(127 - sb): exponent field 254 - sb, or the subnormal 2^-127 for sb = 254
      const int z = 254 - (int)sb;
      mul0 = mul1 = z >= 1 ? __uint_as_float((uint32_t)z << 23) : __uint_as_float(1u << 22);
    } else {
      const int64_t nkb = p.cols >> 4, k = c0 >> 4;
      const float S_t = *p.tensor_scale;
      float m[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t sb = p.scales[p.sf_mma ? sf_mma_offset(r, k + h, nkb) : r * nkb + k + h];
        float rr = 0.0f;
        if (S_t > 0.0f && sb) {
          rr = __frcp_rn(__fmul_rn(e4m3_to_f32(sb), S_t));
          if (isinf(rr)) rr = FLT_MAX;
        }
        m[h] = rr;
      }
      mul0 = m[0];
      mul1 = m[1];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int t = i + 16 * hh;   // element of the chunk: P[i].x is t = i, P[i].y is t = 16 + i
        const float v = __fmul_rn(hh ? P[i].y : P[i].x, hh ? mul1 : mul0);
        const uint32_t k = (cws[t >> 3] >> (4 * (t & 7))) & 7u;
        const double e = (double)grid_level<GRID>(k) - fabs((double)v);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if ((int)k == kk) {
            acc[kk] += e;
            acc[8 + kk] += 1.0;
          }
        }
      }
    }
  }
  reduce_to<16>(acc, p.workspace, p.out);
}

struct RelErrParams {
  const float* ref;
  const float* approx;
  int64_t n;
  void* workspace;
  double* out;   // sum of (|approx| - |ref|) / |ref| over ref != 0, their count
};

__global__ void __launch_bounds__(kDiagThreads) rel_error_kernel(const RelErrParams p) {
  double acc[2] = {0.0, 0.0};
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += (int64_t)gridDim.x * blockDim.x) {
    const double r = p.ref[i], a = p.approx[i];
    if (r != 0.0) {
      acc[0] += (fabs(a) - fabs(r)) / fabs(r);
      acc[1] += 1.0;
    }
  }
  reduce_to<2>(acc, p.workspace, p.out);
}

template <int GRID, int SCALE>
cudaError_t launch_grid_error_nh(const GridErrParams& p, int nh, int blocks, cudaStream_t s) {
  switch (nh) {
    case 16: grid_error_kernel<GRID, SCALE, 16><<<blocks, kDiagThreads, 0, s>>>(p); break;
    case 32: grid_error_kernel<GRID, SCALE, 32><<<blocks, kDiagThreads, 0, s>>>(p); break;
    default: grid_error_kernel<GRID, SCALE, 0><<<blocks, kDiagThreads, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t zero_counter(void* workspace, cudaStream_t s) {
  return cudaMemsetAsync(static_cast<unsigned char*>(workspace) + (size_t)kDiagMaxBlocks * kDiagMaxVals * 8, 0, 4,
                         s);
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace fp4q

extern "C" size_t fp4q_diag_workspace_bytes(void) { return fp4q::diag_workspace(); }

extern "C" int32_t fp4q_grid_error(const void* x, int64_t rows, int64_t cols, int64_t ld, const fp4q_config* cfg,
                                   const fp4q_operand* row_copy, void* workspace, size_t ws_bytes, void* out,
                                   void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_grid_error");
  using namespace fp4q;
  if (!cfg || !row_copy || !out || !x) return FP4Q_ERR_INVALID_ARG;
  if (cfg->grid != FP4Q_GRID_E2M1 && cfg->grid != FP4Q_GRID_E1M2 && cfg->grid != FP4Q_GRID_E2M1_R4)
    return FP4Q_ERR_INVALID_ARG;
  if (cfg->scale != FP4Q_SCALE_MX && cfg->scale != FP4Q_SCALE_NV) return FP4Q_ERR_INVALID_ARG;
  if (cfg->rot != FP4Q_ROT_NONE && cfg->rot != FP4Q_ROT_H16 && cfg->rot != FP4Q_ROT_H32) return FP4Q_ERR_INVALID_ARG;
  if (cfg->sf_layout != FP4Q_SF_PLAIN && cfg->sf_layout != FP4Q_SF_MMA) return FP4Q_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || cols % 32 != 0 || ld < cols) return FP4Q_ERR_INVALID_ARG;
  if (cfg->sf_layout == FP4Q_SF_MMA && (rows % 128 != 0 || (cols / (cfg->scale == FP4Q_SCALE_MX ? 32 : 16)) % 4 != 0))
    return FP4Q_ERR_INVALID_ARG;
  if (!row_copy->codes || !row_copy->scales) return FP4Q_ERR_INVALID_ARG;
  if (cfg->scale == FP4Q_SCALE_NV && !row_copy->tensor_scale) return FP4Q_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < diag_workspace()) return FP4Q_ERR_WORKSPACE;
  if (!aligned_to(x, 16) || ld % 8 != 0 || !aligned_to(row_copy->codes, 16) || !aligned_to(out, 8) ||
      !aligned_to(workspace, 16))
    return FP4Q_ERR_ALIGNMENT;
  GridErrParams p;
  memset(&p, 0, sizeof p);
  p.x = static_cast<const uint16_t*>(x);
  p.rows = rows;
  p.cols = cols;
  p.ld = ld;
  p.codes = row_copy->codes;
  p.scales = row_copy->scales;
  p.tensor_scale = row_copy->tensor_scale;
  p.sf_mma = cfg->sf_layout == FP4Q_SF_MMA;
  for (int t = 0; t < 32; ++t)
    p.sgn[t] = (cfg->rot && ((cfg->sign_mask_row >> (t % cfg->rot)) & 1u)) ? 0x80000000u : 0u;
  p.workspace = workspace;
  p.out = static_cast<double*>(out);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (zero_counter(workspace, s) != cudaSuccess) return FP4Q_ERR_CUDA;
  const int blocks = diag_blocks(rows * (cols / 32));
  cudaError_t e;
  if (cfg->grid == FP4Q_GRID_E1M2)
    e = cfg->scale == FP4Q_SCALE_NV ? launch_grid_error_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_NV>(p, cfg->rot, blocks, s)
                                    : launch_grid_error_nh<FP4Q_GRID_E1M2, FP4Q_SCALE_MX>(p, cfg->rot, blocks, s);
  else   // the capped grid's codes decode with the E2M1 levels
    e = cfg->scale == FP4Q_SCALE_NV ? launch_grid_error_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_NV>(p, cfg->rot, blocks, s)
                                    : launch_grid_error_nh<FP4Q_GRID_E2M1, FP4Q_SCALE_MX>(p, cfg->rot, blocks, s);
  return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

extern "C" int32_t fp4q_rel_error(const float* ref, const float* approx, int64_t n, void* workspace,
                                  size_t ws_bytes, void* out, void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_rel_error");
  using namespace fp4q;
  if (n < 0 || !out) return FP4Q_ERR_INVALID_ARG;
  if (n > 0 && (!ref || !approx)) return FP4Q_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < diag_workspace()) return FP4Q_ERR_WORKSPACE;
  if (!aligned_to(out, 8) || !aligned_to(workspace, 16)) return FP4Q_ERR_ALIGNMENT;
  RelErrParams p;
  p.ref = ref;
  p.approx = approx;
  p.n = n;
  p.workspace = workspace;
  p.out = static_cast<double*>(out);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (zero_counter(workspace, s) != cudaSuccess) return FP4Q_ERR_CUDA;
  rel_error_kernel<<<diag_blocks(n), kDiagThreads, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}
