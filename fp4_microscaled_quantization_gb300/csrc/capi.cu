// capi.cu -- the extern "C" entry points of libfp4q.so declared in
// include/fp4q.h: argument validation, status codes and kernel launches.
// Nothing here allocates device memory; scratch comes from the caller.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "../../include/fp4q.h"
#include "fp4q_dev.cuh"
#include "fp4q_internal.h"

using namespace fp4q;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_cfg(const fp4q_config* c) {
  if (!c) return false;
  if (c->grid != FP4Q_GRID_E2M1 && c->grid != FP4Q_GRID_E1M2 && c->grid != FP4Q_GRID_E2M1_R4) return false;
  if (c->scale != FP4Q_SCALE_MX && c->scale != FP4Q_SCALE_NV) return false;
  if (c->rot != FP4Q_ROT_NONE && c->rot != FP4Q_ROT_H16 && c->rot != FP4Q_ROT_H32) return false;
  if (c->round != FP4Q_RTNE && c->round != FP4Q_SR) return false;
  if (c->sf_layout != FP4Q_SF_PLAIN && c->sf_layout != FP4Q_SF_MMA) return false;
  return true;
}

int block_of(int32_t scale) { return scale == FP4Q_SCALE_MX ? 32 : 16; }

// Sign words of a 32-element chunk: bit 31 set where element t of its n-block
// is negated.
void sign_words(uint32_t mask, int nh, uint32_t* out) {
  for (int t = 0; t < 32; ++t) out[t] = (nh && ((mask >> (t % nh)) & 1u)) ? 0x80000000u : 0u;
}

// Checks of one output copy with `crow` rows and `ccol` columns.
int32_t check_copy(const fp4q_operand* o, int64_t crow, int64_t ccol, const fp4q_config* c) {
  if (!o || !o->codes || !o->scales) return FP4Q_ERR_INVALID_ARG;
  if (!aligned(o->codes, 16)) return FP4Q_ERR_ALIGNMENT;
  if (c->scale == FP4Q_SCALE_NV) {
    if (!o->tensor_scale) return FP4Q_ERR_INVALID_ARG;
    if (!aligned(o->scales, 2) || !aligned(o->tensor_scale, 4)) return FP4Q_ERR_ALIGNMENT;
  }
  if (c->emit_e4m3) {
    if (!o->e4m3) return FP4Q_ERR_INVALID_ARG;
    if (!aligned(o->e4m3, 16)) return FP4Q_ERR_ALIGNMENT;
  }
  if (c->sf_layout == FP4Q_SF_MMA) {
    if (crow % 128 != 0 || (ccol / block_of(c->scale)) % 4 != 0) return FP4Q_ERR_INVALID_ARG;
  }
  return FP4Q_OK;
}

int32_t cuda_status(cudaError_t e) { return e == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA; }

// Shared validation + parameter block of the quantizer family.
int32_t prepare(const void* x, int64_t rows, int64_t cols, int64_t ld, const fp4q_config* cfg,
                QuantParams& p) {
  if (!valid_cfg(cfg)) return FP4Q_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ld < cols) return FP4Q_ERR_INVALID_ARG;
  if (!cfg->want_row && !cfg->want_col) return FP4Q_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP4Q_OK;
  if (!x) return FP4Q_ERR_INVALID_ARG;
  if (cols % 32 != 0) return FP4Q_ERR_INVALID_ARG;
  if (cfg->want_col && rows % 32 != 0) return FP4Q_ERR_INVALID_ARG;
  if ((rows + 63) / 64 > 65535) return FP4Q_ERR_INVALID_ARG;
  if (!aligned(x, 16) || ld % 8 != 0) return FP4Q_ERR_ALIGNMENT;
  memset(&p, 0, sizeof p);
  p.x = static_cast<const uint16_t*>(x);
  p.rows = rows;
  p.cols = cols;
  p.ld = ld;
  p.sr_seed = cfg->sr_seed;
  philox_round_keys(cfg->sr_seed, p.sr_keys);
  p.want_row = cfg->want_row ? 1 : 0;
  p.want_col = cfg->want_col ? 1 : 0;
  p.sf_mma = cfg->sf_layout == FP4Q_SF_MMA ? 1 : 0;
  p.emit_e4m3 = cfg->emit_e4m3 ? 1 : 0;
  sign_words(cfg->sign_mask_row, cfg->rot, p.sgn_row);
  sign_words(cfg->sign_mask_col, cfg->rot, p.sgn_col);
  for (int k = 0; k < 16; ++k) p.sw_row[k] = (p.sgn_row[2 * k] >> 16) | p.sgn_row[2 * k + 1];
  for (int i = 0; i < 32; ++i) p.sw_col[i] = p.sgn_col[i] | (p.sgn_col[i] >> 16);
  p.stall_tile = -1;
  p.wait_limit_ns = 0;
  return FP4Q_OK;
}

}  // namespace

extern "C" {

const char* fp4q_status_str(int32_t s) {
  switch (s) {
    case FP4Q_OK: return "ok";
    case FP4Q_ERR_INVALID_ARG: return "invalid argument";
    case FP4Q_ERR_UNSUPPORTED: return "unsupported combination";
    case FP4Q_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case FP4Q_ERR_CUDA: return "CUDA runtime error";
    case FP4Q_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int32_t fp4q_version(void) { return 10000 * 1 + 1031; }

uint32_t fp4q_sign_mask_from_seed(uint64_t seed, int32_t n_h) {
  const Philox4 r = philox4x32_10(0u, 0u, 0x5349474Eu, 0u, (uint32_t)seed, (uint32_t)(seed >> 32));
  if (n_h >= 32) return r.v[0];
  if (n_h <= 0) return 0u;
  return r.v[0] & ((1u << n_h) - 1u);
}

size_t fp4q_workspace_bytes(int64_t rows, int64_t cols, const fp4q_config* cfg) {
  (void)rows;
  (void)cols;
  if (!cfg) return 0;
  return (cfg->scale == FP4Q_SCALE_NV && cfg->global_amax == nullptr) ? 256 : 0;
}

}  // extern "C"

namespace {
// fp4q_rht_quantize with the bounded-wait test parameters (stall_tile < 0: none).
int32_t rht_quantize_impl(const void* x, int64_t rows, int64_t cols, int64_t ld, const fp4q_config* cfg,
                          const fp4q_operand* row_out, const fp4q_operand* col_out, void* workspace,
                          size_t ws_bytes, uint32_t* d_status, void* stream, int32_t stall_tile,
                          uint32_t wait_limit_ns) {
  QuantParams p;
  int32_t st = prepare(x, rows, cols, ld, cfg, p);
  if (st != FP4Q_OK || rows == 0 || cols == 0) return st;
  if (cfg->want_row) {
    if ((st = check_copy(row_out, rows, cols, cfg)) != FP4Q_OK) return st;
    p.row = CopyOut{row_out->codes, row_out->scales, row_out->e4m3, row_out->tensor_scale};
  }
  if (cfg->want_col) {
    if ((st = check_copy(col_out, cols, rows, cfg)) != FP4Q_OK) return st;
    p.col = CopyOut{col_out->codes, col_out->scales, col_out->e4m3, col_out->tensor_scale};
  }
  p.status = d_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cfg->scale == FP4Q_SCALE_NV) {
    if (cfg->global_amax) {
      if (!aligned(cfg->global_amax, 4)) return FP4Q_ERR_ALIGNMENT;
      p.gamax = cfg->global_amax;
    } else {
      if (!workspace || ws_bytes < 8) return FP4Q_ERR_WORKSPACE;
      if (!aligned(workspace, 16)) return FP4Q_ERR_ALIGNMENT;
      float* g = static_cast<float*>(workspace);
      if ((st = cuda_status(launch_rotated_amax(p, cfg->rot, g, s))) != FP4Q_OK) return st;
      p.gamax = g;
    }
  }
  p.stall_tile = stall_tile;
  p.wait_limit_ns = wait_limit_ns;
  return cuda_status(launch_rht_quant(p, cfg->grid, cfg->scale, cfg->rot, cfg->round, s));
}
}  // namespace

extern "C" {

int32_t fp4q_rht_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, const fp4q_config* cfg,
                          const fp4q_operand* row_out, const fp4q_operand* col_out, void* workspace,
                          size_t ws_bytes, uint32_t* d_status, void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_rht_quantize");
  return rht_quantize_impl(x, rows, cols, ld, cfg, row_out, col_out, workspace, ws_bytes, d_status, stream, -1, 0);
}

int32_t fp4q_test_quantize_wait_expiry(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                       const fp4q_config* cfg, const fp4q_operand* row_out,
                                       const fp4q_operand* col_out, void* workspace, size_t ws_bytes,
                                       uint32_t* d_status, int32_t stall_tile, uint32_t wait_limit_us,
                                       void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_test_quantize_wait_expiry");
  if (stall_tile < 0 || wait_limit_us == 0 || wait_limit_us > 2000000u) return FP4Q_ERR_INVALID_ARG;
  return rht_quantize_impl(x, rows, cols, ld, cfg, row_out, col_out, workspace, ws_bytes, d_status, stream,
                           stall_tile, wait_limit_us * 1000u);
}

int32_t fp4q_rotated_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, const fp4q_config* cfg,
                          float* amax_out, uint32_t* d_status, void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_rotated_amax");
  QuantParams p;
  int32_t st = prepare(x, rows, cols, ld, cfg, p);
  if (st != FP4Q_OK) return st;
  if (!amax_out) return FP4Q_ERR_INVALID_ARG;
  if (!aligned(amax_out, 4)) return FP4Q_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rows == 0 || cols == 0) return cuda_status(cudaMemsetAsync(amax_out, 0, 2 * sizeof(float), s));
  p.status = d_status;
  return cuda_status(launch_rotated_amax(p, cfg->rot, amax_out, s));
}

int32_t fp4q_dequantize(const fp4q_operand* q, int64_t rows, int64_t cols, const fp4q_config* cfg,
                        int32_t orient, int32_t unrotate, float* out, void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_dequantize");
  if (!valid_cfg(cfg) || !q || (orient != 0 && orient != 1)) return FP4Q_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0) return FP4Q_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP4Q_OK;
  if (cols % 32 != 0 || !q->codes || !q->scales || !out) return FP4Q_ERR_INVALID_ARG;
  if (cfg->sf_layout != FP4Q_SF_PLAIN) return FP4Q_ERR_UNSUPPORTED;
  if (cfg->scale == FP4Q_SCALE_NV && !q->tensor_scale) return FP4Q_ERR_INVALID_ARG;
  if (!aligned(q->codes, 16) || !aligned(out, 16)) return FP4Q_ERR_ALIGNMENT;
  if (rows * (cols / 32) / 256 + 1 > 0x7FFFFFFFLL) return FP4Q_ERR_INVALID_ARG;
  DequantParams d;
  d.codes = q->codes;
  d.scales = q->scales;
  d.tensor_scale = q->tensor_scale;
  d.out = out;
  d.rows = rows;
  d.cols = cols;
  d.sign_mask = orient ? cfg->sign_mask_col : cfg->sign_mask_row;
  d.unrotate = unrotate ? 1 : 0;
  return cuda_status(launch_dequant(d, cfg->grid, cfg->scale, cfg->rot, static_cast<cudaStream_t>(stream)));
}

size_t fp4q_bias_stats_workspace_bytes(int64_t n) { return bias_stats_workspace(n); }

int32_t fp4q_bias_stats(const float* ref, const float* approx, int64_t n, const uint8_t* codes,
                        void* workspace, size_t ws_bytes, void* out, void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_bias_stats");
  if (n < 0 || !out) return FP4Q_ERR_INVALID_ARG;
  if (n > 0 && (!ref || !approx)) return FP4Q_ERR_INVALID_ARG;
  if (codes && (n % 2 != 0)) return FP4Q_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < bias_stats_workspace(n)) return FP4Q_ERR_WORKSPACE;
  if (!aligned(out, 8) || !aligned(workspace, 16)) return FP4Q_ERR_ALIGNMENT;
  if (n > 0 && (!aligned(ref, 16) || !aligned(approx, 16))) return FP4Q_ERR_ALIGNMENT;
  StatsParams sp;
  sp.ref = ref;
  sp.approx = approx;
  sp.codes = codes;
  sp.n = n;
  sp.workspace = workspace;
  sp.out = out;
  return cuda_status(launch_bias_stats(sp, static_cast<cudaStream_t>(stream)));
}

void fp4q_stats_finalize(const double* s, double* sqnr_db, double* alpha, double* shrinkage) {
  if (!s) return;
  if (sqnr_db) *sqnr_db = s[1] > 0 ? 10.0 * log10(s[0] / s[1]) : INFINITY;
  if (alpha) *alpha = s[0] > 0 ? s[2] / s[0] : NAN;
  if (shrinkage) *shrinkage = s[3] > 0 ? s[4] / s[3] : NAN;
}

int32_t fp4q_hadamard_rotate_bf16(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t rot,
                                  uint32_t sign_mask_row, uint32_t sign_mask_col, void* y_row, void* y_col,
                                  void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_hadamard_rotate_bf16");
  if (rot != FP4Q_ROT_H16 && rot != FP4Q_ROT_H32) return FP4Q_ERR_INVALID_ARG;
  if (!y_row && !y_col) return FP4Q_ERR_INVALID_ARG;
  fp4q_config c;
  memset(&c, 0, sizeof c);
  c.rot = rot;
  c.sign_mask_row = sign_mask_row;
  c.sign_mask_col = sign_mask_col;
  c.want_row = y_row != nullptr;
  c.want_col = y_col != nullptr;
  QuantParams p;
  int32_t st = prepare(x, rows, cols, ld, &c, p);
  if (st != FP4Q_OK || rows == 0 || cols == 0) return st;
  if ((y_row && !aligned(y_row, 16)) || (y_col && !aligned(y_col, 16))) return FP4Q_ERR_ALIGNMENT;
  return cuda_status(launch_rotate_bf16(p, rot, static_cast<uint16_t*>(y_row), static_cast<uint16_t*>(y_col),
                                        static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
