// fp4q_internal.h -- parameter blocks shared by the C-ABI layer and the
// kernels of libfp4q.so (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

namespace fp4q {

// NVTX range over one C-ABI call: named in profiler timelines (ncu can filter
// launches by it), a no-op when no profiler is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// One output copy of the quantizer (device pointers).
struct CopyOut {
  uint8_t* codes;
  uint8_t* scales;
  uint8_t* e4m3;
  float* tensor_scale;
};

// Kernel parameters of the quantizer family (passed by value; the sign words
// are read straight from the constant bank).
struct QuantParams {
  const uint16_t* x;   // bf16 input
  int64_t rows, cols, ld;
  CopyOut row, col;
  const float* gamax;  // NV: G of the (row, col) copies
  uint32_t* status;
  uint64_t sr_seed;
  uint32_t sr_keys[20];  // Philox round keys of sr_seed (philox_round_keys)
  int32_t want_row, want_col, sf_mma, emit_e4m3;
  uint32_t sgn_row[32];  // bit 31 set: negate element t of a 32-element chunk (row-wise)
  uint32_t sgn_col[32];  // same, column-wise copy
  // The same signs for packed bf16 pairs (bit 15 negates the low element, bit
  // 31 the high one): sw_row[k] for elements 2k, 2k+1 of a row-wise chunk;
  // sw_col[i] for element i of both column chunks of a column pair.
  uint32_t sw_row[16];
  uint32_t sw_col[32];
  // Bounded-wait test (fp4q_test_quantize_wait_expiry only; 0 / -1 otherwise):
  // CTA 0 waits for its tile stall_tile on a barrier nothing arrives at, giving
  // up after wait_limit_ns instead of the usual ~2 s.
  int32_t stall_tile;
  uint32_t wait_limit_ns;
};

// 2-D tensor map (inner dimension contiguous) and the device's SM count.
bool encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw);
int num_sms();

struct DequantParams {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* tensor_scale;
  float* out;
  int64_t rows, cols;
  uint32_t sign_mask;
  int32_t unrotate;
};

cudaError_t launch_rht_quant(const QuantParams& p, int grid_kind, int scale, int nh, int round, cudaStream_t s);
cudaError_t launch_rotated_amax(const QuantParams& p, int nh, float* amax, cudaStream_t s);
cudaError_t launch_dequant(const DequantParams& d, int grid_kind, int scale, int nh, cudaStream_t s);
cudaError_t launch_rotate_bf16(const QuantParams& p, int nh, uint16_t* y_row, uint16_t* y_col, cudaStream_t s);

struct StatsParams {
  const float* ref;
  const float* approx;
  const uint8_t* codes;
  int64_t n;
  void* workspace;
  void* out;
};
cudaError_t launch_bias_stats(const StatsParams& sp, cudaStream_t s);
size_t bias_stats_workspace(int64_t n);

}  // namespace fp4q
