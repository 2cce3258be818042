// stats.cu -- bias statistics of a reconstruction against its reference:
// the fp64 sums behind SQNR, the attenuation factor alpha = <approx, ref> /
// ||ref||^2 and the magnitude shrinkage ("Repensando o Vies de Encolhimento",
// Metodologia 1 "Impacto Sistemico"; Resultados, quantization diagnostics),
// plus a histogram of the packed 4-bit codes (codebook use).
//
// HBM-bound streaming reduction.  The grid is four CTAs per SM of the device
// (at most kStatsMaxBlocks), every thread accumulates a grid-stride slice in
// fp64, CTAs reduce in a fixed tree and the last CTA to finish sums the
// per-CTA partials in CTA order, so results are bit-reproducible run to run
// on a given device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "fp4q_dev.cuh"
#include "fp4q_internal.h"

namespace fp4q {

constexpr int kStatsThreads = 256;
constexpr int kStatsMaxBlocks = 640;   // workspace bound: four CTAs per SM up to 160 SMs
constexpr int kSums = 5;

int stats_blocks() {
  const int b = 4 * num_sms();
  return b < kStatsMaxBlocks ? b : kStatsMaxBlocks;
}

// Workspace: [kStatsMaxBlocks][kSums] doubles, [kStatsMaxBlocks][16] uint64
// histogram partials, then one uint32 arrival counter.
size_t bias_stats_workspace(int64_t /*n*/) {
  return (size_t)kStatsMaxBlocks * (kSums + 16) * 8 + 256;
}

__global__ void __launch_bounds__(kStatsThreads) bias_stats_kernel(StatsParams sp) {
  double* part = reinterpret_cast<double*>(sp.workspace);
  unsigned long long* hpart = reinterpret_cast<unsigned long long*>(part + kStatsMaxBlocks * kSums);
  unsigned int* counter = reinterpret_cast<unsigned int*>(hpart + kStatsMaxBlocks * 16);
  __shared__ double red[kSums][kStatsThreads / 32];
  __shared__ unsigned int hist[16];
  __shared__ bool last;
  if (threadIdx.x < 16) hist[threadIdx.x] = 0;
  __syncthreads();

  double s[kSums] = {0, 0, 0, 0, 0};
  const int64_t n4 = sp.n >> 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const float4* r4 = reinterpret_cast<const float4*>(sp.ref);
  const float4* a4 = reinterpret_cast<const float4*>(sp.approx);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 rv = __ldcs(r4 + i), av = __ldcs(a4 + i);
    const float rr[4] = {rv.x, rv.y, rv.z, rv.w}, aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const double r = rr[k], a = aa[k], e = r - a;
      s[0] += r * r;
      s[1] += e * e;
      s[2] += r * a;
      s[3] += fabs(r);
      s[4] += fabs(a) - fabs(r);
    }
  }
  // tail (n not a multiple of 4)
  for (int64_t i = (n4 << 2) + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < sp.n; i += stride) {
    const double r = sp.ref[i], a = sp.approx[i], e = r - a;
    s[0] += r * r;
    s[1] += e * e;
    s[2] += r * a;
    s[3] += fabs(r);
    s[4] += fabs(a) - fabs(r);
  }
  if (sp.codes) {
    const int64_t nbytes = sp.n >> 1;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nbytes; i += stride) {
      const uint32_t b = sp.codes[i];
      atomicAdd(&hist[b & 15u], 1u);
      atomicAdd(&hist[b >> 4], 1u);
    }
  }
  // fixed-order block reduction: warp butterfly, then warps in order
#pragma unroll
  for (int k = 0; k < kSums; ++k) {
    double v = s[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if ((threadIdx.x & 31) == 0) red[k][threadIdx.x >> 5] = v;
  }
  __syncthreads();
  if (threadIdx.x < kSums) {
    double v = 0;
    for (int w = 0; w < kStatsThreads / 32; ++w) v += red[threadIdx.x][w];
    part[blockIdx.x * kSums + threadIdx.x] = v;
  }
  if (threadIdx.x < 16) hpart[blockIdx.x * 16 + threadIdx.x] = hist[threadIdx.x];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(counter, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  double* out = reinterpret_cast<double*>(sp.out);
  unsigned long long* oh = reinterpret_cast<unsigned long long*>(sp.out);
  if (threadIdx.x < kSums) {
    double v = 0;
    for (int b = 0; b < (int)gridDim.x; ++b) v += ((volatile double*)part)[b * kSums + threadIdx.x];
    out[threadIdx.x] = v;
  } else if (threadIdx.x >= 32 && threadIdx.x < 48) {
    const int c = threadIdx.x - 32;
    unsigned long long v = 0;
    for (int b = 0; b < (int)gridDim.x; ++b) v += ((volatile unsigned long long*)hpart)[b * 16 + c];
    oh[6 + c] = v;
  } else if (threadIdx.x == 64) {
    oh[5] = (unsigned long long)sp.n;
    *counter = 0u;   // ready for the next call on this workspace
  }
}

cudaError_t launch_bias_stats(const StatsParams& sp, cudaStream_t s) {
  unsigned char* ws = reinterpret_cast<unsigned char*>(sp.workspace);
  cudaError_t e = cudaMemsetAsync(ws + (size_t)kStatsMaxBlocks * (kSums + 16) * 8, 0, 4, s);
  if (e != cudaSuccess) return e;
  bias_stats_kernel<<<stats_blocks(), kStatsThreads, 0, s>>>(sp);
  return cudaGetLastError();
}

}  // namespace fp4q

// ------------------------------------------------------------------------
// Allocation-free variant of the bias statistics.
//
// The reduction's scratch (per-CTA partial sums, histogram partials and the
// arrival counter) lives in this file-scope device array instead of a caller
// workspace, so a caller that may not allocate device memory can still run
// it.  Every GPU that loads the library keeps the array until the process
// exits.  Its device address is looked up once per device (the first call on
// that device, with the device current) and cached in an atomic per device, so
// concurrent first calls from several host threads are safe; after
// cudaDeviceReset the module is loaded again and the address may change, so a
// reset must be followed by fp4q_bias_stats_noalloc_reset().  In host code the
// symbol is only a host-side stand-in and must never be handed to a kernel
// directly.
// All calls share the array: the counter is cleared on every call and the
// partials are overwritten, but two calls that overlap on the GPU (different
// streams, or different host threads) race on it.
// ------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocScratchBytes = 128 * 1024;
constexpr int kMaxDevices = 64;
__device__ __align__(256) unsigned char g_stats_scratch[kNoAllocScratchBytes];
std::atomic<void*> g_scratch_addr[kMaxDevices];
}  // namespace

extern "C" void fp4q_bias_stats_noalloc_reset(void) {
  for (int d = 0; d < kMaxDevices; ++d) g_scratch_addr[d].store(nullptr, std::memory_order_release);
}

extern "C" int32_t fp4q_bias_stats_noalloc(const float* ref, const float* approx, int64_t n,
                                           const uint8_t* codes, void* out, void* stream) {
  fp4q::NvtxRange nvtx_range("fp4q_bias_stats_noalloc");
  using namespace fp4q;
  if (n < 0 || !out) return FP4Q_ERR_INVALID_ARG;
  if (n > 0 && (!ref || !approx)) return FP4Q_ERR_INVALID_ARG;
  if (codes && (n % 2 != 0)) return FP4Q_ERR_INVALID_ARG;
  if (bias_stats_workspace(n) > kNoAllocScratchBytes) return FP4Q_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(out) % 8) != 0) return FP4Q_ERR_ALIGNMENT;
  if (n > 0 && ((reinterpret_cast<uintptr_t>(ref) | reinterpret_cast<uintptr_t>(approx)) % 16) != 0)
    return FP4Q_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4Q_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FP4Q_ERR_UNSUPPORTED;
  void* scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!scratch) {
    if (cudaGetSymbolAddress(&scratch, g_stats_scratch) != cudaSuccess || !scratch) return FP4Q_ERR_CUDA;
    g_scratch_addr[dev].store(scratch, std::memory_order_release);   // every thread stores the same address
  }
  StatsParams sp;
  sp.ref = ref;
  sp.approx = approx;
  sp.codes = codes;
  sp.n = n;
  sp.workspace = scratch;
  sp.out = out;
  return launch_bias_stats(sp, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}
