/*
 * fp4q.h -- C ABI of the GB300 (sm_103a) fused Hadamard rotation + 4-bit
 * microscaled quantizer and block-scaled FP4 GEMM (libfp4q.so).
 *
 * Sources cited below (web pages, by title and section):
 *  [SB]  "Resumo Tecnico: Repensando o Vies de Encolhimento (Shrinkage Bias) no
 *        Pre-treinamento de LLMs em FP4" (gist.science, paper 2606.20381).
 *  [MX]  "Resumo Tecnico: Pre-treinamento de Modelos de Linguagem Grandes com
 *        MXFP4" (gist.science, paper 2605.09825).
 *  [HTX] HTX news article on arXiv 2605.09825, sections "Que es MXFP4?" and
 *        "Experimento de diagnostico".
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or keeps device memory; scratch comes from the
 *    caller's workspace argument.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on it; nothing is synchronised unless stated.  The quantizer
 *    and GEMM kernels launch as programmatic dependents of the stream's
 *    previous kernel (their launch and on-chip setup may overlap its tail);
 *    each waits for that kernel to complete before touching global memory,
 *    so stream order holds as for any launch.
 *  - Every call that launches work is an NVTX range named after the entry
 *    point (for profiler timelines and `ncu --nvtx` filters; a no-op when no
 *    profiler is attached).
 *  - Arguments are validated before any launch.  A rejected call returns a
 *    non-zero fp4q_status and launches nothing.  A launch failure returns
 *    FP4Q_ERR_CUDA.
 *  - Conditions seen only on the device (non-finite input, a wait that ran out
 *    of iterations) are OR-ed as FP4Q_DEV_* bits into *d_status (a device
 *    uint32 the caller zeroes and reads after synchronising).  d_status may be
 *    NULL.  Kernels never trap.
 *  - Matrices are row-major.  "Row-wise copy": blocks along the columns,
 *    stored rows x cols.  "Column-wise copy": blocks along the rows, stored
 *    TRANSPOSED (cols x rows) so that every GEMM operand is K-major.
 */
#ifndef FP4Q_H
#define FP4Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
  FP4Q_OK = 0,
  FP4Q_ERR_INVALID_ARG = 1,  /* bad size, null pointer, bad enum value      */
  FP4Q_ERR_UNSUPPORTED = 2,  /* valid values, unsupported combination       */
  FP4Q_ERR_ALIGNMENT = 3,    /* pointer or leading dimension not aligned    */
  FP4Q_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
  FP4Q_ERR_WORKSPACE = 5     /* workspace missing or smaller than required   */
} fp4q_status;

/* Bits OR-ed into *d_status by kernels. */
#define FP4Q_DEV_NONFINITE 0x1u  /* a block held NaN/Inf (input or rotation overflow) */
#define FP4Q_DEV_TIMEOUT 0x2u    /* a pipeline wait gave up; outputs are incomplete   */

/* 4-bit element grids ([SB] Declaracao do Problema; Metodologia 2):
 * E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; E1M2 magnitudes {k/4, k = 0..7}.
 * E2M1_R4 ([SB] Resultados, ablation of a range-restricted E2M1): E2M1 with
 * its maximum capped at 4 (codes 0..6, E2M1 bit patterns, e_max = 1).
 * A code is (sign << 3) | k. */
enum { FP4Q_GRID_E2M1 = 0, FP4Q_GRID_E1M2 = 1, FP4Q_GRID_E2M1_R4 = 2 };

/* Block scaling.
 * MX ([HTX] Que es MXFP4?): 32-element blocks sharing one E8M0 exponent,
 *    e = clamp(floor(log2 amax) - e_max, -127, 127), byte = e + 127,
 *    e_max = 2 (E2M1), 0 (E1M2) or 1 (E2M1_R4); element v = y * 2^-e.
 * NV (NVFP4-style, named in [SB] Declaracao do Problema): 16-element blocks,
 *    fp32 tensor scale S_t = G / (448 q_max) from the global amax G of the
 *    rotated copy, E4M3 block scale sb = E4M3_rtne_sat(fl(fl(amax/q_max)/S_t)),
 *    element v = y * fl(1 / fl(sb * S_t)). */
enum { FP4Q_SCALE_MX = 0, FP4Q_SCALE_NV = 1 };

/* Rotation ([MX] Metodologia 3: deterministic 16x16 / 32x32 Hadamard;
 * [SB] Metodologia 1 and [HTX] Experimento de diagnostico: random Hadamard
 * with sign flips).  y = c_n H_n D x per n-block along the blocked axis,
 * Sylvester order, butterfly stages in ascending stride in fp32, c_16 = 1/4,
 * c_32 = fl32(1/sqrt 32).  D = diag(+-1) from the orientation's sign mask. */
enum { FP4Q_ROT_NONE = 0, FP4Q_ROT_H16 = 16, FP4Q_ROT_H32 = 32 };

/* Rounding ([SB] Metodologia 2: RTNE everywhere, SR on dY only).
 * RTNE: nearest level, ties to the even code, saturating at q_max.
 * SR: with g_k <= |v| < g_k+1 and f = (|v| - g_k)/(g_k+1 - g_k), round up iff
 *     r / 2^16 < f, r = 16-bit half (low for even, high for odd index) of word
 *     (idx >> 1) & 3 of Philox4x32-10(key = sr_seed,
 *     counter = (lo32(idx >> 3), hi32(idx >> 3), orient, 0)), idx = index of
 *     the element in its stored copy, orient 0 row-wise / 1 column-wise. */
enum { FP4Q_RTNE = 0, FP4Q_SR = 1 };

/* Scale-factor layout of a copy (rows x cols of the stored copy, b = block).
 * PLAIN: row-major [rows][cols/b].
 * MMA:   the layout the block-scaled GEMM reads: 512-byte chunks, one per
 *        (128-row group R0, group of 4 consecutive blocks K0), ordered
 *        [rows/128][cols/(4b)]; inside a chunk the scale of row r, block k
 *        sits at byte 16*(r % 32) + 4*((r / 32) % 4) + (k % 4).
 *        Requires rows % 128 == 0 and (cols / b) % 4 == 0. */
enum { FP4Q_SF_PLAIN = 0, FP4Q_SF_MMA = 1 };

/* Per-call quantizer configuration (plain integers for a stable ABI). */
typedef struct {
  int32_t grid;            /* FP4Q_GRID_*                                         */
  int32_t scale;           /* FP4Q_SCALE_*                                        */
  int32_t rot;             /* FP4Q_ROT_*                                          */
  int32_t round;           /* FP4Q_RTNE or FP4Q_SR                                */
  uint32_t sign_mask_row;  /* bit j negates element j of each n-block, row-wise   */
  uint32_t sign_mask_col;  /* same for the column-wise copy (0 = deterministic H) */
  uint64_t sr_seed;        /* Philox key for SR                                   */
  int32_t want_row;        /* produce the row-wise copy                           */
  int32_t want_col;        /* produce the column-wise copy                        */
  int32_t sf_layout;       /* FP4Q_SF_PLAIN or FP4Q_SF_MMA                        */
  int32_t emit_e4m3;       /* also write one E4M3 byte per element (exact code value) */
  const float* global_amax;/* NV only: device float[2] = G of (row, col) copies, or
                              NULL to compute G in a pre-pass (needs workspace)  */
} fp4q_config;

/* One quantized copy; all device pointers, caller-owned. */
typedef struct {
  uint8_t* codes;          /* rows x cols/2 bytes, element 2t in the low nibble   */
  uint8_t* scales;         /* (rows x cols/b) bytes in the config's sf_layout     */
  float* tensor_scale;     /* NV: 1 float (S_t); MX: unused (may be NULL)         */
  uint8_t* e4m3;           /* rows x cols bytes when emit_e4m3, else unused       */
} fp4q_operand;

/* Text for a status code (static storage). */
const char* fp4q_status_str(int32_t status);

/* Library version and the device architecture it was built for (e.g. 1031). */
int32_t fp4q_version(void);

/* Rademacher sign mask for a random Hadamard rotation of size n_h (16 or 32):
 * the low n_h bits of word 0 of Philox4x32-10(key = seed,
 * counter = (0, 0, 0x5349474E, 0)).  Host-side, pure. */
uint32_t fp4q_sign_mask_from_seed(uint64_t seed, int32_t n_h);

/* Workspace bytes fp4q_rht_quantize needs for this configuration (0 unless
 * NV-style without caller-supplied global amax). */
size_t fp4q_workspace_bytes(int64_t rows, int64_t cols, const fp4q_config* cfg);

/* Fused blockwise (random) Hadamard rotation + 4-bit microscaled quantization
 * of one bf16 operand, both copies from one read
 * ([SB] Metodologia 2 and Eficiencia: rotation fused with FP4 quantization;
 *  [HTX] Que es MXFP4? and Experimento de diagnostico: every GEMM operand).
 *  x        device bf16, rows x cols, row stride ld elements (ld >= cols,
 *           ld % 8 == 0, x 16-byte aligned)
 *  rows     >= 0; a multiple of 32 when want_col (the MMA scale layout also
 *           needs the copy's rows % 128 == 0 and its blocks per row % 4 == 0)
 *  cols     >= 0, a multiple of 32
 *  row_out  row-wise copy (rows x cols), used when cfg->want_row
 *  col_out  column-wise copy stored transposed (cols x rows), when want_col
 *  workspace/ws_bytes  device scratch of fp4q_workspace_bytes() bytes
 *  d_status device uint32 for FP4Q_DEV_* bits, or NULL
 * Empty matrices return FP4Q_OK without launching. */
int32_t fp4q_rht_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                          const fp4q_config* cfg, const fp4q_operand* row_out,
                          const fp4q_operand* col_out, void* workspace, size_t ws_bytes,
                          uint32_t* d_status, void* stream);

/* Global amax pass of the NVFP4-style recipe: G of the rotated row-wise and
 * column-wise copies, written to amax_out[0..1] (device floats, overwritten).
 * The same rotation parameters as fp4q_rht_quantize are taken from cfg. */
int32_t fp4q_rotated_amax(const void* x, int64_t rows, int64_t cols, int64_t ld,
                          const fp4q_config* cfg, float* amax_out, uint32_t* d_status,
                          void* stream);

/* Reconstruction of one stored copy ([HTX] Que es MXFP4?: element = shared
 * scale times the 4-bit value):
 *   MX: out = g[k] * 2^(byte - 127) (exact);  NV: out = fl(fl(g[k] * sb) * S_t).
 *  q        the copy (codes, scales in PLAIN layout, tensor_scale for NV)
 *  rows, cols  the stored copy's own shape (a column-wise copy is cols x rows of
 *           its source)
 *  cfg      grid, scale, rot and sign mask (orient selects row/col mask)
 *  unrotate 1: apply the inverse rotation (same butterfly, c_n, then the signs)
 *  out      device fp32 rows x cols */
int32_t fp4q_dequantize(const fp4q_operand* q, int64_t rows, int64_t cols,
                        const fp4q_config* cfg, int32_t orient, int32_t unrotate, float* out,
                        void* stream);

/* Block-scaled 4-bit GEMM D = alpha_g * A B^T on tcgen05 tensor cores
 * ([HTX] Experimento de diagnostico: Fprop Y = X W^T, Dgrad dX = dY W,
 *  Wgrad dW = dY^T X, each written with K-major operands).
 *  A        M x K copy (codes; scales in FP4Q_SF_MMA layout; e4m3 for E1M2)
 *  B        N x K copy, same form
 *  grid, scale   the operands' recipe (E2M1_R4 runs as E2M1).  E2M1+MX runs kind::mxf4, E2M1+NV runs
 *           kind::mxf4nvf4 with E4M3 scales, E1M2+MX runs kind::mxf8f6f4 on the
 *           E4M3 bytes (E1M2 levels are exact in E4M3).  E1M2+NV is
 *           FP4Q_ERR_UNSUPPORTED.  alpha_g = S_t(A) * S_t(B) for NV, else 1.
 *  M % 128 == 0, N % 128 == 0, K % 128 == 0 (K % 64 for NV), all > 0
 *  D_bf16   device bf16 M x N (row-major), or NULL
 *  D_f32    device fp32 M x N, or NULL (at least one output)
 *  d_status device uint32 for FP4Q_DEV_TIMEOUT, or NULL */
int32_t fp4q_gemm(const fp4q_operand* A, const fp4q_operand* B, int64_t M, int64_t N, int64_t K,
                  int32_t grid, int32_t scale, void* D_bf16, float* D_f32, uint32_t* d_status,
                  void* stream);

/* Several block-scaled GEMMs of one recipe (grid, scale) in one launch, each
 * exactly as fp4q_gemm computes it (the same tiles, bit for bit): for the
 * GEMMs of one training phase, e.g. Dgrad and Wgrad of a linear layer, whose
 * tiles cost differently (K), so that one persistent launch over a
 * cost-balanced static tile list keeps every SM busy to the end.
 *  problems  count descriptions, each as fp4q_gemm's arguments (A, B, M, N, K,
 *           D_bf16, D_f32; at least one output each)
 *  count    1 .. 4
 *  Returns FP4Q_ERR_UNSUPPORTED when the GEMMs have more than 8192 256 x 256
 *  tiles together (call fp4q_gemm for each then), otherwise as fp4q_gemm.
 *  The outputs must not overlap one another or the inputs. */
typedef struct {
  const fp4q_operand* A;
  const fp4q_operand* B;
  int64_t M, N, K;
  void* D_bf16;
  float* D_f32;
} fp4q_gemm_problem;
int32_t fp4q_gemm_group(const fp4q_gemm_problem* problems, int32_t count, int32_t grid, int32_t scale,
                        uint32_t* d_status, void* stream);

/* The same GEMM, quantizing its own output in the epilogue: `out` receives
 * the row-wise copy of bf16(D) that fp4q_rht_quantize would produce from the
 * stored bf16 D with `out_cfg`, bit for bit, without D making a round trip
 * through HBM.  This is the step after the hot path that the linear-layer
 * recipe uses between layers: Fprop's Y becomes the next layer's X, Dgrad's dX
 * the previous layer's dY ("Repensando o Vies de Encolhimento", Metodologia 2:
 * every GEMM operand quantized, with the rotation, RTNE on activations and
 * weights and SR on gradients).
 *  A, B, M, N, K, grid, scale, d_status   as fp4q_gemm
 *  D_bf16   device bf16 M x N, or NULL (the output is then only quantized)
 *  out_cfg  the copy's recipe: grid, rot and sign_mask_row (along N, the next
 *           GEMM's contraction axis), round and sr_seed (element index = r*N + c
 *           of the M x N copy, orientation 0), sf_layout, emit_e4m3.  It must
 *           ask for MX scales and the row-wise copy only (want_row = 1,
 *           want_col = 0); NV scaling needs the amax of the whole rotated
 *           output before the first block is encoded and is FP4Q_ERR_UNSUPPORTED,
 *           as is a column-wise copy.
 *  out      device copy: codes M x N/2 (16-byte aligned), scales M x N/32,
 *           e4m3 M x N when emit_e4m3
 * Non-finite GEMM outputs set FP4Q_DEV_NONFINITE in *d_status. */
int32_t fp4q_gemm_quantize(const fp4q_operand* A, const fp4q_operand* B, int64_t M, int64_t N, int64_t K,
                           int32_t grid, int32_t scale, void* D_bf16, const fp4q_config* out_cfg,
                           fp4q_operand* out, uint32_t* d_status, void* stream);

/* Bias statistics over n element pairs ([SB] Metodologia 1: attenuation
 * alpha = <approx, ref>/||ref||^2 and the magnitude shrinkage; Resultados:
 * SQNR).  Sums in fp64, in a fixed order (deterministic).
 *  ref, approx  device fp32[n];  codes  device packed codes (n/2 bytes) or NULL
 *  workspace    device scratch of fp4q_bias_stats_workspace_bytes(n) bytes
 *  out          device buffer of 22 8-byte words: doubles sum ref^2,
 *               sum (ref-approx)^2, sum ref*approx, sum |ref|,
 *               sum (|approx| - |ref|), then uint64 n and hist[16] */
size_t fp4q_bias_stats_workspace_bytes(int64_t n);
int32_t fp4q_bias_stats(const float* ref, const float* approx, int64_t n, const uint8_t* codes,
                        void* workspace, size_t ws_bytes, void* out, void* stream);

/* Allocation-free form of fp4q_bias_stats.  The pages have no counterpart:
 * this exists for callers that cannot allocate device memory -- a host
 * framework or serving runtime that owns every device byte through its own
 * pre-reserved pool, a plugin running inside another program's fixed memory
 * budget, or a path that must not pay for cudaMalloc's implicit device
 * synchronisation.  They still pass the inputs and the output buffer; the reduction's scratch is a 128 KiB device array
 * built into the library (held on every GPU that loads it until the process
 * exits).  Same arguments, results and determinism as fp4q_bias_stats.
 *  - Calls whose scratch need (fp4q_bias_stats_workspace_bytes(n)) exceeds the
 *    built-in 128 KiB return FP4Q_ERR_WORKSPACE; the current reduction needs
 *    about 105 KiB for every n, so every n >= 0 fits.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it (safe when several host threads make
 *    that first call at once); make that first call before any stream
 *    capture.  After cudaDeviceReset the library's device array is loaded
 *    anew: call fp4q_bias_stats_noalloc_reset() so that the next call looks
 *    the address up again.
 *  - All calls share the one array: two calls that overlap on the GPU (other
 *    streams, other host threads) race and give undefined sums.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine. */
int32_t fp4q_bias_stats_noalloc(const float* ref, const float* approx, int64_t n, const uint8_t* codes,
                                void* out, void* stream);
/* Forget the cached device addresses of that array (host only; after a
 * device reset). */
void fp4q_bias_stats_noalloc_reset(void);

/* Host helper: SQNR (dB), alpha and shrinkage from the five sums above. */
void fp4q_stats_finalize(const double* sums5, double* sqnr_db, double* alpha, double* shrinkage);

/* Diagnostics of the shrinkage bias ([SB] Metodologia 1, "Origem
 * Geometrica"), deterministic fp64 reductions like fp4q_bias_stats.
 *
 * fp4q_grid_error: the rounding error in grid units of a ROW-WISE copy of the
 * rows x cols bf16 x (row stride ld): per element, its position
 * v = y * step^-1 on the grid (y the rotated value under cfg's rot and
 * sign_mask_row, the step exactly as fp4q_rht_quantize takes it: 2^(127-sb)
 * for MX, fl(1/fl(e4m3(sb) S_t)) for NV, 0 where an NV scale byte is 0) and
 * its code's level g[k], k = code & 7.  out (device, 16 8-byte words): doubles
 * sum over the elements of level k of g[k] - |v| for k = 0..7, then the counts
 * of level k as doubles.  The mean of level k is the page's E[q - x | bin] =
 * (l_i - r_i)/2 on locally uniform data.  cfg supplies grid, scale, rot,
 * sign_mask_row and sf_layout (the copy's scale layout); a column-wise copy
 * is the row-wise copy of the transposed input.
 *
 * fp4q_rel_error: sum over ref != 0 of (|approx| - |ref|) / |ref| and the
 * number of such elements, two doubles in out (device): the per-element
 * mean signed relative error is their quotient, reported beside the
 * aggregate shrinkage of fp4q_bias_stats.
 *
 * Both take a device workspace of fp4q_diag_workspace_bytes() bytes
 * (FP4Q_ERR_WORKSPACE if smaller) and are asynchronous on `stream`.
 * Arguments: rows, cols > 0, cols % 32 == 0, ld >= cols with ld % 8 == 0,
 * 16-byte aligned x, codes and workspace, 8-byte aligned out. */
size_t fp4q_diag_workspace_bytes(void);
int32_t fp4q_grid_error(const void* x, int64_t rows, int64_t cols, int64_t ld, const fp4q_config* cfg,
                        const fp4q_operand* row_copy, void* workspace, size_t ws_bytes, void* out, void* stream);
int32_t fp4q_rel_error(const float* ref, const float* approx, int64_t n, void* workspace, size_t ws_bytes,
                       void* out, void* stream);

/* Test of the quantizer's bounded waits (no page counterpart): the same call
 * as fp4q_rht_quantize, except that CTA 0 waits for its tile number
 * stall_tile (0 = its first tile) on a pipeline barrier that nothing arrives
 * at, and gives up after wait_limit_us microseconds (1 .. 2000000) instead of
 * the usual ~2 s.  That CTA then raises FP4Q_DEV_TIMEOUT in *d_status, waits
 * (bounded) for its own tile loads in flight and returns, leaving its tiles
 * unwritten; the other CTAs finish normally and the context stays usable.
 * A stall_tile past CTA 0's last tile changes nothing.  Returns
 * FP4Q_ERR_INVALID_ARG for stall_tile < 0 or a limit outside that range,
 * otherwise as fp4q_rht_quantize. */
int32_t fp4q_test_quantize_wait_expiry(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                       const fp4q_config* cfg, const fp4q_operand* row_out,
                                       const fp4q_operand* col_out, void* workspace, size_t ws_bytes,
                                       uint32_t* d_status, int32_t stall_tile, uint32_t wait_limit_us,
                                       void* stream);

/* Unfused comparison arm (measurement only, [SB] Eficiencia: fused versus
 * unfused rotation + quantization): rotate x blockwise along its rows
 * (orient 0) or columns (orient 1) and write the rotated tensor in bf16
 * (RNE), y_row rows x cols and/or y_col rows x cols (same orientation as x),
 * from one read.  Either output may be NULL. */
int32_t fp4q_hadamard_rotate_bf16(const void* x, int64_t rows, int64_t cols, int64_t ld,
                                  int32_t rot, uint32_t sign_mask_row, uint32_t sign_mask_col,
                                  void* y_row, void* y_col, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* FP4Q_H */
