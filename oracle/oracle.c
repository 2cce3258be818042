/*
 * oracle.c -- plain, slow CPU oracle for the fused Hadamard rotation + 4-bit
 * microscaled quantizer, its dequantizer, the GEMM entry and the bias
 * statistics.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file.  The CUDA library shares no
 * code, header, table or constant with it.
 *
 * Every step is written element by element in the order the method states it,
 * in IEEE fp32 with round-to-nearest where the method is an fp32 encoding, and
 * in fp64 for the statistics and GEMM sums.  Build with -ffp-contract=off and
 * without fast-math so that no multiply-add is fused and no step is reordered.
 *
 * Sources (web pages, cited by title and section):
 *  [SB]  "Resumo Tecnico: Repensando o Vies de Encolhimento (Shrinkage Bias)
 *         no Pre-treinamento de LLMs em FP4" (gist.science, paper 2606.20381),
 *         and its Korean mirror with the same sections.
 *  [MX]  "Resumo Tecnico: Pre-treinamento de Modelos de Linguagem Grandes com
 *         MXFP4" (gist.science, paper 2605.09825).
 *  [HTX] HTX news article on arXiv 2605.09825 ("New AMD paper overturns
 *         conventional wisdom: FP4 training..."), sections "Que es MXFP4?"
 *         and "Experimento de diagnostico".
 *
 * Readings of points the pages leave open are stated beside the step they
 * govern.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Enumerations, mirrored by value in oracle/__init__.py                     */
/* ------------------------------------------------------------------------ */
enum { ORC_GRID_E2M1 = 0, ORC_GRID_E1M2 = 1, ORC_GRID_E2M1_R4 = 2 };
enum { ORC_SCALE_MX = 0, ORC_SCALE_NV = 1 };
enum { ORC_RTNE = 0, ORC_SR = 1 };

/* Return codes of orc_quantize. */
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_NONFINITE = 2 };

/* ------------------------------------------------------------------------ */
/* 4-bit grids                                                              */
/* ------------------------------------------------------------------------ */
/* E2M1: 2 exponent bits, 1 mantissa bit ([SB] Declaracao do Problema).
 * Magnitudes of codes 0..7; the non-uniform spacing 0.5 -> 1 -> 2 is the
 * source of the bin asymmetry ([SB] Metodologia 1, "Origem Geometrica"). */
static const float E2M1_LEVELS[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
/* E1M2: 1 exponent bit, 2 mantissa bits, uniform spacing 1/4 so that every
 * left and right bin width agree ([SB] Metodologia 2, "Grade Uniforme"). */
static const float E1M2_LEVELS[8] = {0.0f, 0.25f, 0.5f, 0.75f, 1.0f, 1.25f, 1.5f, 1.75f};

/* Range-restricted E2M1 ([SB] Resultados, ablation "Restricao de Alcance":
 * E2M1 with its largest values cut to mimic a uniform grid).  Reading: the
 * maximum is capped at 4 (levels 0 .. 4, codes 0..6 -- still E2M1 bit
 * patterns, decoded with the E2M1 table), and the shared exponent uses
 * e_max = 1 so that block maxima land in [2, 4) and never clip. */

float orc_grid_level(int grid, int k)
{
    if (k < 0 || k > 7) return NAN;
    return grid == ORC_GRID_E1M2 ? E1M2_LEVELS[k] : E2M1_LEVELS[k];
}

/* Index of the largest code a grid produces (7, or 6 for the capped grid). */
int orc_grid_top(int grid) { return grid == ORC_GRID_E2M1_R4 ? 6 : 7; }

/* Largest magnitude of the grid. */
float orc_grid_qmax(int grid) { return orc_grid_level(grid, orc_grid_top(grid)); }

/* Exponent of the power of two the block maximum is scaled to: 2 for E2M1
 * (largest power of two not above 6), 0 for E1M2 (1 <= 1.75), 1 for the
 * capped grid (block maxima in [2, 4)). */
int orc_grid_emax(int grid)
{
    if (grid == ORC_GRID_E1M2) return 0;
    return grid == ORC_GRID_E2M1_R4 ? 1 : 2;
}

/* Value of a 4-bit code: bit 3 is the sign, bits 0..2 the magnitude index. */
float orc_code_value(int grid, int code)
{
    float m = orc_grid_level(grid, code & 7);
    return (code & 8) ? -m : m;
}

/* ------------------------------------------------------------------------ */
/* bf16 input                                                               */
/* ------------------------------------------------------------------------ */
float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 (block scales of the NVFP4-style recipe)                        */
/* Format: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; subnormals    */
/* m * 2^-9; largest finite 448 (0x7E); 0x7F is NaN; no infinities.         */
/* ------------------------------------------------------------------------ */
float orc_e4m3_decode(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexpf((float)m, -9);
    else v = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return s ? -v : v;
}

/* Round x >= 0 to the nearest E4M3 value, ties to the even mantissa, and
 * saturate anything at or above the largest finite value (448) to 448.
 * Written as a search over the 127 non-negative finite values. */
uint8_t orc_e4m3_encode(float x)
{
    if (isnan(x)) return 0x7F;
    int neg = signbit(x) ? 1 : 0;
    float a = fabsf(x);
    uint8_t best;
    if (a >= 448.0f) {
        best = 0x7E;
    } else {
        best = 0;
        for (int c = 0; c < 0x7E; ++c) {
            float lo = orc_e4m3_decode((uint8_t)c), hi = orc_e4m3_decode((uint8_t)(c + 1));
            if (a >= lo && a <= hi) {
                double mid = 0.5 * ((double)lo + (double)hi);
                if ((double)a < mid) best = (uint8_t)c;
                else if ((double)a > mid) best = (uint8_t)(c + 1);
                else best = (uint8_t)((c & 1) ? c + 1 : c); /* tie: even mantissa */
                break;
            }
        }
    }
    return (uint8_t)(best | (neg ? 0x80 : 0));
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as   */
/* easy as 1, 2, 3", SC'11).  Counter-based: the output depends only on the  */
/* counter and the key.                                                     */
/* ------------------------------------------------------------------------ */
void orc_philox4x32_10(uint32_t out[4], const uint32_t ctr_in[4], const uint32_t key_in[2])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Rademacher sign mask D of the random Hadamard transform ([HTX] Experimento
 * de diagnostico: the randomized rotation flips signs at random before the
 * Hadamard transform; [MX] Metodologia 3).
 * Reading: one n_h-bit mask per call and orientation, shared by every block;
 * bit j set negates element j of each block.  Drawn from Philox with
 * key = seed and counter (0, 0, 0x5349474E, 0); the low n_h bits of word 0. */
uint32_t orc_sign_mask_from_seed(uint64_t seed, int n_h)
{
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {0u, 0u, 0x5349474Eu, 0u};
    uint32_t out[4];
    orc_philox4x32_10(out, ctr, key);
    if (n_h >= 32) return out[0];
    if (n_h <= 0) return 0u;
    return out[0] & ((1u << n_h) - 1u);
}

/* 16-bit uniform numerator for stochastic rounding of the element at index
 * idx of a stored copy (orient 0 = row-wise, 1 = column-wise).
 * Reading: Philox keyed by the seed, counter (lo32(idx>>3), hi32(idx>>3),
 * orient, 0); word (idx>>1)&3 of the output; its low half for even idx, its
 * high half for odd idx.  The uniform is r / 2^16. */
uint32_t orc_sr_uniform16(uint64_t seed, uint64_t idx, uint32_t orient)
{
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint64_t blk = idx >> 3;
    uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), orient, 0u};
    uint32_t out[4];
    orc_philox4x32_10(out, ctr, key);
    uint32_t w = out[(idx >> 1) & 3];
    return (idx & 1) ? (w >> 16) : (w & 0xFFFFu);
}

/* ------------------------------------------------------------------------ */
/* Blockwise Hadamard rotation ([MX] Metodologia 3: deterministic 16x16 and  */
/* 32x32 Hadamard; [SB] Metodologia 1: random Hadamard transform).           */
/* Reading: y = c_n * H_n * D * u, H_n in Sylvester (natural) order, the     */
/* sign flips D applied first, the butterfly stages in ascending stride, one */
/* final multiply by c_16 = 1/4 or c_32 = fl32(1/sqrt(32)).                  */
/* ------------------------------------------------------------------------ */
static float rot_scale(int n)
{
    if (n == 16) return 0.25f;
    /* 1/sqrt(32) rounded once to fp32 (0x3E3504F3). */
    return (float)(1.0 / sqrt(32.0));
}

void orc_rotate_block(float *u, int n, uint32_t sign_mask)
{
    for (int j = 0; j < n; ++j)
        if ((sign_mask >> j) & 1u) u[j] = -u[j];
    for (int h = 1; h < n; h <<= 1) {
        for (int i = 0; i < n; ++i) {
            if (i & h) continue;
            float a = u[i], b = u[i + h];
            u[i] = a + b;
            u[i + h] = a - b;
        }
    }
    float c = rot_scale(n);
    for (int j = 0; j < n; ++j) u[j] = u[j] * c;
}

/* Inverse of orc_rotate_block up to the rounding of c_32: the same butterfly
 * and scale, then the sign flips (H_n * H_n = n I, c_n^2 * n = 1). */
void orc_unrotate_block(float *u, int n, uint32_t sign_mask)
{
    for (int h = 1; h < n; h <<= 1) {
        for (int i = 0; i < n; ++i) {
            if (i & h) continue;
            float a = u[i], b = u[i + h];
            u[i] = a + b;
            u[i + h] = a - b;
        }
    }
    float c = rot_scale(n);
    for (int j = 0; j < n; ++j) u[j] = u[j] * c;
    for (int j = 0; j < n; ++j)
        if ((sign_mask >> j) & 1u) u[j] = -u[j];
}

/* ------------------------------------------------------------------------ */
/* Rounding onto the grid                                                   */
/* ------------------------------------------------------------------------ */
/* Round-to-nearest-even onto the grid ([SB] Declaracao do Problema and
 * Metodologia 2: RTNE for every operand but dY; [HTX] Que es MXFP4?: each
 * element is the nearest value the 4-bit format can represent).
 * Magnitudes at or above q_max saturate to code 7.  An exact tie between
 * levels k and k+1 goes to the even code.  The sign bit is the sign of v, so
 * a negative value that rounds to zero keeps its sign (code 8). */
int orc_round_rtne(int grid, float v)
{
    int sign = signbit(v) ? 8 : 0;
    float a = fabsf(v);
    int top = orc_grid_top(grid);
    float qmax = orc_grid_qmax(grid);
    if (!(a < qmax)) return sign | top;
    for (int k = 0; k < top; ++k) {
        float lo = orc_grid_level(grid, k), hi = orc_grid_level(grid, k + 1);
        float mid = (lo + hi) * 0.5f; /* exact for every grid */
        if (a < mid) return sign | k;
        if (a == mid) return sign | ((k & 1) ? k + 1 : k);
    }
    return sign | top;
}

/* Stochastic rounding ([SB] Metodologia 2: SR on dY only, to preserve the
 * gradient's expectation; [HTX] Experimento de diagnostico: SR makes the
 * expected rounding error zero).  With g_k <= |v| < g_{k+1} and
 * f = (|v| - g_k)/(g_{k+1} - g_k), round up iff r/2^16 < f, r the 16-bit
 * uniform numerator.  Saturates at q_max like RTNE. */
int orc_round_sr(int grid, float v, uint32_t r16)
{
    int sign = signbit(v) ? 8 : 0;
    float a = fabsf(v);
    int top = orc_grid_top(grid);
    float qmax = orc_grid_qmax(grid);
    if (!(a < qmax)) return sign | top;
    for (int k = 0; k < top; ++k) {
        float lo = orc_grid_level(grid, k), hi = orc_grid_level(grid, k + 1);
        if (a >= lo && a < hi) {
            float f = (a - lo) / (hi - lo); /* exact: Sterbenz and a power-of-two gap */
            float u = (float)r16 * (1.0f / 65536.0f);
            return sign | (u < f ? k + 1 : k);
        }
    }
    return sign | top;
}

/* ------------------------------------------------------------------------ */
/* One quantized copy                                                       */
/* ------------------------------------------------------------------------ */
/* Quantize one stored copy of an R x C bf16 matrix (row stride ld elements).
 *
 *   orient = 0: row-wise copy.  Rotation and quant blocks run along C; the
 *               codes are stored R x C/2 bytes, scales R x C/b bytes.
 *   orient = 1: column-wise copy.  Blocks run along R; the copy is stored
 *               transposed (C x R/2 code bytes, C x R/b scale bytes).  It is
 *               formed by transposing the input and quantizing its rows.
 *
 *   grid      ORC_GRID_E2M1, ORC_GRID_E1M2 or ORC_GRID_E2M1_R4
 *   scale     ORC_SCALE_MX: b = 32, E8M0 shared exponent ([HTX] Que es MXFP4?)
 *             ORC_SCALE_NV: b = 16, E4M3 block scale, fp32 tensor scale,
 *             v = y * fl(1 / (sb * S_t)) per element
 *   n_h       0 (no rotation), 16 or 32
 *   sign_mask bit j negates element j of every n_h block (0 = deterministic H)
 *   round     ORC_RTNE or ORC_SR (SR uses sr_seed and the stored index)
 *   given_amax NV only: NULL to compute the global amax of the rotated copy,
 *             else a pointer to the caller's value
 *   codes     out, packed nibbles: element 2t in the low nibble of byte t
 *   scales    out, one byte per block, row-major [rows][cols/b] of the copy
 *   tensor_scale  out (NV only): S_t
 *   e4m3_bytes optional out: one E4M3 byte per element holding the exact
 *             value of its code (an 8-bit GEMM-ready copy), or NULL
 *
 * Returns ORC_OK, ORC_BAD_ARG or ORC_NONFINITE (an input is NaN/Inf).
 */
int orc_quantize(const uint16_t *x, int64_t R, int64_t C, int64_t ld, int orient,
                 int grid, int scale, int n_h, uint32_t sign_mask, int round,
                 uint64_t sr_seed, const float *given_amax,
                 uint8_t *codes, uint8_t *scales, float *tensor_scale, uint8_t *e4m3_bytes)
{
    int b = (scale == ORC_SCALE_MX) ? 32 : 16;
    if (n_h != 0 && n_h != 16 && n_h != 32) return ORC_BAD_ARG;
    if (R < 0 || C < 0 || ld < C) return ORC_BAD_ARG;

    /* The copy's own rows (rows_out x len): the input rows, or its columns. */
    int64_t rows_out = orient ? C : R;
    int64_t len = orient ? R : C;
    if (len % b != 0) return ORC_BAD_ARG;
    if (n_h && len % n_h != 0) return ORC_BAD_ARG;

    /* Step 1: bf16 -> fp32 (exact), arranged as the copy's rows. */
    float *y = (float *)malloc(sizeof(float) * (size_t)(rows_out * len > 0 ? rows_out * len : 1));
    if (!y) return ORC_BAD_ARG;
    for (int64_t i = 0; i < R; ++i) {
        for (int64_t j = 0; j < C; ++j) {
            float v = orc_bf16_to_f32(x[i * ld + j]);
            if (!isfinite(v)) { free(y); return ORC_NONFINITE; }
            if (orient == 0) y[i * len + j] = v;
            else y[j * len + i] = v;
        }
    }

    /* Step 2: sign flips and Hadamard rotation of each n_h block. */
    if (n_h) {
        for (int64_t r = 0; r < rows_out; ++r)
            for (int64_t j0 = 0; j0 < len; j0 += n_h)
                orc_rotate_block(&y[r * len + j0], n_h, sign_mask);
    }

    /* Step 3 (NV only): the fp32 tensor scale from the global amax G of the
     * rotated copy.  Reading: S_t = G / (448 * q_max), so that the block
     * holding G gets the largest E4M3 scale. */
    float qmax = orc_grid_qmax(grid);
    float S_t = 0.0f;
    if (scale == ORC_SCALE_NV) {
        float G = 0.0f;
        if (given_amax) {
            G = *given_amax;
        } else {
            for (int64_t t = 0; t < rows_out * len; ++t) {
                float a = fabsf(y[t]);
                if (a > G) G = a;
            }
        }
        float denom = 448.0f * qmax; /* 2688 or 784, exact */
        S_t = G / denom;
        if (tensor_scale) *tensor_scale = S_t;
    }

    int64_t nblk = len / b;
    for (int64_t r = 0; r < rows_out; ++r) {
        for (int64_t kb = 0; kb < nblk; ++kb) {
            float *blk = &y[r * len + kb * b];

            /* Step 4: block amax. */
            float m = 0.0f;
            for (int t = 0; t < b; ++t) {
                float a = fabsf(blk[t]);
                if (a > m) m = a;
            }

            /* Step 5: scale.  v_t = y_t / scale. */
            float vmul = 0.0f;   /* MX: exact power of two 2^-e; NV: 1 / (sb * S_t) */
            int zero_block = 0;
            uint8_t sbyte;
            if (scale == ORC_SCALE_MX) {
                /* E8M0 shared exponent ([HTX] Que es MXFP4?: the block's shared
                 * exponent, 8-bit E8M0).  Reading: e = floor(log2 m) - e_max,
                 * clamped to [-127, 127]; all-zero blocks take e = -127.  This
                 * puts the block maximum at [2^e_max, 2^(e_max+1)) in grid
                 * units, so every grid level is reachable. */
                int e;
                if (m == 0.0f) {
                    e = -127;
                } else {
                    int ex;
                    (void)frexpf(m, &ex); /* m = f * 2^ex, f in [0.5, 1) */
                    e = (ex - 1) - orc_grid_emax(grid);
                    if (e < -127) e = -127;
                    if (e > 127) e = 127;
                }
                sbyte = (uint8_t)(e + 127);
                vmul = ldexpf(1.0f, -e);
            } else {
                /* E4M3 block scale = amax / q_max relative to S_t.
                 * Reading: the pages only name NVFP4; the element step uses the
                 * block's reciprocal dequantization step r = fl(1 / (sb * S_t))
                 * (one division per block, v = fl(y * r)); an infinite r is
                 * replaced by the largest finite float. */
                if (S_t > 0.0f) {
                    float t1 = m / qmax;
                    float t2 = t1 / S_t;
                    sbyte = orc_e4m3_encode(t2);
                } else {
                    sbyte = 0;
                }
                if (sbyte == 0) {
                    zero_block = 1;
                } else {
                    float d = orc_e4m3_decode(sbyte) * S_t;
                    vmul = 1.0f / d;
                    if (isinf(vmul)) vmul = FLT_MAX;
                }
            }
            scales[r * nblk + kb] = sbyte;

            /* Step 6: round every element of the block onto the grid. */
            for (int t = 0; t < b; ++t) {
                int64_t col = kb * b + t;
                int64_t idx = r * len + col; /* index in the stored copy */
                int code;
                if (zero_block) {
                    code = signbit(blk[t]) ? 8 : 0;
                } else {
                    float v = blk[t] * vmul;
                    if (round == ORC_SR)
                        code = orc_round_sr(grid, v, orc_sr_uniform16(sr_seed, (uint64_t)idx, (uint32_t)orient));
                    else
                        code = orc_round_rtne(grid, v);
                }
                /* Step 7: pack two codes per byte, even element low. */
                uint8_t *byte = &codes[idx >> 1];
                if ((idx & 1) == 0) *byte = (uint8_t)((*byte & 0xF0) | code);
                else *byte = (uint8_t)((*byte & 0x0F) | (code << 4));
                if (e4m3_bytes) {
                    float g = orc_grid_level(grid, code & 7);
                    e4m3_bytes[idx] = (uint8_t)(orc_e4m3_encode(g) | ((code & 8) ? 0x80 : 0));
                }
            }
        }
    }
    free(y);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequantization ([HTX] Que es MXFP4?: reconstruction x = 2^E * Q(x/2^E))   */
/* ------------------------------------------------------------------------ */
/* Reconstruct one stored copy (rows x cols of the copy itself) in fp32.
 *   MX:  x = g[k] * 2^(byte-127), exact in fp32.
 *   NV:  x = fl(fl(g[k] * sb) * S_t); with_tensor_scale = 0 leaves out S_t.
 * With n_h > 0 and unrotate = 1 the inverse rotation is applied per block. */
void orc_dequantize(const uint8_t *codes, const uint8_t *scales, float tensor_scale,
                    int64_t rows, int64_t cols, int grid, int scale, int with_tensor_scale,
                    int n_h, uint32_t sign_mask, int unrotate, float *out)
{
    int b = (scale == ORC_SCALE_MX) ? 32 : 16;
    int64_t nblk = cols / b;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            int64_t idx = r * cols + c;
            int code = (codes[idx >> 1] >> ((idx & 1) * 4)) & 15;
            float g = orc_code_value(grid, code);
            uint8_t sb = scales[r * nblk + c / b];
            float v;
            if (scale == ORC_SCALE_MX) {
                v = g * ldexpf(1.0f, (int)sb - 127);
            } else {
                v = g * orc_e4m3_decode(sb);
                if (with_tensor_scale) v = v * tensor_scale;
            }
            out[idx] = v;
        }
        if (n_h && unrotate)
            for (int64_t c0 = 0; c0 < cols; c0 += n_h)
                orc_unrotate_block(&out[r * cols + c0], n_h, sign_mask);
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM entries ([HTX] Experimento de diagnostico: Fprop Y = X W^T, Dgrad    */
/* dX = dY W, Wgrad dW = dY^T X; every operand stored K-major so each is     */
/* D = A B^T).  fp64 dot products of dequantized operands.                   */
/* ------------------------------------------------------------------------ */
void orc_gemm_entries(const float *A, const float *B, int64_t K, double alpha,
                      const int64_t *ii, const int64_t *jj, int64_t n, double *out)
{
    for (int64_t t = 0; t < n; ++t) {
        const float *a = &A[ii[t] * K];
        const float *bb = &B[jj[t] * K];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += (double)a[k] * (double)bb[k];
        out[t] = alpha * s;
    }
}

/* ------------------------------------------------------------------------ */
/* Bias statistics ([SB] Metodologia 1: attenuation factor alpha < 1;        */
/* Resultados: SQNR and the shift of magnitudes).                            */
/* sums[0] = sum ref^2, sums[1] = sum (ref - approx)^2,                      */
/* sums[2] = sum ref*approx, sums[3] = sum |ref|,                            */
/* sums[4] = sum (|approx| - |ref|); hist[16] counts the packed codes.       */
/* ------------------------------------------------------------------------ */
void orc_bias_sums(const float *ref, const float *approx, int64_t n,
                   const uint8_t *codes, double *sums, uint64_t *hist)
{
    double s0 = 0, s1 = 0, s2 = 0, s3 = 0, s4 = 0;
    for (int64_t t = 0; t < n; ++t) {
        double r = ref[t], a = approx[t];
        s0 += r * r;
        s1 += (r - a) * (r - a);
        s2 += r * a;
        s3 += fabs(r);
        s4 += fabs(a) - fabs(r);
    }
    sums[0] = s0; sums[1] = s1; sums[2] = s2; sums[3] = s3; sums[4] = s4;
    if (hist) {
        for (int c = 0; c < 16; ++c) hist[c] = 0;
        if (codes)
            for (int64_t t = 0; t < n; ++t) hist[(codes[t >> 1] >> ((t & 1) * 4)) & 15] += 1;
    }
}

/* ------------------------------------------------------------------------ */
/* Rounding error in grid units, per level ([SB] Metodologia 1, "Origem      */
/* Geometrica": the expected error of the elements that round to level q_i, */
/* (l_i - r_i)/2 under a uniform density, is negative where the level's bin  */
/* is wider above it than below).                                          */
/* ------------------------------------------------------------------------ */
/* For the row-wise copy (codes, plain scales, tensor scale) of the R x C bf16
 * matrix x: every element's position v = y * step^-1 in grid units (y the
 * rotated value, the element step exactly as orc_quantize computes it), its
 * code's level g[k], k = code & 7, and per level k the sum of g[k] - |v| in
 * fp64 (sums[k]) and the number of elements (counts[k]).  Elements of a block
 * whose NV scale byte is 0 have v = 0. */
void orc_grid_error(const uint16_t *x, int64_t R, int64_t C, int64_t ld, int grid, int scale, int n_h,
                    uint32_t sign_mask, const uint8_t *codes, const uint8_t *scales, float tensor_scale,
                    double *sums, uint64_t *counts)
{
    int b = (scale == ORC_SCALE_MX) ? 32 : 16;
    int64_t nblk = C / b;
    float *y = (float *)malloc(sizeof(float) * (size_t)(C > 0 ? C : 1));
    if (!y) return;
    for (int k = 0; k < 8; ++k) { sums[k] = 0.0; counts[k] = 0; }
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t j = 0; j < C; ++j) y[j] = orc_bf16_to_f32(x[r * ld + j]);
        if (n_h)
            for (int64_t j0 = 0; j0 < C; j0 += n_h) orc_rotate_block(&y[j0], n_h, sign_mask);
        for (int64_t kb = 0; kb < nblk; ++kb) {
            uint8_t sb = scales[r * nblk + kb];
            float vmul;
            if (scale == ORC_SCALE_MX) {
                vmul = ldexpf(1.0f, 127 - (int)sb);
            } else if (sb == 0 || !(tensor_scale > 0.0f)) {
                vmul = 0.0f;
            } else {
                float d = orc_e4m3_decode(sb) * tensor_scale;
                vmul = 1.0f / d;
                if (isinf(vmul)) vmul = FLT_MAX;
            }
            for (int t = 0; t < b; ++t) {
                int64_t idx = r * C + kb * b + t;
                int code = (codes[idx >> 1] >> ((idx & 1) * 4)) & 15;
                float v = y[kb * b + t] * vmul;
                int k = code & 7;
                sums[k] += (double)orc_grid_level(grid, k) - fabs((double)v);
                counts[k] += 1;
            }
        }
    }
    free(y);
}

/* Mean signed relative error of approx against ref over the elements with
 * ref != 0: sums[0] = sum (|approx| - |ref|) / |ref| (each term in fp64),
 * sums[1] = their number.  The per-element form of the shrinkage, reported
 * beside the aggregate sum(|approx| - |ref|) / sum |ref|. */
void orc_rel_error_sums(const float *ref, const float *approx, int64_t n, double *sums)
{
    double s = 0.0, c = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        double r = ref[t], a = approx[t];
        if (r != 0.0) {
            s += (fabs(a) - fabs(r)) / fabs(r);
            c += 1.0;
        }
    }
    sums[0] = s;
    sums[1] = c;
}
