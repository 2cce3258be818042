"""Plain CPU oracle for the fused Hadamard + 4-bit microscaled quantizer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product path never imports it.  It
shares no code with the CUDA library.  The arithmetic lives in ``oracle.c``
(single-threaded C, fp32 steps with contraction off, fp64 sums); this module
only compiles it with gcc, marshals numpy arrays and, for the full GEMM, calls
numpy's fp64 matrix product as a library step.

Parity status of each function (pins live in tests/test_oracle_*.py):
  grid tables, E4M3 codec, Philox4x32-10, rotation, RTNE, SR, MX and NV
  scales, dequantize, GEMM entries, bias sums, effective bucket ratio, the
  per-level error in grid units and the per-element relative error -- pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

GRID_E2M1, GRID_E1M2, GRID_E2M1_R4 = 0, 1, 2
SCALE_MX, SCALE_NV = 0, 1
RTNE, SR = 0, 1

_CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-fexcess-precision=standard"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, u32, u64 = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
        L.orc_grid_level.restype = ctypes.c_float
        L.orc_grid_level.argtypes = [i32, i32]
        L.orc_grid_qmax.restype = ctypes.c_float
        L.orc_grid_qmax.argtypes = [i32]
        L.orc_grid_emax.restype = i32
        L.orc_grid_emax.argtypes = [i32]
        L.orc_grid_top.restype = i32
        L.orc_grid_top.argtypes = [i32]
        L.orc_code_value.restype = ctypes.c_float
        L.orc_code_value.argtypes = [i32, i32]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_e4m3_decode.restype = ctypes.c_float
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_philox4x32_10.restype = None
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_sign_mask_from_seed.restype = u32
        L.orc_sign_mask_from_seed.argtypes = [u64, i32]
        L.orc_sr_uniform16.restype = u32
        L.orc_sr_uniform16.argtypes = [u64, u64, u32]
        L.orc_rotate_block.restype = None
        L.orc_rotate_block.argtypes = [P, i32, u32]
        L.orc_unrotate_block.restype = None
        L.orc_unrotate_block.argtypes = [P, i32, u32]
        L.orc_round_rtne.restype = i32
        L.orc_round_rtne.argtypes = [i32, ctypes.c_float]
        L.orc_round_sr.restype = i32
        L.orc_round_sr.argtypes = [i32, ctypes.c_float, u32]
        L.orc_quantize.restype = i32
        L.orc_quantize.argtypes = [P, i64, i64, i64, i32, i32, i32, i32, u32, i32, u64, P, P, P, P, P]
        L.orc_dequantize.restype = None
        L.orc_dequantize.argtypes = [P, P, ctypes.c_float, i64, i64, i32, i32, i32, i32, u32, i32, P]
        L.orc_gemm_entries.restype = None
        L.orc_gemm_entries.argtypes = [P, P, i64, ctypes.c_double, P, P, i64, P]
        L.orc_bias_sums.restype = None
        L.orc_bias_sums.argtypes = [P, P, i64, P, P, P]
        L.orc_grid_error.restype = None
        L.orc_grid_error.argtypes = [P, i64, i64, i64, i32, i32, i32, u32, P, P, ctypes.c_float, P, P]
        L.orc_rel_error_sums.restype = None
        L.orc_rel_error_sums.argtypes = [P, P, i64, P]
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- scalars
def grid_levels(grid: int) -> np.ndarray:
    return np.array([lib().orc_grid_level(grid, k) for k in range(8)], dtype=np.float32)


def grid_qmax(grid: int) -> float:
    return float(lib().orc_grid_qmax(grid))


def grid_emax(grid: int) -> int:
    return int(lib().orc_grid_emax(grid))


def grid_top(grid: int) -> int:
    return int(lib().orc_grid_top(grid))


def code_value(grid: int, code: int) -> float:
    return float(lib().orc_code_value(grid, code))


def e4m3_encode(x: float) -> int:
    return int(lib().orc_e4m3_encode(float(x)))


def e4m3_decode(b: int) -> float:
    return float(lib().orc_e4m3_decode(int(b)))


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(out), _ptr(c), _ptr(k))
    return out


def sign_mask_from_seed(seed: int, n_h: int) -> int:
    return int(lib().orc_sign_mask_from_seed(seed, n_h))


def sr_uniform16(seed: int, idx: int, orient: int) -> int:
    return int(lib().orc_sr_uniform16(seed, idx, orient))


def rotate_block(u, n_h: int, sign_mask: int = 0) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(u, dtype=np.float32).copy())
    assert v.size == n_h
    lib().orc_rotate_block(_ptr(v), n_h, sign_mask)
    return v


def unrotate_block(u, n_h: int, sign_mask: int = 0) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(u, dtype=np.float32).copy())
    lib().orc_unrotate_block(_ptr(v), n_h, sign_mask)
    return v


def round_rtne(grid: int, v: float) -> int:
    return int(lib().orc_round_rtne(grid, float(v)))


def round_sr(grid: int, v: float, r16: int) -> int:
    return int(lib().orc_round_sr(grid, float(v), int(r16)))


# ---------------------------------------------------------------- arrays
class OracleError(RuntimeError):
    pass


def quantize(x_bf16: np.ndarray, orient: int, grid: int, scale: int, n_h: int,
             sign_mask: int = 0, round_mode: int = RTNE, sr_seed: int = 0,
             given_amax: float | None = None, want_e4m3: bool = False) -> dict:
    """Quantize one stored copy of the bf16 matrix ``x_bf16`` (uint16 bits).

    orient 0: row-wise copy (R x C/2 codes); orient 1: column-wise copy stored
    transposed (C x R/2 codes).  Returns codes, scales, tensor_scale and the
    optional E4M3 bytes.
    """
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, C = x.shape
    rows, cols = (C, R) if orient else (R, C)
    b = 32 if scale == SCALE_MX else 16
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows, cols // b), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    e4 = np.zeros((rows, cols), dtype=np.uint8) if want_e4m3 else None
    ga = None if given_amax is None else np.array([given_amax], dtype=np.float32)
    rc = lib().orc_quantize(_ptr(x), R, C, C, orient, grid, scale, n_h, sign_mask, round_mode,
                            sr_seed, _ptr(ga), _ptr(codes), _ptr(scales), _ptr(ts), _ptr(e4))
    if rc != 0:
        raise OracleError(f"orc_quantize returned {rc}")
    return {"codes": codes, "scales": scales, "tensor_scale": float(ts[0]), "e4m3": e4}


def dequantize(codes: np.ndarray, scales: np.ndarray, tensor_scale: float, grid: int, scale: int,
               with_tensor_scale: bool = True, n_h: int = 0, sign_mask: int = 0,
               unrotate: bool = False) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows = codes.shape[0]
    cols = codes.shape[1] * 2
    out = np.zeros((rows, cols), dtype=np.float32)
    lib().orc_dequantize(_ptr(codes), _ptr(scales), float(tensor_scale), rows, cols, grid, scale,
                         int(with_tensor_scale), n_h, sign_mask, int(unrotate), _ptr(out))
    return out


def gemm_ref(A_deq: np.ndarray, B_deq: np.ndarray, alpha: float = 1.0) -> np.ndarray:
    """D = alpha * A B^T in fp64 (numpy's fp64 matrix product as the step)."""
    return alpha * (A_deq.astype(np.float64) @ B_deq.astype(np.float64).T)


def gemm_entries(A_deq: np.ndarray, B_deq: np.ndarray, ii, jj, alpha: float = 1.0) -> np.ndarray:
    """Sampled entries D[i, j] = alpha * sum_k A[i, k] B[j, k], one fp64 dot each."""
    A = np.ascontiguousarray(A_deq, dtype=np.float32)
    B = np.ascontiguousarray(B_deq, dtype=np.float32)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    out = np.zeros(ii.size, dtype=np.float64)
    lib().orc_gemm_entries(_ptr(A), _ptr(B), A.shape[1], float(alpha), _ptr(ii), _ptr(jj), ii.size, _ptr(out))
    return out


def bias_stats(ref: np.ndarray, approx: np.ndarray, codes: np.ndarray | None = None) -> dict:
    """SQNR (dB), attenuation alpha and shrinkage, from fp64 sums."""
    r = np.ascontiguousarray(ref, dtype=np.float32).ravel()
    a = np.ascontiguousarray(approx, dtype=np.float32).ravel()
    c = None if codes is None else np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    sums = np.zeros(5, dtype=np.float64)
    hist = np.zeros(16, dtype=np.uint64)
    lib().orc_bias_sums(_ptr(r), _ptr(a), r.size, _ptr(c), _ptr(sums), _ptr(hist))
    s_ref2, s_err2, s_ra, s_absref, s_absdiff = (float(v) for v in sums)
    sqnr = 10.0 * np.log10(s_ref2 / s_err2) if s_err2 > 0 else float("inf")
    alpha = s_ra / s_ref2 if s_ref2 > 0 else float("nan")
    shrink = s_absdiff / s_absref if s_absref > 0 else float("nan")
    return {"sums": sums, "hist": hist, "n": r.size, "sqnr_db": sqnr, "alpha": alpha, "shrinkage": shrink}


def grid_error(x_bf16: np.ndarray, grid: int, scale: int, n_h: int, sign_mask: int, codes: np.ndarray,
               scales: np.ndarray, tensor_scale: float = 0.0) -> dict:
    """Per level k: sum and count of g[k] - |v| (v in grid units) over the
    row-wise copy (plain scales) of x; the mean over all elements."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, C = x.shape
    sums = np.zeros(8, dtype=np.float64)
    counts = np.zeros(8, dtype=np.uint64)
    lib().orc_grid_error(_ptr(x), R, C, C, grid, scale, n_h, sign_mask,
                         _ptr(np.ascontiguousarray(codes, dtype=np.uint8)),
                         _ptr(np.ascontiguousarray(scales, dtype=np.uint8)), float(tensor_scale),
                         _ptr(sums), _ptr(counts))
    total = int(counts.sum())
    return {"sums": sums, "counts": counts, "mean": float(sums.sum() / total) if total else float("nan")}


def rel_error(ref: np.ndarray, approx: np.ndarray) -> dict:
    """Mean of (|approx| - |ref|) / |ref| over ref != 0 (fp64 sums)."""
    r = np.ascontiguousarray(ref, dtype=np.float32).ravel()
    a = np.ascontiguousarray(approx, dtype=np.float32).ravel()
    sums = np.zeros(2, dtype=np.float64)
    lib().orc_rel_error_sums(_ptr(r), _ptr(a), r.size, _ptr(sums))
    return {"sum": float(sums[0]), "count": int(sums[1]),
            "mean": float(sums[0] / sums[1]) if sums[1] else float("nan")}


def effective_bucket_ratio(hist16, grid: int) -> float:
    """Effective number of magnitude levels used, over the levels the grid can
    produce ("Repensando o Vies de Encolhimento", Resultados, Diagnosticos de
    Quantizacao e GEMM, names the ratio without a formula).  Reading: fold the
    16-code histogram onto the 8 magnitudes (code & 7), take the Shannon
    entropy H in nats of that distribution, and return exp(H) / L with L = 8
    (7 for the grid capped at 4, which has no code 7)."""
    counts = [0.0] * 8
    for code in range(16):
        counts[code & 7] += float(hist16[code])
    total = sum(counts)
    if total == 0:
        return float("nan")
    H = 0.0
    for c in counts:
        if c > 0:
            p = c / total
            H -= p * np.log(p)
    L = 7 if grid == GRID_E2M1_R4 else 8
    return float(np.exp(H) / L)
