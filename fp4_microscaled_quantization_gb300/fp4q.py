"""ctypes binding of libfp4q.so (include/fp4q.h), same names as the C ABI.

Argument marshalling only: every step of the method runs in the CUDA
library.  PyTorch supplies device memory (outputs are allocated here with
``torch.empty``) and the current CUDA stream.  There is no fallback: if the
library has not been built, or the call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp4q.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "fp4q.h")

# enums (values fixed by include/fp4q.h)
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_CUDA, ERR_WORKSPACE = range(6)
DEV_NONFINITE, DEV_TIMEOUT = 0x1, 0x2
GRID_E2M1, GRID_E1M2, GRID_E2M1_R4 = 0, 1, 2
SCALE_MX, SCALE_NV = 0, 1
ROT_NONE, ROT_H16, ROT_H32 = 0, 16, 32
RTNE, SR = 0, 1
SF_PLAIN, SF_MMA = 0, 1


class Fp4qError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: status {status} ({status_str(status)})")
        self.status = status


class CConfig(ctypes.Structure):
    _fields_ = [
        ("grid", ctypes.c_int32), ("scale", ctypes.c_int32), ("rot", ctypes.c_int32),
        ("round", ctypes.c_int32), ("sign_mask_row", ctypes.c_uint32), ("sign_mask_col", ctypes.c_uint32),
        ("sr_seed", ctypes.c_uint64), ("want_row", ctypes.c_int32), ("want_col", ctypes.c_int32),
        ("sf_layout", ctypes.c_int32), ("emit_e4m3", ctypes.c_int32), ("global_amax", ctypes.c_void_p),
    ]


class COperand(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("e4m3", ctypes.c_void_p)]


class CGemmProblem(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("D_bf16", ctypes.c_void_p), ("D_f32", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libfp4q.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m fp4_microscaled_quantization_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, u32, u64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                     ctypes.c_uint64, ctypes.c_size_t)
        L.fp4q_status_str.restype = ctypes.c_char_p
        L.fp4q_status_str.argtypes = [i32]
        L.fp4q_version.restype = i32
        L.fp4q_version.argtypes = []
        L.fp4q_sign_mask_from_seed.restype = u32
        L.fp4q_sign_mask_from_seed.argtypes = [u64, i32]
        L.fp4q_workspace_bytes.restype = sz
        L.fp4q_workspace_bytes.argtypes = [i64, i64, P]
        L.fp4q_rht_quantize.restype = i32
        L.fp4q_rht_quantize.argtypes = [P, i64, i64, i64, P, P, P, P, sz, P, P]
        L.fp4q_diag_workspace_bytes.restype = sz
        L.fp4q_diag_workspace_bytes.argtypes = []
        L.fp4q_grid_error.restype = i32
        L.fp4q_grid_error.argtypes = [P, i64, i64, i64, P, P, P, sz, P, P]
        L.fp4q_rel_error.restype = i32
        L.fp4q_rel_error.argtypes = [P, P, i64, P, sz, P, P]
        L.fp4q_test_quantize_wait_expiry.restype = i32
        L.fp4q_test_quantize_wait_expiry.argtypes = [P, i64, i64, i64, P, P, P, P, sz, P, i32, u32, P]
        L.fp4q_rotated_amax.restype = i32
        L.fp4q_rotated_amax.argtypes = [P, i64, i64, i64, P, P, P, P]
        L.fp4q_dequantize.restype = i32
        L.fp4q_dequantize.argtypes = [P, i64, i64, P, i32, i32, P, P]
        L.fp4q_gemm.restype = i32
        L.fp4q_gemm.argtypes = [P, P, i64, i64, i64, i32, i32, P, P, P, P]
        L.fp4q_gemm_quantize.restype = i32
        L.fp4q_gemm_quantize.argtypes = [P, P, i64, i64, i64, i32, i32, P, P, P, P, P]
        L.fp4q_gemm_group.restype = i32
        L.fp4q_gemm_group.argtypes = [P, i32, i32, i32, P, P]
        L.fp4q_bias_stats_workspace_bytes.restype = sz
        L.fp4q_bias_stats_workspace_bytes.argtypes = [i64]
        L.fp4q_bias_stats.restype = i32
        L.fp4q_bias_stats.argtypes = [P, P, i64, P, P, sz, P, P]
        L.fp4q_bias_stats_noalloc.restype = i32
        L.fp4q_bias_stats_noalloc.argtypes = [P, P, i64, P, P, P]
        L.fp4q_stats_finalize.restype = None
        L.fp4q_stats_finalize.argtypes = [P, P, P, P]
        L.fp4q_hadamard_rotate_bf16.restype = i32
        L.fp4q_hadamard_rotate_bf16.argtypes = [P, i64, i64, i64, i32, u32, u32, P, P, P]
        _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().fp4q_status_str(int(s)).decode()


def _check(fn: str, s: int):
    if s != OK:
        raise Fp4qError(fn, s)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _p(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


# ------------------------------------------------------------------ config
@dataclass
class Config:
    """Python mirror of fp4q_config (see include/fp4q.h)."""
    grid: int = GRID_E2M1
    scale: int = SCALE_MX
    rot: int = ROT_H16
    round: int = RTNE
    sign_mask_row: int = 0
    sign_mask_col: int = 0
    sr_seed: int = 0
    want_row: bool = True
    want_col: bool = True
    sf_layout: int = SF_PLAIN
    emit_e4m3: bool = False
    global_amax: torch.Tensor | None = None   # device float32[2] or None

    @property
    def block(self) -> int:
        return 32 if self.scale == SCALE_MX else 16

    def c(self) -> CConfig:
        return CConfig(self.grid, self.scale, self.rot, self.round, self.sign_mask_row & 0xFFFFFFFF,
                       self.sign_mask_col & 0xFFFFFFFF, self.sr_seed & (2 ** 64 - 1), int(self.want_row),
                       int(self.want_col), self.sf_layout, int(self.emit_e4m3), _p(self.global_amax))


@dataclass
class Operand:
    """One quantized copy (torch tensors on the device)."""
    codes: torch.Tensor            # uint8 [rows, cols/2]
    scales: torch.Tensor           # uint8 [rows, cols/b] (or the MMA layout, same size)
    tensor_scale: torch.Tensor | None = None   # float32 [1] (NV)
    e4m3: torch.Tensor | None = None           # uint8 [rows, cols]
    rows: int = 0
    cols: int = 0
    grid: int = GRID_E2M1
    scale: int = SCALE_MX
    sf_layout: int = SF_PLAIN
    extra: dict = field(default_factory=dict)

    def c(self) -> COperand:
        return COperand(_p(self.codes), _p(self.scales), _p(self.tensor_scale), _p(self.e4m3))


def alloc_operand(rows: int, cols: int, cfg: Config, device) -> Operand:
    b = cfg.block
    return Operand(
        codes=torch.empty((rows, cols // 2), dtype=torch.uint8, device=device),
        scales=torch.empty((rows, cols // b), dtype=torch.uint8, device=device),
        tensor_scale=torch.empty(1, dtype=torch.float32, device=device) if cfg.scale == SCALE_NV else None,
        e4m3=torch.empty((rows, cols), dtype=torch.uint8, device=device) if cfg.emit_e4m3 else None,
        rows=rows, cols=cols, grid=cfg.grid, scale=cfg.scale, sf_layout=cfg.sf_layout)


# ------------------------------------------------------------------ calls
def sign_mask_from_seed(seed: int, n_h: int) -> int:
    return int(lib().fp4q_sign_mask_from_seed(seed & (2 ** 64 - 1), n_h))


def workspace_bytes(rows: int, cols: int, cfg: Config) -> int:
    cc = cfg.c()
    return int(lib().fp4q_workspace_bytes(rows, cols, ctypes.byref(cc)))


def rht_quantize(x: torch.Tensor, cfg: Config, row_out: Operand | None = None, col_out: Operand | None = None,
                 workspace: torch.Tensor | None = None, status: torch.Tensor | None = None, stream=None):
    """Fused rotation + quantization of a 2-D bf16 CUDA tensor (row stride x.stride(0)).

    Returns (row_copy, col_copy); a copy not requested is None."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    dev = x.device
    if cfg.want_row and row_out is None:
        row_out = alloc_operand(R, C, cfg, dev)
    if cfg.want_col and col_out is None:
        col_out = alloc_operand(C, R, cfg, dev)
    need = workspace_bytes(R, C, cfg)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    cc = cfg.c()
    ro = row_out.c() if cfg.want_row else None
    co = col_out.c() if cfg.want_col else None
    s = lib().fp4q_rht_quantize(
        x.data_ptr(), R, C, x.stride(0), ctypes.byref(cc),
        ctypes.byref(ro) if ro is not None else None, ctypes.byref(co) if co is not None else None,
        _p(workspace), 0 if workspace is None else workspace.numel(), _p(status), _stream(stream))
    _check("fp4q_rht_quantize", s)
    return (row_out if cfg.want_row else None), (col_out if cfg.want_col else None)


def test_quantize_wait_expiry(x: torch.Tensor, cfg: Config, row_out: Operand, col_out: Operand | None,
                              status: torch.Tensor, stall_tile: int, wait_limit_us: int, stream=None):
    """fp4q_test_quantize_wait_expiry: fp4q_rht_quantize with CTA 0's wait for
    its tile stall_tile made to run out after wait_limit_us (tests the bounded
    waits; FP4Q_DEV_TIMEOUT is expected in `status`)."""
    R, C = x.shape
    need = workspace_bytes(R, C, cfg)
    workspace = torch.empty(need, dtype=torch.uint8, device=x.device) if need else None
    cc = cfg.c()
    ro = row_out.c() if cfg.want_row else None
    co = col_out.c() if cfg.want_col else None
    _check("fp4q_test_quantize_wait_expiry", lib().fp4q_test_quantize_wait_expiry(
        x.data_ptr(), R, C, x.stride(0), ctypes.byref(cc), ctypes.byref(ro) if ro is not None else None,
        ctypes.byref(co) if co is not None else None, _p(workspace), 0 if workspace is None else workspace.numel(),
        _p(status), stall_tile, wait_limit_us, _stream(stream)))


def rotated_amax(x: torch.Tensor, cfg: Config, out: torch.Tensor | None = None, status=None, stream=None):
    R, C = x.shape
    if out is None:
        out = torch.empty(2, dtype=torch.float32, device=x.device)
    cc = cfg.c()
    _check("fp4q_rotated_amax", lib().fp4q_rotated_amax(x.data_ptr(), R, C, x.stride(0), ctypes.byref(cc),
                                                         out.data_ptr(), _p(status), _stream(stream)))
    return out


def dequantize(q: Operand, cfg: Config, orient: int = 0, unrotate: bool = False, out=None, stream=None):
    if out is None:
        out = torch.empty((q.rows, q.cols), dtype=torch.float32, device=q.codes.device)
    cc = cfg.c()
    qc = q.c()
    _check("fp4q_dequantize", lib().fp4q_dequantize(ctypes.byref(qc), q.rows, q.cols, ctypes.byref(cc), orient,
                                                     int(unrotate), out.data_ptr(), _stream(stream)))
    return out


def gemm(A: Operand, B: Operand, grid: int, scale: int, want_bf16: bool = True, want_f32: bool = True,
         D_bf16=None, D_f32=None, status=None, stream=None):
    """D = alpha_g * A B^T for quantized copies A (M x K) and B (N x K)."""
    M, K = A.rows, A.cols
    N = B.rows
    dev = A.codes.device
    if want_bf16 and D_bf16 is None:
        D_bf16 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if want_f32 and D_f32 is None:
        D_f32 = torch.empty((M, N), dtype=torch.float32, device=dev)
    ac, bc = A.c(), B.c()
    _check("fp4q_gemm", lib().fp4q_gemm(ctypes.byref(ac), ctypes.byref(bc), M, N, K, grid, scale, _p(D_bf16),
                                         _p(D_f32), _p(status), _stream(stream)))
    return D_bf16, D_f32


def gemm_group(pairs, grid: int, scale: int, want_bf16: bool = True, want_f32: bool = False, outs=None,
               status=None, stream=None):
    """Several GEMMs D_i = alpha_g * A_i B_i^T of one recipe in one launch
    (fp4q_gemm_group).  pairs: [(A_i, B_i)]; outs: optional [(D_bf16, D_f32)].
    Returns [(D_bf16, D_f32)] per GEMM."""
    keep, probs, res = [], [], []
    for i, (A, B) in enumerate(pairs):
        M, K, N = A.rows, A.cols, B.rows
        dev = A.codes.device
        db, df = outs[i] if outs is not None else (None, None)
        if db is None and want_bf16:
            db = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if df is None and want_f32:
            df = torch.empty((M, N), dtype=torch.float32, device=dev)
        ac, bc = A.c(), B.c()
        keep += [ac, bc]
        probs.append(CGemmProblem(ctypes.addressof(ac), ctypes.addressof(bc), M, N, K, _p(db), _p(df)))
        res.append((db, df))
    arr = (CGemmProblem * len(probs))(*probs)
    _check("fp4q_gemm_group", lib().fp4q_gemm_group(ctypes.cast(arr, ctypes.c_void_p), len(probs), grid, scale,
                                                     _p(status), _stream(stream)))
    del keep
    return res


def gemm_quantize(A: Operand, B: Operand, grid: int, scale: int, out_cfg: Config, want_bf16: bool = False,
                  D_bf16=None, out: Operand | None = None, status=None, stream=None):
    """D = alpha_g * A B^T with the row-wise copy of bf16(D) under out_cfg made in
    the GEMM's epilogue.  Returns (D_bf16 or None, out)."""
    M, K = A.rows, A.cols
    N = B.rows
    dev = A.codes.device
    if want_bf16 and D_bf16 is None:
        D_bf16 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if out is None:
        out = alloc_operand(M, N, out_cfg, dev)
    ac, bc, oc, cc = A.c(), B.c(), out.c(), out_cfg.c()
    _check("fp4q_gemm_quantize", lib().fp4q_gemm_quantize(
        ctypes.byref(ac), ctypes.byref(bc), M, N, K, grid, scale, _p(D_bf16), ctypes.byref(cc), ctypes.byref(oc),
        _p(status), _stream(stream)))
    return D_bf16, out


def bias_stats_workspace_bytes(n: int) -> int:
    return int(lib().fp4q_bias_stats_workspace_bytes(n))


def bias_stats(ref: torch.Tensor, approx: torch.Tensor, codes: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, out: torch.Tensor | None = None, stream=None,
               sync: bool = True):
    """fp64 sums, SQNR, alpha and shrinkage of approx against ref (fp32 CUDA tensors)."""
    n = ref.numel()
    dev = ref.device
    if workspace is None:
        workspace = torch.empty(bias_stats_workspace_bytes(n), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(22, dtype=torch.float64, device=dev)
    _check("fp4q_bias_stats", lib().fp4q_bias_stats(ref.data_ptr(), approx.data_ptr(), n, _p(codes),
                                                     workspace.data_ptr(), workspace.numel(), out.data_ptr(),
                                                     _stream(stream)))
    if not sync:
        return out
    host = out.cpu()
    sums = host[:5].numpy().copy()
    ints = host.view(torch.int64)[5:].numpy().astype("uint64")
    sq, al, sh = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    lib().fp4q_stats_finalize(sums.ctypes.data_as(ctypes.c_void_p), ctypes.byref(sq), ctypes.byref(al),
                              ctypes.byref(sh))
    return {"sums": sums, "n": int(ints[0]), "hist": ints[1:17], "sqnr_db": sq.value, "alpha": al.value,
            "shrinkage": sh.value}


def grid_error(x: torch.Tensor, cfg: Config, row_copy: Operand, stream=None) -> dict:
    """fp4q_grid_error: per level k, sum and count of g[k] - |v| (grid units)
    over the row-wise copy of x; the overall mean."""
    R, C = x.shape
    ws = torch.empty(int(lib().fp4q_diag_workspace_bytes()), dtype=torch.uint8, device=x.device)
    out = torch.empty(16, dtype=torch.float64, device=x.device)
    cc, qc = cfg.c(), row_copy.c()
    _check("fp4q_grid_error", lib().fp4q_grid_error(x.data_ptr(), R, C, x.stride(0), ctypes.byref(cc),
                                                     ctypes.byref(qc), ws.data_ptr(), ws.numel(), out.data_ptr(),
                                                     _stream(stream)))
    h = out.cpu().numpy()
    sums, counts = h[:8].copy(), h[8:].astype("uint64")
    total = int(counts.sum())
    return {"sums": sums, "counts": counts, "mean": float(sums.sum() / total) if total else float("nan")}


def rel_error(ref: torch.Tensor, approx: torch.Tensor, stream=None) -> dict:
    """fp4q_rel_error: mean of (|approx| - |ref|) / |ref| over ref != 0."""
    ws = torch.empty(int(lib().fp4q_diag_workspace_bytes()), dtype=torch.uint8, device=ref.device)
    out = torch.empty(2, dtype=torch.float64, device=ref.device)
    _check("fp4q_rel_error", lib().fp4q_rel_error(ref.data_ptr(), approx.data_ptr(), ref.numel(), ws.data_ptr(),
                                                   ws.numel(), out.data_ptr(), _stream(stream)))
    s, c = out.cpu().tolist()
    return {"sum": s, "count": int(c), "mean": s / c if c else float("nan")}


def hadamard_rotate_bf16(x: torch.Tensor, rot: int, sign_mask_row: int = 0, sign_mask_col: int = 0,
                         want_row: bool = True, want_col: bool = True, y_row=None, y_col=None, stream=None):
    R, C = x.shape
    if want_row and y_row is None:
        y_row = torch.empty((R, C), dtype=torch.bfloat16, device=x.device)
    if want_col and y_col is None:
        y_col = torch.empty((R, C), dtype=torch.bfloat16, device=x.device)
    if not want_row:
        y_row = None
    if not want_col:
        y_col = None
    _check("fp4q_hadamard_rotate_bf16", lib().fp4q_hadamard_rotate_bf16(
        x.data_ptr(), R, C, x.stride(0), rot, sign_mask_row & 0xFFFFFFFF, sign_mask_col & 0xFFFFFFFF,
        _p(y_row), _p(y_col), _stream(stream)))
    return y_row, y_col
