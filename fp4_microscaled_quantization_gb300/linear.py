"""One linear layer's three training GEMMs in 4 bits, under a named recipe.

Host-side orchestration only: every quantization and GEMM is one call into
libfp4q.so through the binding (fp4q.py).

Recipes ("Repensando o Vies de Encolhimento", Metodologia 2, "A Receita UFP4";
HTX article on arXiv 2605.09825, "Experimento de diagnostico"):

  ufp4   E1M2 grid for X, W and dY; random Hadamard H16 on the operands of all
         three GEMMs; RTNE for X and W, stochastic rounding for dY.  The E1M2
         GEMMs run on the exact E4M3 byte copies (kind::mxf8f6f4).
  e2m1   E2M1 grid (MXFP4); the rotation only on the Wgrad operands (the
         column-wise copies of dY and X), as the earlier E2M1 recipes do;
         RTNE for X and W, stochastic rounding for dY.

The rotation of the two operands of one GEMM uses the same sign mask along the
contraction axis, so the rotation cancels in the product: X-row and W-row share
mask_K (d_in), dY-row and W-col share mask_N (d_out), dY-col and X-col share
mask_M (tokens).

Shapes: X [M, K] (tokens x d_in), W [N, K] (d_out x d_in), dY [M, N].
Fprop Y = X W^T [M, N]; Dgrad dX = dY W [M, K]; Wgrad dW = dY^T X [N, K].
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import fp4q

RECIPES = ("ufp4", "e2m1")


@dataclass
class LayerResult:
    Y: torch.Tensor
    dX: torch.Tensor
    dW: torch.Tensor
    copies: dict


class Fp4Linear:
    """Quantize X, W, dY and run Fprop / Dgrad / Wgrad under one recipe."""

    def __init__(self, recipe: str = "ufp4", seed: int = 1005, n_h: int = 16, out_f32: bool = False):
        if recipe not in RECIPES:
            raise ValueError(f"recipe must be one of {RECIPES}")
        self.recipe = recipe
        self.n_h = n_h
        self.out_f32 = out_f32
        self.mask_K = fp4q.sign_mask_from_seed(seed, n_h)
        self.mask_N = fp4q.sign_mask_from_seed(seed + 1, n_h)
        self.mask_M = fp4q.sign_mask_from_seed(seed + 2, n_h)
        self.sr_seed = seed + 3
        self.grid = fp4q.GRID_E1M2 if recipe == "ufp4" else fp4q.GRID_E2M1

    # -------------------------------------------------------------- configs
    def _cfg(self, mask_row: int, mask_col: int, rot: int, sr: bool, row: bool, col: bool) -> fp4q.Config:
        return fp4q.Config(grid=self.grid, scale=fp4q.SCALE_MX, rot=rot, round=fp4q.SR if sr else fp4q.RTNE,
                           sign_mask_row=mask_row, sign_mask_col=mask_col, sr_seed=self.sr_seed,
                           want_row=row, want_col=col, sf_layout=fp4q.SF_MMA,
                           emit_e4m3=(self.grid == fp4q.GRID_E1M2))

    def _quantize(self, x: torch.Tensor, mask_row: int, mask_col: int, sr: bool, rot_row: bool, rot_col: bool,
                  stream=None):
        """Row-wise and column-wise copies of x; each copy rotated or not."""
        H = self.n_h
        if rot_row == rot_col:
            rot = H if rot_row else fp4q.ROT_NONE
            mr, mc = (mask_row, mask_col) if rot_row else (0, 0)
            return fp4q.rht_quantize(x, self._cfg(mr, mc, rot, sr, True, True), stream=stream)
        row, _ = fp4q.rht_quantize(x, self._cfg(mask_row if rot_row else 0, 0, H if rot_row else fp4q.ROT_NONE,
                                                sr, True, False), stream=stream)
        _, col = fp4q.rht_quantize(x, self._cfg(0, mask_col if rot_col else 0, H if rot_col else fp4q.ROT_NONE,
                                                sr, False, True), stream=stream)
        return row, col

    def quantize_all(self, X, W, dY, stream=None) -> dict:
        every = self.recipe == "ufp4"
        # e2m1: only the Wgrad operands (column-wise copies of X and dY) are rotated
        Xr, Xc = self._quantize(X, self.mask_K, self.mask_M, False, every, True, stream)
        Wr, Wc = self._quantize(W, self.mask_K, self.mask_N, False, every, every, stream)
        Gr, Gc = self._quantize(dY, self.mask_N, self.mask_M, True, every, True, stream)
        return {"Xr": Xr, "Xc": Xc, "Wr": Wr, "Wc": Wc, "Gr": Gr, "Gc": Gc}

    def gemms(self, q: dict, stream=None):
        g = self.grid
        kw = dict(want_bf16=True, want_f32=self.out_f32, stream=stream)
        Yb, Yf = fp4q.gemm(q["Xr"], q["Wr"], g, fp4q.SCALE_MX, **kw)      # Fprop  [M, N]
        # the backward GEMMs, Dgrad [M, K] and Wgrad [N, K], in one balanced launch
        (dXb, dXf), (dWb, dWf) = fp4q.gemm_group([(q["Gr"], q["Wc"]), (q["Gc"], q["Xc"])], g, fp4q.SCALE_MX, **kw)
        if self.out_f32:
            return Yf, dXf, dWf
        return Yb, dXb, dWb

    def __call__(self, X, W, dY, stream=None) -> LayerResult:
        q = self.quantize_all(X, W, dY, stream)
        Y, dX, dW = self.gemms(q, stream)
        return LayerResult(Y, dX, dW, q)


def reference_gemms(X: torch.Tensor, W: torch.Tensor, dY: torch.Tensor):
    """The three GEMMs of the unquantized bf16 operands in fp32 (the quality
    reference of the recipe comparison; cuBLAS through torch, not the path)."""
    Xf, Wf, dYf = X.float(), W.float(), dY.float()
    return Xf @ Wf.T, dYf @ Wf, dYf.T @ Xf


def output_quality(result: LayerResult, ref) -> dict:
    """SQNR (dB) and attenuation alpha of each GEMM output against the reference,
    computed on the device by the bias-statistics kernel."""
    out = {}
    for name, got, want in zip(("fprop", "dgrad", "wgrad"), (result.Y, result.dX, result.dW), ref):
        s = fp4q.bias_stats(want.contiguous().view(-1), got.float().contiguous().view(-1))
        out[name] = {"sqnr_db": s["sqnr_db"], "alpha": s["alpha"], "shrinkage": s["shrinkage"]}
    return out
