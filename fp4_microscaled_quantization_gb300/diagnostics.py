"""Quantization and GEMM diagnostics built from the library's kernels.

Host orchestration only: every quantization, dequantization, GEMM and
statistics reduction is one call into libfp4q.so through the binding.  The
fp32 quality references (the unquantized product, the bf16 input widened to
fp32) are plain torch operations: they are the yardstick, not the path.

* ``effective_bucket_ratio`` -- how evenly a quantized tensor uses the levels
  of its grid ("Repensando o Vies de Encolhimento", Resultados, Diagnosticos de
  Quantizacao e GEMM: the rotation raises the effective bucket ratio of
  outlier-heavy tensors for both grids).  The page gives no formula; the
  reading here is the effective number of magnitude levels, exp of the Shannon
  entropy (natural log) of the sign-folded code histogram, divided by the
  number of magnitude levels the grid can produce (8; 7 for the grid capped
  at 4, which never produces level 6).
* ``quantizer_report`` / ``delta_sqnr_sweep`` -- SQNR, attenuation, shrinkage
  and bucket ratio of one quantized copy after the inverse rotation, and the
  SQNR change that the rotation brings at rising outlier strength (same
  section: E1M2 gains SQNR after the rotation, E2M1 often loses it), with the
  per-element mean signed relative error and the rounding error in grid
  units per level (Metodologia 1, "Origem Geometrica").
* ``depth_chain`` -- K quantized GEMMs in a row, each layer's attenuation
  alpha_k against the exact product of its own input, their product, the
  first-order form exp(-sum delta_k) with delta_k = 1 - alpha_k, and the
  end-to-end attenuation of the chain against the unquantized chain
  (Metodologia 1, "Impacto Sistemico": the per-GEMM factors compound
  multiplicatively over depth).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import fp4q, synth

GRID_NAMES = {fp4q.GRID_E2M1: "e2m1", fp4q.GRID_E1M2: "e1m2", fp4q.GRID_E2M1_R4: "e2m1_cap4"}


def grid_levels_reachable(grid: int) -> int:
    """Magnitude levels a grid can produce (the capped E2M1 grid never makes code 7)."""
    return 7 if grid == fp4q.GRID_E2M1_R4 else 8


def effective_bucket_ratio(hist16, grid: int) -> float:
    """exp(H) / L for the sign-folded code histogram (H in nats, L reachable levels)."""
    h = np.asarray(hist16, dtype=np.float64).reshape(16)
    mag = h[:8] + h[8:]
    total = mag.sum()
    if total == 0:
        return float("nan")
    p = mag[mag > 0] / total
    return float(math.exp(-(p * np.log(p)).sum()) / grid_levels_reachable(grid))


def quantizer_report(x: torch.Tensor, grid: int, rot: int, sign_mask: int = 0, scale: int = fp4q.SCALE_MX,
                     round_mode: int = fp4q.RTNE, sr_seed: int = 0, stream=None) -> dict:
    """Quantize the row-wise copy of the bf16 CUDA matrix x, dequantize it with
    the inverse rotation, and compare with x on the device."""
    cfg = fp4q.Config(grid=grid, scale=scale, rot=rot, round=round_mode, sign_mask_row=sign_mask if rot else 0,
                      sr_seed=sr_seed, want_col=False)
    row, _ = fp4q.rht_quantize(x, cfg, stream=stream)
    deq = fp4q.dequantize(row, cfg, orient=0, unrotate=bool(rot), stream=stream)
    ref = x.float()
    s = fp4q.bias_stats(ref.reshape(-1), deq.reshape(-1), row.codes.reshape(-1), stream=stream)
    rel = fp4q.rel_error(ref.reshape(-1), deq.reshape(-1), stream=stream)
    ge = fp4q.grid_error(x, cfg, row, stream=stream)
    return {"sqnr_db": s["sqnr_db"], "alpha": s["alpha"], "shrinkage": s["shrinkage"],
            "bucket_ratio": effective_bucket_ratio(s["hist"], grid), "hist": s["hist"], "sums": s["sums"],
            "mean_rel_error": rel["mean"], "grid_error": ge}


def delta_sqnr_sweep(rows: int, cols: int, strengths, grids=(fp4q.GRID_E2M1, fp4q.GRID_E1M2, fp4q.GRID_E2M1_R4),
                     seed: int = 2024, n_channels: int = 8, n_h: int = 16, device="cuda") -> list:
    """For each outlier strength (whole channels scaled by it), each grid: the
    report without rotation and with a random-sign H_{n_h}, and the SQNR change."""
    mask = fp4q.sign_mask_from_seed(seed, n_h)
    out = []
    for si, s in enumerate(strengths):
        bits = synth.normal_channel_outliers(rows, cols, seed + si, n_channels, float(s))
        x = synth.as_torch(bits).to(device)
        for g in grids:
            plain = quantizer_report(x, g, 0)
            rht = quantizer_report(x, g, n_h, mask)
            out.append({"strength": float(s), "grid": GRID_NAMES[g],
                        "sqnr_plain_db": plain["sqnr_db"], "sqnr_rht_db": rht["sqnr_db"],
                        "delta_sqnr_db": rht["sqnr_db"] - plain["sqnr_db"],
                        "bucket_ratio_plain": plain["bucket_ratio"], "bucket_ratio_rht": rht["bucket_ratio"],
                        "alpha_plain": plain["alpha"], "alpha_rht": rht["alpha"]})
    return out


def depth_chain(x_bits: np.ndarray, weights: list, grid: int, rot: int = 16, seed: int = 77,
                scale: int = fp4q.SCALE_MX, keep: bool = False, device="cuda") -> dict:
    """Run h_k = Q(h_{k-1}) Q(W_k)^T for the bf16 input x_bits [M, d] and bf16
    weights W_k [d_k, d_{k-1}] (uint16 bit arrays); h_k is stored as bf16, as an
    activation would be.  Layer k's rotation mask (along its contraction axis)
    comes from seed + k."""
    h = synth.as_torch(x_bits).to(device)
    h_ref = h.float()
    per = []
    kept = []
    for k, wb in enumerate(weights):
        w = synth.as_torch(wb).to(device)
        mask = fp4q.sign_mask_from_seed(seed + k, rot) if rot else 0
        cfg = fp4q.Config(grid=grid, scale=scale, rot=rot, sign_mask_row=mask, want_col=False,
                          sf_layout=fp4q.SF_MMA, emit_e4m3=(grid == fp4q.GRID_E1M2))
        A, _ = fp4q.rht_quantize(h, cfg)
        B, _ = fp4q.rht_quantize(w, cfg)
        yb, yf = fp4q.gemm(A, B, grid, scale, want_bf16=True, want_f32=True)
        exact = h.float() @ w.float().T
        s = fp4q.bias_stats(exact.reshape(-1), yf.reshape(-1))
        per.append({"alpha": s["alpha"], "shrinkage": s["shrinkage"], "sqnr_db": s["sqnr_db"]})
        if keep:
            kept.append({"input_bf16": h, "weight_bf16": w, "mask": mask, "out_f32": yf, "out_bf16": yb})
        h_ref = h_ref @ w.float().T
        h = yb
    end = fp4q.bias_stats(h_ref.reshape(-1), h.float().reshape(-1))
    alphas = [p["alpha"] for p in per]
    res = {"grid": GRID_NAMES[grid], "rot": rot, "layers": per,
           "prod_alpha": float(np.prod(alphas)),
           "exp_minus_sum_delta": float(math.exp(-sum(1.0 - a for a in alphas))),
           "end_to_end_alpha": end["alpha"], "end_to_end_sqnr_db": end["sqnr_db"]}
    if keep:
        res["kept"] = kept
    return res


def chain_weights(d: int, depth: int, seed: int = 3030) -> list:
    """Square bf16 weights N(0, 1/d): each layer keeps the signal's variance."""
    return [synth.normal(d, d, seed + k, 1.0 / math.sqrt(d)) for k in range(depth)]
