"""Pins of the oracle's GEMM entries and bias statistics: numpy's fp64 matrix
product, the rotation-invariance of D = A B^T when both operands share the
sign mask along K (and its failure when they do not), a hand-checkable case,
and the hand-computed statistics fixture."""
import os

import numpy as np
import pytest

from fp4_microscaled_quantization_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_gemm_entries_match_library_product(orc):
    rng = np.random.default_rng(0)
    A = rng.standard_normal((40, 96)).astype(np.float32)
    B = rng.standard_normal((24, 96)).astype(np.float32)
    full = orc.gemm_ref(A, B, 0.5)
    ii = rng.integers(0, 40, 300)
    jj = rng.integers(0, 24, 300)
    got = orc.gemm_entries(A, B, ii, jj, 0.5)
    assert np.allclose(got, full[ii, jj], rtol=1e-12, atol=1e-12)
    assert np.allclose(full, 0.5 * (A.astype(np.float64) @ B.astype(np.float64).T), rtol=1e-13)


def _rotate_rows(orc, M, n_h, mask):
    out = M.copy()
    for r in range(M.shape[0]):
        for c0 in range(0, M.shape[1], n_h):
            out[r, c0:c0 + n_h] = orc.rotate_block(M[r, c0:c0 + n_h], n_h, mask)
    return out


def test_rotation_invariance_needs_shared_mask(orc):
    rng = np.random.default_rng(1)
    A = rng.standard_normal((16, 64)).astype(np.float32)
    B = rng.standard_normal((8, 64)).astype(np.float32)
    D = orc.gemm_ref(A, B)
    for n_h in (16, 32):
        mk = orc.sign_mask_from_seed(5, n_h)
        Dr = orc.gemm_ref(_rotate_rows(orc, A, n_h, mk), _rotate_rows(orc, B, n_h, mk))
        assert np.abs(Dr - D).max() <= 1e-5 * np.abs(D).max()
        mk2 = orc.sign_mask_from_seed(6, n_h)
        Dbad = orc.gemm_ref(_rotate_rows(orc, A, n_h, mk), _rotate_rows(orc, B, n_h, mk2))
        assert np.abs(Dbad - D).max() > 0.1 * np.abs(D).max()


def test_gemm_of_quantized_block_by_hand(orc):
    """K = 32, one block per row: a = [6, 0, ...] at scale 2^0 and b = [1, 1, ...]
    at scale 2^-2 (values 1 -> code for 4 at e = -2) gives D = 6 * 1 = 6."""
    a = np.zeros((1, 32), np.float32)
    a[0, 0] = 6.0
    b = np.ones((1, 32), np.float32)
    qa = orc.quantize(synth.to_bf16_bits(a), 0, 0, orc.SCALE_MX, 0)
    qb = orc.quantize(synth.to_bf16_bits(b), 0, 0, orc.SCALE_MX, 0)
    assert qa["scales"][0, 0] == 127 and qb["scales"][0, 0] == 125
    da = orc.dequantize(qa["codes"], qa["scales"], 0, 0, orc.SCALE_MX)
    db = orc.dequantize(qb["codes"], qb["scales"], 0, 0, orc.SCALE_MX)
    assert orc.gemm_entries(da, db, [0], [0])[0] == 6.0


def _golden_stats():
    d = {}
    for line in open(os.path.join(GOLDEN, "stats_example.txt")):
        if line.strip() and not line.startswith("#"):
            k, *v = line.split()
            d[k] = [float(t) for t in v]
    return d


def test_stats_hand_example(orc):
    g = _golden_stats()
    s = orc.bias_stats(np.array(g["ref"], np.float32), np.array(g["approx"], np.float32))
    assert abs(s["sqnr_db"] - g["sqnr_db"][0]) < 1e-12
    assert abs(s["alpha"] - g["alpha"][0]) < 1e-15
    assert abs(s["shrinkage"] - g["shrinkage"][0]) < 1e-15


def test_stats_histogram_counts_codes(orc):
    codes = np.array([0x10, 0x32, 0xFF], np.uint8)  # codes 0,1,2,3,15,15
    s = orc.bias_stats(np.ones(6, np.float32), np.ones(6, np.float32), codes)
    want = np.zeros(16, np.uint64)
    for c in (0, 1, 2, 3, 15, 15):
        want[c] += 1
    assert np.array_equal(s["hist"], want)
    assert s["sqnr_db"] == float("inf") and s["alpha"] == 1.0


def test_e2m1_attenuates_more_than_e1m2_after_rotation(orc):
    """Directional report (not a parity pin): on Gaussian data rotated by H16,
    the E2M1 reconstruction shrinks magnitudes (alpha < 1) and E1M2 does not."""
    x = synth.normal(128, 256, 31)
    y = np.zeros((128, 256), np.float32)
    for r in range(128):
        for c0 in range(0, 256, 16):
            y[r, c0:c0 + 16] = orc.rotate_block(synth.bf16_bits_to_f32(x[r, c0:c0 + 16]), 16, 0)
    out = {}
    for grid in (0, 1):
        q = orc.quantize(x, 0, grid, orc.SCALE_MX, 16, 0)
        d = orc.dequantize(q["codes"], q["scales"], 0, grid, orc.SCALE_MX)
        out[grid] = orc.bias_stats(y, d)
    print({g: (round(v["alpha"], 5), round(v["shrinkage"], 5), round(v["sqnr_db"], 3)) for g, v in out.items()})
    assert out[0]["alpha"] < 1.0


def test_effective_bucket_ratio_closed_forms(orc):
    """exp(entropy)/levels: 1 for a uniform use of every level, 1/L for a single
    level, the sign folded away, and the two-level closed form."""
    uni = np.zeros(16)
    uni[:8] = 10
    assert orc.effective_bucket_ratio(uni, orc.GRID_E2M1) == pytest.approx(1.0, abs=1e-15)
    one = np.zeros(16)
    one[3], one[11] = 5, 7                     # +level 3 and -level 3: one magnitude
    assert orc.effective_bucket_ratio(one, orc.GRID_E1M2) == pytest.approx(1 / 8, abs=1e-15)
    two = np.zeros(16)
    two[1], two[12] = 1, 3                     # p = (1/4, 3/4) over levels 1 and 4
    H = -(0.25 * np.log(0.25) + 0.75 * np.log(0.75))
    assert orc.effective_bucket_ratio(two, orc.GRID_E2M1) == pytest.approx(np.exp(H) / 8, rel=1e-14)
    cap = np.zeros(16)
    cap[:7] = 4                                 # every level the capped grid can make
    assert orc.effective_bucket_ratio(cap, orc.GRID_E2M1_R4) == pytest.approx(1.0, abs=1e-15)
    assert np.isnan(orc.effective_bucket_ratio(np.zeros(16), orc.GRID_E2M1))


def test_effective_bucket_ratio_of_quantized_uniform_data(orc):
    """Data spread evenly over the E1M2 grid's bins (every block holding one
    value at the top so that the scale is 2^0) fills all 8 levels equally."""
    R, C = 32, 256
    lv = orc.grid_levels(orc.GRID_E1M2)
    vals = np.tile(np.repeat(lv, 4), (R, 1)).astype(np.float32)     # 32 values per block, 4 per level
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)            # exact in bf16
    q = orc.quantize(bits, 0, orc.GRID_E1M2, orc.SCALE_MX, 0)
    st = orc.bias_stats(vals.ravel(), orc.dequantize(q["codes"], q["scales"], 0, orc.GRID_E1M2, 0).ravel(),
                        q["codes"])
    assert st["sqnr_db"] == float("inf")
    assert orc.effective_bucket_ratio(st["hist"], orc.GRID_E1M2) == pytest.approx(1.0, abs=1e-15)


def test_rel_error_hand_example(orc):
    """Per-element mean signed relative error over ref != 0, against the hand
    value in the golden file; elements with ref = 0 are left out."""
    g = _golden_stats()
    s = orc.rel_error(np.array(g["ref"], np.float32), np.array(g["approx"], np.float32))
    assert s["mean"] == g["mean_rel_error"][0] and s["count"] == 2
    s0 = orc.rel_error(np.array(g["ref"] + [0.0], np.float32), np.array(g["approx"] + [5.0], np.float32))
    assert s0["mean"] == g["mean_rel_error"][0] and s0["count"] == 2


def _bin_midpoints(lo, hi, w):
    """Midpoints of the strata of width w that tile [lo, hi)."""
    n = int(round((hi - lo) / w))
    return lo + (np.arange(n) + 0.5) * w


# (grid, level, RTNE bin of the level, stratum width, block maximum in another level)
_BIN_CASES = [(0, 2.0, (1.75, 2.5), 1 / 32, 6.0), (0, 4.0, (3.5, 5.0), 1 / 16, 6.0),
              (0, 1.5, (1.25, 1.75), 1 / 32, 6.0), (0, 3.0, (2.5, 3.5), 1 / 32, 6.0),
              (1, 0.75, (0.625, 0.875), 1 / 128, 1.75), (1, 1.25, (1.125, 1.375), 1 / 64, 1.75)]


@pytest.mark.parametrize("grid,level,bin_,w,vmax", _BIN_CASES)
def test_grid_error_per_level_equals_half_bin_asymmetry(orc, grid, level, bin_, w, vmax):
    """Inputs spread evenly over one level's RTNE bin (stratum midpoints, all
    exact in bf16), one block maximum in another level so that the block scale
    is 1: the level's mean error in grid units is the page's (l_i - r_i)/2
    (golden, "Repensando o Vies de Encolhimento", Metodologia 1), exactly,
    since the error is linear in x within the bin."""
    want = {(g, lvl): w_ for g, lvl, w_ in _golden_cond_error()}[(grid, level)]
    vals = _bin_midpoints(*bin_, w).astype(np.float32)
    per_block = 16
    nb = (vals.size + per_block - 1) // per_block
    x = np.zeros((1, 32 * nb), np.float32)
    for b in range(nb):
        part = vals[b * per_block:(b + 1) * per_block]
        x[0, 32 * b] = vmax
        x[0, 32 * b + 1:32 * b + 1 + part.size] = part
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), x)   # exact in bf16
    q = orc.quantize(bits, 0, grid, orc.SCALE_MX, 0)
    assert np.all(q["scales"] == 127)
    ge = orc.grid_error(bits, grid, orc.SCALE_MX, 0, 0, q["codes"], q["scales"])
    k = int(np.where(orc.grid_levels(grid) == np.float32(level))[0][0])
    assert int(ge["counts"][k]) == vals.size
    assert ge["sums"][k] / ge["counts"][k] == want


def _golden_cond_error():
    out = []
    for line in open(os.path.join(GOLDEN, "conditional_error.txt")):
        if line.strip() and not line.startswith("#"):
            g, lvl, want = line.split()
            out.append(({"e2m1": 0, "e1m2": 1, "e2m1r4": 2}[g], float(lvl), float(want)))
    return out


@pytest.mark.parametrize("grid,scale,rot", [(0, 0, 16), (1, 0, 32), (0, 1, 16), (2, 0, 0)])
def test_grid_error_within_each_bin(orc, grid, scale, rot):
    """Every element's error in grid units lies within its level's RTNE bin
    (-r_i <= g - |v| <= l_i, saturated elements below -r only), on rotated
    random data with MX and NVFP4-style scales; zero blocks count at level 0."""
    bits = synth.normal_channel_outliers(64, 256, 77, 4, 30.0)
    bits[:, 32:64] = 0
    q = orc.quantize(bits, 0, grid, scale, rot, 0x2A5B)
    ge = orc.grid_error(bits, grid, scale, rot, 0x2A5B, q["codes"], q["scales"], q["tensor_scale"])
    L = orc.grid_levels(grid).astype(np.float64)
    top = orc.grid_top(grid)
    assert int(ge["counts"].sum()) == bits.size
    for k in range(top + 1):
        if ge["counts"][k] == 0:
            continue
        left = (L[k] - L[k - 1]) / 2 if k > 0 else 0.0
        mean = ge["sums"][k] / ge["counts"][k]
        assert mean <= left + 1e-12, (k, mean)
        if k < top:
            right = (L[k + 1] - L[k]) / 2
            assert mean >= -right - 1e-12, (k, mean)
