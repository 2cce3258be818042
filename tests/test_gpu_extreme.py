"""Extreme aspect ratios: very wide and very tall quantizer inputs, and GEMMs
with many tiles along one dimension and a short K.  They exercise the large
row/column/tile indices of the kernels.  The GPU copies are compared bit for
bit with the oracle on sampled rows and 32-row groups (a row-wise copy of a
row depends only on that row; a column-wise block only on its 32 rows, so
the oracle runs on those slices); GEMM outputs are sampled entries against the
oracle's fp64 dot products of the dequantized operands, within 1e-3 relative
Frobenius error over the sample."""
import numpy as np
import pytest
import torch

from fp4_microscaled_quantization_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp4_microscaled_quantization_gb300 import fp4q
    fp4q.lib()
    return fp4q


def check_rows(orc, bits, cfg, ro, rows):
    codes = ro.codes.cpu().numpy()
    scales = ro.scales.cpu().numpy()
    for r in rows:
        want = orc.quantize(bits[r:r + 1], 0, cfg.grid, cfg.scale, cfg.rot, cfg.sign_mask_row)
        assert np.array_equal(codes[r], want["codes"][0]), f"row {r}"
        assert np.array_equal(scales[r], want["scales"][0]), f"row {r} scales"


def check_col_groups(orc, bits, cfg, co, r0s):
    """Column-wise copy (cols x rows/2) restricted to source rows [r0, r0 + 32)."""
    codes = co.codes.cpu().numpy()
    scales = co.scales.cpu().numpy()
    b = cfg.block
    for r0 in r0s:
        want = orc.quantize(np.ascontiguousarray(bits[r0:r0 + 32]), 1, cfg.grid, cfg.scale, cfg.rot,
                            cfg.sign_mask_col)
        assert np.array_equal(codes[:, r0 // 2:(r0 + 32) // 2], want["codes"]), f"rows {r0}.."
        assert np.array_equal(scales[:, r0 // b:(r0 + 32) // b], want["scales"]), f"rows {r0}.. scales"


# the last shape is the most rows the quantizer accepts, (rows + 63) / 64 = 65535
@pytest.mark.parametrize("R,C", [(64, 1 << 19), (1 << 20, 32), (65535 * 64, 32)])
def test_quantizer_wide_and_tall(fq, orc, R, C):
    bits = synth.normal_point_outliers(R, C, R + C, 0.001, 40.0)
    cfg = fq.Config(rot=16, sign_mask_row=0x2D4B, sign_mask_col=0x8E31)
    x = synth.as_torch(bits).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ro, co = fq.rht_quantize(x, cfg, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rng = np.random.default_rng(R ^ C)
    check_rows(orc, bits, cfg, ro, sorted({0, R - 1, *rng.integers(0, R, 6).tolist()}))
    groups = sorted({0, (R - 32) // 32 * 32, *(rng.integers(0, R // 32, 6) * 32).tolist()})
    check_col_groups(orc, bits, cfg, co, groups)


def mma_layout(plain):
    """Scale bytes [rows, nkb] placed in the MMA scale layout (512-byte groups
    of 128 rows by four K-blocks)."""
    rows, nkb = plain.shape
    r = np.arange(rows)[:, None]
    k = np.arange(nkb)[None, :]
    off = ((r // 128) * (nkb // 4) + k // 4) * 512 + 16 * (r % 32) + 4 * ((r // 32) % 4) + k % 4
    out = np.empty(rows * nkb, dtype=np.uint8)
    out[off.reshape(-1)] = plain.reshape(-1)
    return out.reshape(rows, nkb)


def test_gemm_maximum_m(fq, orc):
    """The largest M the GEMM accepts (M / 128 = 65535, so its last 256-row
    tile is a 128-row tail) on sampled entries against the oracle.  A is made
    of seeded random E2M1 code bytes and E8M0 scale bytes 2^-7 .. 2^7 (the
    quantizer takes at most 65535 * 64 rows in one call)."""
    M, N, K = 65535 * 128, 128, 128
    rng = np.random.default_rng(65535)
    a_codes = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    a_scales = rng.integers(120, 135, (M, K // 32), dtype=np.uint8)
    A = fq.Operand(codes=torch.from_numpy(a_codes).cuda(), scales=torch.from_numpy(mma_layout(a_scales)).cuda(),
                   rows=M, cols=K, sf_layout=fq.SF_MMA)
    b = synth.normal(N, K, 77, 0.05)
    cfg = fq.Config(rot=16, sign_mask_row=0x3C5A, want_col=False, sf_layout=fq.SF_MMA)
    B, _ = fq.rht_quantize(synth.as_torch(b).cuda(), cfg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, D = fq.gemm(A, B, 0, 0, want_bf16=False, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ii = np.concatenate([[0, 127, M - 256, M - 129, M - 128, M - 1], rng.integers(0, M, 250)])
    jj = rng.integers(0, N, ii.size)
    rows_a = np.unique(ii)
    da = orc.dequantize(np.ascontiguousarray(a_codes[rows_a]), np.ascontiguousarray(a_scales[rows_a]), 0, 0, 0)
    qb = orc.quantize(b, 0, 0, 0, 16, cfg.sign_mask_row)
    db = orc.dequantize(qb["codes"], qb["scales"], 0, 0, 0)
    want = orc.gemm_entries(da, db, np.searchsorted(rows_a, ii), jj)
    got = D[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].double().cpu().numpy()
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel <= 1e-3, f"sampled relative Frobenius error {rel:.3e}"


@pytest.mark.parametrize("M,N,K", [(1 << 17, 128, 128), (128, 1 << 16, 256), (256, 256, 1 << 16)])
def test_gemm_long_dimensions(fq, orc, M, N, K):
    a = synth.normal(M, K, M + K, 1.0)
    b = synth.normal(N, K, N + 2 * K, 0.05)
    cfg = fq.Config(rot=16, sign_mask_row=0x6A09, want_col=False, sf_layout=fq.SF_MMA)
    A, _ = fq.rht_quantize(synth.as_torch(a).cuda(), cfg)
    B, _ = fq.rht_quantize(synth.as_torch(b).cuda(), cfg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, D = fq.gemm(A, B, 0, 0, want_bf16=False, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rng = np.random.default_rng(M + N + K)
    ii = np.concatenate([[0, M - 1], rng.integers(0, M, 254)])
    jj = np.concatenate([[N - 1, 0], rng.integers(0, N, 254)])
    rows_a, rows_b = np.unique(ii), np.unique(jj)
    qa = orc.quantize(np.ascontiguousarray(a[rows_a]), 0, 0, 0, 16, cfg.sign_mask_row)
    qb = orc.quantize(np.ascontiguousarray(b[rows_b]), 0, 0, 0, 16, cfg.sign_mask_row)
    da = orc.dequantize(qa["codes"], qa["scales"], 0, 0, 0)
    db = orc.dequantize(qb["codes"], qb["scales"], 0, 0, 0)
    want = orc.gemm_entries(da, db, np.searchsorted(rows_a, ii), np.searchsorted(rows_b, jj))
    got = D.cpu().numpy()[ii, jj].astype(np.float64)
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel <= 1e-3, f"sampled relative Frobenius error {rel:.3e}"
