"""GPU parity of the two error diagnostics against the oracle
("Repensando o Vies de Encolhimento", Metodologia 1, "Origem Geometrica"):
the rounding error in grid units per level (fp4q_grid_error) and the
per-element mean signed relative error (fp4q_rel_error).

Each side quantizes the same seeded input with its own quantizer (the codes
are compared bit for bit first), then measures its own copy.  Counts per level
are exact; the fp64 sums agree to 1e-9 relative plus a term for the position
v, which both sides compute in fp32 from a rotation whose fp32 rounding may
differ in the last bit (one ulp of |v| <= 8 per element at most)."""
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


def _plain_scales(fq, op, rows, cols, cfg):
    """Scale bytes in the plain row-major layout; an MMA-layout copy is read
    back at the interleaved offset that include/fp4q.h gives for (r, k)."""
    s = op.scales.cpu().numpy().reshape(-1)
    if cfg.sf_layout == fq.SF_PLAIN:
        return s.reshape(rows, -1)
    nkb = cols // cfg.block
    r = np.arange(rows)[:, None]
    k = np.arange(nkb)[None, :]
    off = ((r // 128) * (nkb // 4) + k // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (k % 4)
    return s[off]


def _sums_close(got, want, counts):
    tol = 1e-9 * np.abs(want) + counts.astype(np.float64) * 8.0 * 2.0 ** -23
    assert np.all(np.abs(got - want) <= tol), (got, want)


CASES = [
    # grid, scale, rot, sf_layout, rows, cols
    (0, 0, 16, 0, 96, 640),
    (0, 0, 0, 0, 96, 640),
    (1, 0, 32, 0, 96, 640),
    (2, 0, 16, 0, 96, 640),
    (0, 1, 16, 0, 96, 640),
    (1, 1, 0, 0, 96, 640),
    (0, 0, 32, 1, 256, 1024),
    (1, 1, 16, 1, 256, 1024),
]


@pytest.mark.parametrize("grid,scale,rot,sfl,R,C", CASES)
def test_grid_error_matches_oracle(fq, orc, grid, scale, rot, sfl, R, C):
    bits = synth.normal_channel_outliers(R, C, 71, 8, 30.0)
    mask = orc.sign_mask_from_seed(9, rot) if rot else 0
    cfg = fq.Config(grid=grid, scale=scale, rot=rot, sign_mask_row=mask, want_col=False, sf_layout=sfl)
    x = synth.as_torch(bits).cuda()
    row, _ = fq.rht_quantize(x, cfg)
    got = fq.grid_error(x, cfg, row)
    q = orc.quantize(bits, 0, grid, scale, rot, mask)
    assert np.array_equal(row.codes.cpu().numpy(), q["codes"])
    assert np.array_equal(_plain_scales(fq, row, R, C, cfg), q["scales"])
    want = orc.grid_error(bits, grid, scale, rot, mask, q["codes"], q["scales"], q["tensor_scale"])
    assert np.array_equal(got["counts"], want["counts"])
    _sums_close(got["sums"], want["sums"], want["counts"])
    # every level's mean error lies within half the bin around it
    assert abs(got["mean"]) < 1.0


def test_grid_error_column_copy_is_row_copy_of_transpose(fq, orc):
    R, C = 128, 512
    bits = synth.grad_dy(R, C, 73)
    mask_c = orc.sign_mask_from_seed(11, 16)
    cfg = fq.Config(grid=0, scale=0, rot=16, sign_mask_col=mask_c, want_row=False, want_col=True)
    x = synth.as_torch(bits).cuda()
    _, col = fq.rht_quantize(x, cfg)
    cfg_t = fq.Config(grid=0, scale=0, rot=16, sign_mask_row=mask_c, want_col=False)
    got = fq.grid_error(x.t().contiguous(), cfg_t, col)
    q = orc.quantize(bits, 1, 0, orc.SCALE_MX, 16, mask_c)
    assert np.array_equal(col.codes.cpu().numpy(), q["codes"])
    want = orc.grid_error(np.ascontiguousarray(bits.T), 0, orc.SCALE_MX, 16, mask_c, q["codes"], q["scales"])
    assert np.array_equal(got["counts"], want["counts"])
    _sums_close(got["sums"], want["sums"], want["counts"])


def test_grid_error_strided_input(fq, orc):
    R, C, ld = 64, 256, 384
    full = synth.normal(R, ld, 75)
    bits = np.ascontiguousarray(full[:, :C])
    cfg = fq.Config(grid=1, scale=0, rot=32, sign_mask_row=orc.sign_mask_from_seed(3, 32), want_col=False)
    xs = synth.as_torch(full).cuda()[:, :C]
    row, _ = fq.rht_quantize(xs, cfg)
    got = fq.grid_error(xs, cfg, row)
    q = orc.quantize(bits, 0, 1, orc.SCALE_MX, 32, cfg.sign_mask_row)
    want = orc.grid_error(bits, 1, orc.SCALE_MX, 32, cfg.sign_mask_row, q["codes"], q["scales"])
    assert np.array_equal(got["counts"], want["counts"])
    _sums_close(got["sums"], want["sums"], want["counts"])


@pytest.mark.parametrize("n", [1, 1000, 333_333])
def test_rel_error_matches_oracle(fq, orc, n):
    g = np.random.Generator(np.random.PCG64(n))
    ref = g.standard_normal(n).astype(np.float32)
    ref[:: 7] = 0.0
    approx = (ref * (1.0 + 0.1 * g.standard_normal(n))).astype(np.float32)
    approx[:: 11] = 0.0
    got = fq.rel_error(torch.from_numpy(ref).cuda(), torch.from_numpy(approx).cuda())
    want = orc.rel_error(ref, approx)
    assert got["count"] == want["count"]
    if want["count"]:
        assert got["sum"] == pytest.approx(want["sum"], rel=1e-12, abs=1e-12)


def test_rel_error_empty_and_all_zero(fq):
    z = torch.zeros(64, device="cuda")
    got = fq.rel_error(z, z)
    assert got["count"] == 0 and got["sum"] == 0.0
    e = torch.empty(0, device="cuda")
    got = fq.rel_error(e, e)
    assert got["count"] == 0


def test_diagnostics_are_deterministic(fq, orc):
    bits = synth.act_x(1024, 2048, 77)
    cfg = fq.Config(grid=0, scale=0, rot=16, sign_mask_row=orc.sign_mask_from_seed(1, 16), want_col=False)
    x = synth.as_torch(bits).cuda()
    row, _ = fq.rht_quantize(x, cfg)
    a = fq.grid_error(x, cfg, row)
    b = fq.grid_error(x, cfg, row)
    assert np.array_equal(a["sums"], b["sums"])


def test_invalid_arguments_are_refused(fq):
    x = torch.zeros(32, 48, dtype=torch.bfloat16, device="cuda")
    cfg = fq.Config(grid=0, scale=0, rot=16, want_col=False)
    row = fq.alloc_operand(32, 64, cfg, "cuda")
    with pytest.raises(RuntimeError):
        fq.grid_error(x, cfg, row)   # cols not a multiple of 32
