"""GPU parity of the fused rotation + quantizer, the amax pass, the dequantizer,
the unfused rotation arm and the bias statistics against the CPU oracle.

Codes, scales, tensor scales and E4M3 bytes are compared bit for bit;
dequantized values exactly; statistics within 1e-9 relative (both sides sum in
fp64; only the summation order differs)."""
import itertools

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


def mma_to_plain(flat: np.ndarray, rows: int, nkb: int) -> np.ndarray:
    """Undo the FP4Q_SF_MMA permutation (documented in include/fp4q.h)."""
    r = np.arange(rows)[:, None]
    k = np.arange(nkb)[None, :]
    off = ((r // 128) * (nkb // 4) + k // 4) * 512 + 16 * (r % 32) + 4 * ((r // 32) % 4) + k % 4
    return flat.reshape(-1)[off]


def check_copy(orc, x_bits, orient, cfg, op, given_amax=None):
    mask = cfg.sign_mask_row if orient == 0 else cfg.sign_mask_col
    ref = orc.quantize(x_bits, orient, cfg.grid, cfg.scale, cfg.rot, mask, cfg.round, cfg.sr_seed,
                       given_amax=given_amax, want_e4m3=cfg.emit_e4m3)
    codes = op.codes.cpu().numpy()
    assert codes.shape == ref["codes"].shape
    bad = np.flatnonzero(codes.reshape(-1) != ref["codes"].reshape(-1))
    assert bad.size == 0, f"orient {orient}: {bad.size} code bytes differ, first at {bad[:5]}"
    sc = op.scales.cpu().numpy()
    if cfg.sf_layout == 1:
        sc = mma_to_plain(sc, ref["scales"].shape[0], ref["scales"].shape[1])
    assert np.array_equal(sc, ref["scales"]), f"orient {orient}: scales differ"
    if cfg.scale == 1:
        got = op.tensor_scale.cpu().numpy()[0]
        assert got.view(np.uint32) == np.float32(ref["tensor_scale"]).view(np.uint32)
    if cfg.emit_e4m3:
        assert np.array_equal(op.e4m3.cpu().numpy(), ref["e4m3"])
    return ref


def run_case(fq, orc, x_bits, cfg, given=None):
    x = synth.as_torch(x_bits).cuda()
    if given is not None:
        cfg.global_amax = torch.tensor(given, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ro, co = fq.rht_quantize(x, cfg, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    refs = {}
    if cfg.want_row:
        refs[0] = check_copy(orc, x_bits, 0, cfg, ro, None if given is None else given[0])
    if cfg.want_col:
        refs[1] = check_copy(orc, x_bits, 1, cfg, co, None if given is None else given[1])
    return ro, co, refs


SHAPES = [(96, 800), (160, 288), (64, 256), (32, 32)]   # several tiles, ragged tails, a single chunk


@pytest.mark.parametrize("grid,scale,rot,rnd", list(itertools.product([0, 1, 2], [0, 1], [0, 16, 32], [0, 1])))
def test_quantize_all_modes_small(fq, orc, grid, scale, rot, rnd):
    for si, (R, C) in enumerate(SHAPES):
        x = synth.special_values(R, C, 100 + si) if si % 2 else synth.normal_point_outliers(R, C, 200 + si)
        for mask_seed in ((None, 3) if rot else (None,)):
            mr = orc.sign_mask_from_seed(mask_seed, rot) if mask_seed is not None else 0
            mc = orc.sign_mask_from_seed(mask_seed + 1, rot) if mask_seed is not None else 0
            cfg = fq.Config(grid=grid, scale=scale, rot=rot, round=rnd, sign_mask_row=mr, sign_mask_col=mc,
                            sr_seed=12345 + si, emit_e4m3=True)
            run_case(fq, orc, x, cfg)


@pytest.mark.parametrize("grid,scale", [(0, 0), (1, 0), (0, 1), (1, 1), (2, 0), (2, 1)])
def test_quantize_mma_scale_layout(fq, orc, grid, scale):
    x = synth.normal_channel_outliers(256, 384, 7)
    cfg = fq.Config(grid=grid, scale=scale, rot=16, sign_mask_row=0x1234, sign_mask_col=0xBEEF,
                    sf_layout=1)
    run_case(fq, orc, x, cfg)


def test_row_or_col_only_and_strided_input(fq, orc):
    x = synth.normal(64, 512, 3)
    cfg = fq.Config(want_col=False)
    run_case(fq, orc, x, cfg)
    cfg = fq.Config(want_row=False, grid=1, round=1, sr_seed=9)
    run_case(fq, orc, x, cfg)
    # a strided view: row stride 768 elements
    big = synth.normal(64, 768, 4)
    xt = synth.as_torch(big).cuda()[:, 128:640]
    ro, co = fq.rht_quantize(xt, fq.Config())
    torch.cuda.synchronize()
    sub = np.ascontiguousarray(big[:, 128:640])
    check_copy(orc, sub, 0, fq.Config(), ro)
    check_copy(orc, sub, 1, fq.Config(), co)


def test_nv_given_amax_and_amax_pass(fq, orc):
    x = synth.weight_w(256, 512, 5)
    xt = synth.as_torch(x).cuda()
    for rot in (16, 32):
        cfg = fq.Config(scale=1, rot=rot, sign_mask_row=0xA5A5, sign_mask_col=0x5A5A)
        g = fq.rotated_amax(xt, cfg).cpu().numpy()
        # G = the largest |y| of each rotated copy, from the oracle's rotation
        for orient, mask in ((0, cfg.sign_mask_row), (1, cfg.sign_mask_col)):
            m = x if orient == 0 else np.ascontiguousarray(x.T)
            f = synth.bf16_bits_to_f32(m)
            G = 0.0
            for r in range(f.shape[0]):
                for c0 in range(0, f.shape[1], rot):
                    G = max(G, float(np.abs(orc.rotate_block(f[r, c0:c0 + rot], rot, mask)).max()))
            assert g[orient] == np.float32(G)
        run_case(fq, orc, x, cfg, given=[float(g[0]) * 1.5, float(g[1]) * 0.5])   # caller's G (saturating too)


def planted_sr_ties(orc, rows, cols, grid, seed, orient):
    """Input whose stored copy ``orient`` (rows x cols in the copy's own
    coordinates) has MX scale 1 in every block (element 0 of each block is the
    block maximum 2^emax) and, wherever the draw r of an element's index has at
    most 8 significant bits, an exact SR tie: |v| = (r / 2^16) g_1 on the lowest
    interval [0, g_1), so that u = r / 2^16 equals the fraction and the element
    rounds down.  The other elements are uniform in (-2^emax, 2^emax).  Returns
    the bf16 input (transposed back for the column copy) and the tie mask."""
    g = np.random.default_rng(seed)
    top = np.float32(2.0 ** orc.grid_emax(grid))
    g1 = np.float32(orc.grid_levels(grid)[1])
    z = g.uniform(-1.0, 1.0, (rows, cols)).astype(np.float32) * top
    ties = np.zeros((rows, cols), dtype=bool)
    for i in range(rows):
        for j in range(cols):
            if j % 32 == 0:
                z[i, j] = top if g.integers(2) else -top
                continue
            r = orc.sr_uniform16(seed, i * cols + j, orient)
            if r and (r >> ((r & -r).bit_length() - 1)) < 256:
                z[i, j] = np.float32(r) / np.float32(65536.0) * g1 * (1 if g.integers(2) else -1)
                ties[i, j] = True
    bits = synth.to_bf16_bits(z)
    assert np.array_equal(synth.bf16_bits_to_f32(bits)[ties], z[ties])   # the ties are exact in bf16
    return (bits if orient == 0 else np.ascontiguousarray(bits.T)), ties


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_sr_exact_ties_round_down(fq, orc, grid):
    """SR decides u < f strictly: an element whose fraction f equals its draw
    u = r / 2^16 rounds down, on both copies (each copy draws from its own
    index and orientation)."""
    rows, cols = 64, 256
    for orient in (0, 1):
        seed = 4242 + 10 * grid + orient
        x, ties = planted_sr_ties(orc, rows, cols, grid, seed, orient)
        assert ties.sum() > 150
        cfg = fq.Config(grid=grid, scale=0, rot=0, round=1, sr_seed=seed, want_row=(orient == 0),
                        want_col=(orient == 1))
        _, _, refs = run_case(fq, orc, x, cfg)
        ref = refs[orient]
        assert np.all(ref["scales"] == 127)
        lo = ref["codes"] & 0xF
        hi = ref["codes"] >> 4
        codes = np.stack([lo, hi], axis=-1).reshape(rows, cols)
        assert np.all((codes[ties] & 7) == 0)


def top_of_range_input(top_exp: int) -> np.ndarray:
    """Rows 0-31: equal-sign 2^top_exp (1 + k/8); rows 32-47: normals times
    2^100..2^(top_exp - 3); row 48: half 2^(top_exp - 1), half 1e-38."""
    R, C = 64, 256
    g = np.random.default_rng(77 + top_exp)
    x = g.standard_normal((R, C)).astype(np.float32)
    x[0:32, :] = np.float32(2.0 ** top_exp) * (1 + g.integers(0, 8, (32, C)).astype(np.float32) / 8)
    x[32:48, :] *= np.float32(2.0) ** g.integers(100, top_exp - 2, (16, 1)).astype(np.float32)
    x[48, :128] = np.float32(2.0 ** (top_exp - 1))
    x[48, 128:] = np.float32(1e-38)
    return synth.to_bf16_bits(x)


@pytest.mark.parametrize("grid,rnd", [(0, 0), (1, 0), (2, 0), (1, 1), (0, 1)])
def test_quantize_top_of_range(fq, orc, grid, rnd):
    """Blocks whose rotated values reach the top of the fp32 range, without
    overflowing it (a rotation overflow is a non-finite block, flagged by the
    kernel).  With H16 and MX scales the kernel leaves the rotation's 1/4 to
    the block scale, whose multiplier 2^(125 - sb) is subnormal when the
    unscaled sums reach 2^127 (E1M2, scale byte 252): 16 equal-sign values
    2^123 (1 + k/8) sum to [2^127, 2^128) under the deterministic H16.  H32
    takes 2^122 so that its 32-term sums stay finite."""
    for rot, top, masks in ((16, 123, ((0, 0), (0x5A5A, 0xA5A5))), (32, 122, ((0, 0),))):
        bits = top_of_range_input(top)
        for mr, mc in masks:
            cfg = fq.Config(grid=grid, scale=0, rot=rot, round=rnd, sign_mask_row=mr, sign_mask_col=mc, sr_seed=99,
                            emit_e4m3=(grid == 1))
            run_case(fq, orc, bits, cfg)


def test_empty_and_nonfinite(fq, orc):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    ro, co = fq.rht_quantize(x, fq.Config())
    assert ro.codes.numel() == 0
    bits = synth.normal(64, 64, 1)
    for bad in (0x7F80, 0xFFC0):        # +inf, NaN
        b = bits.copy()
        b[5, 9] = bad
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fq.rht_quantize(synth.as_torch(b).cuda(), fq.Config(rot=0), status=st)
        torch.cuda.synchronize()
        assert st.item() & fq.DEV_NONFINITE


@pytest.mark.parametrize("grid,scale,rot", [(0, 0, 16), (1, 0, 32), (0, 1, 16), (1, 1, 32), (0, 0, 0), (2, 0, 16), (2, 1, 32)])
def test_dequantize_exact(fq, orc, grid, scale, rot):
    x = synth.special_values(64, 256, 17)
    cfg = fq.Config(grid=grid, scale=scale, rot=rot, sign_mask_row=0x0F0F, sign_mask_col=0x3333)
    ro, co, refs = run_case(fq, orc, x, cfg)
    for orient, op in ((0, ro), (1, co)):
        for unrot in (False, True):
            d = fq.dequantize(op, cfg, orient=orient, unrotate=unrot).cpu().numpy()
            mask = cfg.sign_mask_row if orient == 0 else cfg.sign_mask_col
            want = orc.dequantize(refs[orient]["codes"], refs[orient]["scales"], refs[orient]["tensor_scale"],
                                  grid, scale, True, rot, mask, unrot)
            assert np.array_equal(d.view(np.uint32), want.view(np.uint32))


def test_rotate_bf16_arm(fq, orc):
    x = synth.normal_channel_outliers(96, 512, 8)
    for rot in (16, 32):
        yr, yc = fq.hadamard_rotate_bf16(synth.as_torch(x).cuda(), rot, 0x1357, 0x2468)
        f = synth.bf16_bits_to_f32(x)
        want_r = np.zeros_like(f)
        want_c = np.zeros_like(f)
        for r in range(f.shape[0]):
            for c0 in range(0, f.shape[1], rot):
                want_r[r, c0:c0 + rot] = orc.rotate_block(f[r, c0:c0 + rot], rot, 0x1357)
        for c in range(f.shape[1]):
            for r0 in range(0, f.shape[0], rot):
                want_c[r0:r0 + rot, c] = orc.rotate_block(f[r0:r0 + rot, c], rot, 0x2468)
        assert np.array_equal(yr.view(torch.int16).cpu().numpy().view(np.uint16), synth.to_bf16_bits(want_r))
        assert np.array_equal(yc.view(torch.int16).cpu().numpy().view(np.uint16), synth.to_bf16_bits(want_c))


@pytest.mark.parametrize("n", [6, 1000, 1 << 20])
def test_bias_stats(fq, orc, n):
    rng = np.random.default_rng(n)
    ref = rng.standard_normal(n).astype(np.float32)
    approx = (ref * 0.97 + rng.standard_normal(n).astype(np.float32) * 0.01).astype(np.float32)
    codes = rng.integers(0, 256, n // 2, dtype=np.uint8)
    got = fq.bias_stats(torch.from_numpy(ref).cuda(), torch.from_numpy(approx).cuda(),
                        torch.from_numpy(codes).cuda())
    want = orc.bias_stats(ref, approx, codes)
    assert np.allclose(got["sums"], want["sums"], rtol=1e-9, atol=0)
    assert np.array_equal(got["hist"], want["hist"]) and got["n"] == n
    for k in ("sqnr_db", "alpha", "shrinkage"):
        assert abs(got[k] - want[k]) <= 1e-9 * max(1.0, abs(want[k]))
    # repeated calls reuse the workspace and give identical bits
    again = fq.bias_stats(torch.from_numpy(ref).cuda(), torch.from_numpy(approx).cuda(),
                          torch.from_numpy(codes).cuda())
    assert np.array_equal(again["sums"], got["sums"])
