"""Pins of the oracle's number formats and random streams against definitions
that do not come from the oracle itself: the bit-level format definitions, a
library cast (torch float8_e4m3fn) and published Philox known-answer vectors."""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _decode_minifloat(code3: int, exp_bits: int, man_bits: int, bias: int) -> float:
    """Magnitude of a sign-less minifloat bit pattern (subnormals when e == 0)."""
    e = code3 >> man_bits
    m = code3 & ((1 << man_bits) - 1)
    if e == 0:
        return (m / (1 << man_bits)) * 2.0 ** (1 - bias)
    return (1.0 + m / (1 << man_bits)) * 2.0 ** (e - bias)


def test_e2m1_levels_follow_bit_format(orc):
    # E2M1: 2 exponent bits, 1 mantissa bit, bias 1 (the OCP FP4 element type).
    want = [_decode_minifloat(k, 2, 1, 1) for k in range(8)]
    assert list(orc.grid_levels(orc.GRID_E2M1)) == want
    assert want == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e1m2_levels_follow_bit_format_and_are_uniform(orc):
    want = [_decode_minifloat(k, 1, 2, 1) for k in range(8)]
    lv = orc.grid_levels(orc.GRID_E1M2)
    assert list(lv) == want
    gaps = np.diff(lv)
    assert np.all(gaps == gaps[0])            # l_i == r_i: every level's bins are symmetric
    e2 = np.diff(orc.grid_levels(orc.GRID_E2M1))
    assert list(e2) == [0.5, 0.5, 0.5, 0.5, 1, 1, 2]   # spacing grows across binades


@pytest.mark.parametrize("grid", [0, 1])
def test_qmax_emax(orc, grid):
    q = orc.grid_qmax(grid)
    e = orc.grid_emax(grid)
    assert q == orc.grid_levels(grid)[7]
    assert 2.0 ** e <= q < 2.0 ** (e + 1)


def test_code_values_signed(orc):
    for grid in (0, 1):
        lv = orc.grid_levels(grid)
        for c in range(16):
            v = orc.code_value(grid, c)
            assert abs(v) == lv[c & 7]
            assert np.signbit(np.float32(v)) == bool(c & 8)


def test_e4m3_decode_matches_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([orc.e4m3_decode(b) for b in range(256)], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert orc.e4m3_decode(0x7E) == 448.0


def test_e4m3_encode_matches_torch_rne(orc):
    vals = np.array([orc.e4m3_decode(b) for b in range(0x7F)], dtype=np.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        vals, mids,
        np.nextafter(mids.astype(np.float32), np.float32(0)),
        np.nextafter(mids.astype(np.float32), np.float32(1e9)),
        rng.uniform(0, 448, 4000), np.exp(rng.uniform(np.log(1e-5), np.log(448), 4000)),
    ]).astype(np.float32)
    xs = xs[xs <= 448]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates(orc):
    for x in (448.0, 449.0, 464.0, 500.0, 1e30, float("inf")):
        assert orc.e4m3_encode(x) == 0x7E


def test_grids_exact_in_e4m3(orc):
    for grid in (0, 1):
        for v in orc.grid_levels(grid):
            assert orc.e4m3_decode(orc.e4m3_encode(float(v))) == v


def test_philox_known_answers(orc):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) if l.strip() and l[0] != "#"]
    assert len(rows) == 3
    for r in rows:
        ctr = [int(t, 16) for t in r[0:4]]
        key = [int(t, 16) for t in r[4:6]]
        want = [int(t, 16) for t in r[6:10]]
        assert [int(v) for v in orc.philox4x32_10(ctr, key)] == want


def test_sign_mask_is_word0_of_philox_at_its_counter(orc):
    """The sign mask of a seed is word 0 of Philox4x32-10 with key (lo32, hi32)
    of the seed at counter (0, 0, 0x5349474E, 0), masked to n_h bits: the
    reading the oracle states, checked against the known-answer-pinned Philox
    (a different word, counter or key half would fail here)."""
    for seed in (0, 1, 7, 1005, 0xDEADBEEF, 2 ** 40 + 3, 2 ** 64 - 1):
        w = orc.philox4x32_10([0, 0, 0x5349474E, 0], [seed & 0xFFFFFFFF, seed >> 32])
        for n in (16, 32):
            assert orc.sign_mask_from_seed(seed, n) == int(w[0]) & ((1 << n) - 1), (seed, n)


def test_sign_mask_bits_and_determinism(orc):
    for n in (16, 32):
        masks = [orc.sign_mask_from_seed(s, n) for s in range(64)]
        assert all(m < (1 << n) for m in masks)
        assert masks == [orc.sign_mask_from_seed(s, n) for s in range(64)]
        assert len(set(masks)) > 60
    # 16-bit mask is the low half of the 32-bit one (same draw)
    assert orc.sign_mask_from_seed(5, 16) == orc.sign_mask_from_seed(5, 32) & 0xFFFF
    bits = np.array([[(orc.sign_mask_from_seed(s, 32) >> j) & 1 for j in range(32)] for s in range(512)])
    assert abs(bits.mean() - 0.5) < 0.02


def test_sr_uniform_stream_chi2(orc):
    # 2^15 consecutive indices: the 16-bit numerators fill 64 bins evenly
    r = np.array([orc.sr_uniform16(99, i, 0) for i in range(1 << 15)])
    assert r.max() < 65536
    h = np.bincount(r >> 10, minlength=64)
    e = r.size / 64
    chi2 = ((h - e) ** 2 / e).sum()
    assert chi2 < 120  # 63 dof, p ~ 1e-5
    # each uniform is half of one Philox word: cross-check two neighbours
    w = orc.philox4x32_10([0, 0, 0, 0], [99, 0])
    assert r[0] == (w[0] & 0xFFFF) and r[1] == (w[0] >> 16) and r[7] == (w[3] >> 16)
    # orientation changes the stream
    assert [orc.sr_uniform16(99, i, 1) for i in range(8)] != list(r[:8])


def test_capped_e2m1_is_e2m1_without_its_top_level(orc):
    """The range-restricted grid decodes with the E2M1 table, never produces
    code 7 (6.0), saturates at 4 and scales block maxima into [2, 4)."""
    e2 = [_decode_minifloat(k, 2, 1, 1) for k in range(8)]
    assert list(orc.grid_levels(orc.GRID_E2M1_R4)) == e2
    assert orc.grid_top(orc.GRID_E2M1_R4) == 6 and orc.grid_qmax(orc.GRID_E2M1_R4) == 4.0
    assert orc.grid_emax(orc.GRID_E2M1_R4) == 1
    assert max(orc.round_rtne(2, float(v)) & 7 for v in np.linspace(0, 100, 1001)) == 6
