"""Pins of the oracle's rounding onto the 4-bit grids.

RTNE: brute force over every finite bf16 value (and fp32 neighbours of every
midpoint) against an argmin over the grid built from the bit format.
Conditional error per level: the page's (l_i - r_i)/2 (golden fixture), by
stratified integration over the bins the oracle's RTNE induces.
SR: the exact closed form of the round-up probability and an unbiasedness
test through the Philox stream."""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

LEVELS = {
    0: np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64),          # E2M1 from its bit format
    1: np.array([0, 0.25, 0.5, 0.75, 1, 1.25, 1.5, 1.75], np.float64),  # E1M2 from its bit format
    2: np.array([0, 0.5, 1, 1.5, 2, 3, 4], np.float64),             # E2M1 capped at 4
}


def argmin_code(grid: int, v: np.float32) -> int:
    L = LEVELS[grid]
    sign = 8 if np.signbit(v) else 0
    a = abs(float(v))
    if a >= L[-1]:
        return sign | (len(L) - 1)
    d = np.abs(a - L)
    cand = np.flatnonzero(d == d.min())
    if cand.size == 1:
        return sign | int(cand[0])
    even = [int(c) for c in cand if c % 2 == 0]
    assert len(cand) == 2 and len(even) == 1
    return sign | even[0]


def all_finite_bf16() -> np.ndarray:
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_rtne_all_bf16_values(orc, grid):
    vals = all_finite_bf16()
    # restrict to the part of the range where codes change (|v| <= 16) plus a sample beyond
    small = vals[np.abs(vals) <= 16]
    big = vals[np.abs(vals) > 16][::97]
    for v in np.concatenate([small, big]):
        assert orc.round_rtne(grid, float(v)) == argmin_code(grid, v), v


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_rtne_midpoints_and_neighbours(orc, grid):
    L = LEVELS[grid].astype(np.float32)
    mids = (L[:-1] + L[1:]) / np.float32(2)
    for m in mids:
        for v in (m, np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(10))):
            for s in (1, -1):
                vv = np.float32(s * v)
                assert orc.round_rtne(grid, float(vv)) == argmin_code(grid, vv)
    # ties go to the even code
    for k, m in enumerate(mids):
        assert orc.round_rtne(grid, float(m)) & 7 == (k if k % 2 == 0 else k + 1)
    # -0 keeps its sign, saturation at q_max
    top = len(L) - 1
    assert orc.round_rtne(grid, -0.0) == 8
    assert orc.round_rtne(grid, float(L[-1]) * 100) == top
    assert orc.round_rtne(grid, -float(L[-1]) * 1.01) == 8 | top


def _golden_cond_error():
    out = []
    for line in open(os.path.join(GOLDEN, "conditional_error.txt")):
        if line.strip() and not line.startswith("#"):
            g, lvl, want = line.split()
            out.append(({"e2m1": 0, "e1m2": 1, "e2m1r4": 2}[g], float(lvl), float(want)))
    return out


def test_conditional_expected_error_per_level(orc):
    """E[q - x | RTNE(x) = q] for x uniform: the page's (l_i - r_i)/2."""
    cases = _golden_cond_error()
    for grid in (0, 1, 2):
        qmax = LEVELS[grid][-1]
        N = 120_000
        xs = (np.arange(N) + 0.5) / N * qmax
        codes = np.array([orc.round_rtne(grid, float(x)) for x in xs.astype(np.float32)])
        q = LEVELS[grid][codes & 7]
        for g, lvl, want in cases:
            if g != grid:
                continue
            sel = q == lvl
            assert sel.sum() > 1000
            got = float(np.mean(q[sel] - xs[sel]))
            assert abs(got - want) < 2e-4 * max(1.0, lvl), (grid, lvl, got, want)
    # the sign of the bias for every E2M1 level is never positive: shrinkage
    assert all(w <= 0 for g, _, w in cases if g == 0)


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_sr_round_up_probability_closed_form(orc, grid):
    L = LEVELS[grid]
    rng = np.random.default_rng(grid)
    vs = list(rng.uniform(0, 0.99 * L[-1], 6).astype(np.float32)) + [np.float32(L[3]), np.float32((L[2] + L[3]) / 2)]
    for v in vs:
        k = int(np.searchsorted(L, float(v), side="right") - 1)
        f = (float(v) - L[k]) / (L[k + 1] - L[k])
        codes = np.array([orc.round_sr(grid, float(v), r) for r in range(1 << 16)])
        ups = int(np.sum((codes & 7) == k + 1))
        assert np.all(((codes & 7) == k) | ((codes & 7) == k + 1))
        assert ups == int(np.ceil(f * 65536))
        # E[SR(v)] - v = gap * (ceil(f 2^16)/2^16 - f), in [0, gap * 2^-16)
        mean = np.mean(L[codes & 7])
        bias = mean - float(v)
        gap = L[k + 1] - L[k]
        assert 0 <= bias + 1e-15 and bias < gap * 2 ** -16
    # saturation and exact levels
    assert all(orc.round_sr(grid, float(L[-1]) * 2, r) == len(L) - 1 for r in (0, 1, 65535))
    assert all(orc.round_sr(grid, float(L[2]), r) == 2 for r in (0, 1, 65535))
    assert orc.round_sr(grid, -float(L[1]), 0) == 9


def test_sr_unbiased_through_philox(orc):
    grid = 1
    v = np.float32(0.6)   # between 0.5 and 0.75
    n = 200_000
    vals = np.array([orc.code_value(grid, orc.round_sr(grid, float(v), orc.sr_uniform16(1234, i, 0)))
                     for i in range(n)])
    sigma = np.sqrt(0.4 * 0.6) * 0.25 / np.sqrt(n)
    assert abs(vals.mean() - float(v)) < 5 * sigma
