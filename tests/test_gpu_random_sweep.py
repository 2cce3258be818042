"""Seeded random sweep of the quantizer and the GEMM against the oracle: shapes
(multiples of 32 for the quantizer, of 128 for the GEMM), grids, scales,
rotations, rounding, sign masks, the copies requested, the scale layout and
the E4M3 bytes drawn at random, on every input generator.  Each case is
checked exactly as the hand-picked tests check theirs."""
import random

import pytest
import torch

from fp4_microscaled_quantization_gb300 import synth
from test_gpu_gemm import check_gemm
from test_gpu_quant import run_case

pytestmark = pytest.mark.gpu

GENERATORS = [
    lambda R, C, s: synth.normal(R, C, s),
    lambda R, C, s: synth.normal_point_outliers(R, C, s),
    lambda R, C, s: synth.special_values(R, C, s),
    lambda R, C, s: synth.student_t(R, C, s),
    lambda R, C, s: synth.normal_channel_outliers(R, C, s),
]


@pytest.fixture(scope="module")
def fq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp4_microscaled_quantization_gb300 import fp4q
    fp4q.lib()
    return fp4q


@pytest.mark.parametrize("seed", range(40))
def test_quantizer_random_case(fq, orc, seed):
    rng = random.Random(7000 + seed)
    R, C = 32 * rng.randint(1, 48), 32 * rng.randint(1, 48)
    grid, scale, rot, rnd = rng.randint(0, 2), rng.randint(0, 1), rng.choice([0, 16, 32]), rng.randint(0, 1)
    want_row, want_col = rng.choice([(True, True), (True, False), (False, True)])
    b = 32 if scale == 0 else 16
    mma_ok = ((not want_row or (R % 128 == 0 and (C // b) % 4 == 0)) and
              (not want_col or (C % 128 == 0 and (R // b) % 4 == 0)))
    sf = fq.SF_MMA if (mma_ok and rng.random() < 0.5) else fq.SF_PLAIN
    mr = orc.sign_mask_from_seed(rng.randint(1, 10**6), rot) if rot else 0
    mc = orc.sign_mask_from_seed(rng.randint(1, 10**6), rot) if rot else 0
    cfg = fq.Config(grid=grid, scale=scale, rot=rot, round=rnd, sign_mask_row=mr, sign_mask_col=mc,
                    sr_seed=rng.randint(0, 2**40), want_row=want_row, want_col=want_col, sf_layout=sf,
                    emit_e4m3=rng.random() < 0.3)
    x = rng.choice(GENERATORS)(R, C, rng.randint(1, 10**6))
    run_case(fq, orc, x, cfg)


@pytest.mark.parametrize("seed", range(15))
def test_gemm_random_case(fq, orc, seed):
    rng = random.Random(9000 + seed)
    M, N, K = 128 * rng.randint(1, 10), 128 * rng.randint(1, 10), 128 * rng.randint(1, 12)
    grid, scale = rng.choice([(0, 0), (0, 1), (1, 0), (2, 0), (2, 1)])
    rot = rng.choice([0, 16])
    mask = orc.sign_mask_from_seed(rng.randint(1, 10**6), rot) if rot else 0
    a = synth.normal_channel_outliers(M, K, rng.randint(1, 10**6), 4, 20.0)
    b = synth.normal(N, K, rng.randint(1, 10**6), 0.05)
    check_gemm(fq, orc, a, b, grid, scale, rot, mask)
