"""Pins of the oracle's blockwise Hadamard rotation: the Hadamard matrix built
independently from the closed form H_ij = (-1)^popcount(i & j), H H^T = n I,
exactness on integer inputs, the fp32 error bound on random inputs, and the
sign-flip / inverse relations."""
import numpy as np
import pytest


def hadamard(n: int) -> np.ndarray:
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def c_of(n):
    return np.float32(0.25) if n == 16 else np.float32(1.0 / np.sqrt(32.0))


def test_c32_is_fp32_rounding_of_inverse_sqrt32():
    assert np.float32(1.0 / np.sqrt(32.0)).view(np.uint32) == 0x3E3504F3


@pytest.mark.parametrize("n", [16, 32])
def test_unit_vectors_give_hadamard_columns(orc, n):
    H = hadamard(n)
    c = c_of(n)
    cols = []
    for j in range(n):
        e = np.zeros(n, np.float32)
        e[j] = 1.0
        y = orc.rotate_block(e, n, 0)
        assert np.array_equal(y, (H[:, j] * c).astype(np.float32))
        cols.append(np.rint(y / c).astype(np.int64))
    Hm = np.stack(cols, axis=1)
    assert np.array_equal(Hm @ Hm.T, n * np.eye(n, dtype=np.int64))


@pytest.mark.parametrize("n", [16, 32])
def test_integer_inputs_are_exact(orc, n):
    rng = np.random.default_rng(n)
    H = hadamard(n)
    for _ in range(200):
        x = rng.integers(-(1 << 19), 1 << 19, n)
        y = orc.rotate_block(x.astype(np.float32), n, 0)
        want = (H @ x).astype(np.float32) * c_of(n)   # one fp32 rounding of an exact integer
        assert np.array_equal(y, want)


@pytest.mark.parametrize("n", [16, 32])
def test_random_inputs_within_fp32_bound(orc, n):
    rng = np.random.default_rng(100 + n)
    H = hadamard(n).astype(np.float64)
    u = 2.0 ** -24
    stages = int(np.log2(n))
    for _ in range(500):
        x = (rng.standard_normal(n) * np.exp(rng.uniform(-8, 8, n))).astype(np.float32)
        y = orc.rotate_block(x, n, 0).astype(np.float64)
        exact = (H @ x.astype(np.float64)) / np.sqrt(n)
        bound = (stages + 2) * u * np.abs(x).astype(np.float64).sum() / np.sqrt(n) * 1.01
        assert np.all(np.abs(y - exact) <= bound)


@pytest.mark.parametrize("n", [16, 32])
def test_sign_mask_is_a_pre_flip(orc, n):
    rng = np.random.default_rng(3)
    for mask in (0x1, 0xA5A5 & ((1 << n) - 1), (1 << n) - 1, orc.sign_mask_from_seed(11, n)):
        x = rng.standard_normal(n).astype(np.float32)
        s = np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(n)], np.float32)
        assert np.array_equal(orc.rotate_block(x, n, mask), orc.rotate_block(x * s, n, 0))


def test_inverse_h16_exact_on_integers(orc):
    rng = np.random.default_rng(5)
    for mask in (0, 0x3C5A):
        x = rng.integers(-1000, 1000, 16).astype(np.float32)
        assert np.array_equal(orc.unrotate_block(orc.rotate_block(x, 16, mask), 16, mask), x)


def test_rotation_preserves_norm(orc):
    rng = np.random.default_rng(6)
    for n in (16, 32):
        x = rng.standard_normal(n).astype(np.float32)
        y = orc.rotate_block(x, n, orc.sign_mask_from_seed(1, n))
        assert abs(np.linalg.norm(y.astype(np.float64)) / np.linalg.norm(x.astype(np.float64)) - 1) < 1e-6
        z = orc.unrotate_block(y, n, orc.sign_mask_from_seed(1, n))
        assert np.allclose(z, x, rtol=0, atol=1e-6 * np.abs(x).max())
