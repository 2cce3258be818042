"""Pins of the oracle's quantized copies: the MX shared-exponent closed form,
nearest-code brute force per element, NV-style scale invariants, packing,
the GEMM-ready E4M3 bytes, exact dequantization and the column-wise layout."""
import numpy as np
import pytest

from fp4_microscaled_quantization_gb300 import synth

LEVELS = {0: np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64),
          1: np.array([0, 0.25, 0.5, 0.75, 1, 1.25, 1.5, 1.75], np.float64),
          2: np.array([0, 0.5, 1, 1.5, 2, 3, 4], np.float64)}      # E2M1 capped at 4
EMAX = {0: 2, 1: 0, 2: 1}


def unpack(codes: np.ndarray) -> np.ndarray:
    lo = codes & 15
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def rotated_rows(orc, x_bits, n_h, mask):
    y = synth.bf16_bits_to_f32(x_bits).astype(np.float32).copy()
    if n_h:
        for r in range(y.shape[0]):
            for c0 in range(0, y.shape[1], n_h):
                y[r, c0:c0 + n_h] = orc.rotate_block(y[r, c0:c0 + n_h], n_h, mask)
    return y


@pytest.mark.parametrize("grid", [0, 1, 2])
@pytest.mark.parametrize("n_h", [0, 16, 32])
def test_mx_exponent_closed_form_and_nearest_code(orc, grid, n_h):
    x = synth.special_values(64, 128, 11)
    mask = orc.sign_mask_from_seed(3, n_h) if n_h else 0
    q = orc.quantize(x, 0, grid, orc.SCALE_MX, n_h, mask)
    y = rotated_rows(orc, x, n_h, mask)
    codes = unpack(q["codes"])
    L = LEVELS[grid]
    for r in range(y.shape[0]):
        for kb in range(y.shape[1] // 32):
            blk = y[r, kb * 32:(kb + 1) * 32].astype(np.float64)
            m = np.abs(blk).max()
            s = int(q["scales"][r, kb])
            e = s - 127
            if m == 0:
                assert s == 0
            elif e > -127:
                # closed form: the block max lands in [2^e_max, 2^(e_max+1)) grid units
                assert 2.0 ** (e + EMAX[grid]) <= m < 2.0 ** (e + EMAX[grid] + 1)
            else:
                assert m < 2.0 ** (-127 + EMAX[grid] + 1)
            # every code is the nearest grid value of y / 2^e (ties to even, saturating)
            for t in range(32):
                v = blk[t] * 2.0 ** -e
                c = int(codes[r, kb * 32 + t])
                a = abs(v)
                if a >= L[-1]:
                    assert c & 7 == len(L) - 1
                else:
                    d = np.abs(a - L)
                    cand = np.flatnonzero(d == d.min())
                    assert (c & 7) in cand
                    if cand.size == 2:
                        assert (c & 7) % 2 == 0
                assert bool(c & 8) == bool(np.signbit(np.float32(blk[t])))


def test_all_zero_block_and_packing(orc):
    x = np.zeros((1, 64), np.float32)
    x[0, 32] = 6.0      # element 0 of block 1: code 7 in the low nibble of byte 16
    x[0, 33] = -0.0
    x[0, 1] = -0.0      # block 0 stays all zero
    bits = synth.to_bf16_bits(x)
    q = orc.quantize(bits, 0, orc.GRID_E2M1, orc.SCALE_MX, 0)
    assert q["scales"][0, 0] == 0
    assert q["codes"][0, 0] == 0x80          # element 1 is -0 -> code 8 in the high nibble
    assert q["codes"][0, 16] == 0x87         # 6.0 -> 7 (low), -0 -> 8 (high)
    assert q["scales"][0, 1] == 127 + 0      # m = 6: floor(log2 6) - 2 = 0


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_mx_dequant_is_exact(orc, grid):
    x = synth.special_values(32, 256, 12)
    q = orc.quantize(x, 0, grid, orc.SCALE_MX, 16, 0)
    d = orc.dequantize(q["codes"], q["scales"], 0.0, grid, orc.SCALE_MX)
    codes = unpack(q["codes"])
    want = np.where(codes & 8, -1.0, 1.0) * LEVELS[grid][codes & 7] * \
        np.exp2(np.repeat(q["scales"].astype(np.float64) - 127, 32, axis=1))
    assert np.array_equal(d.astype(np.float64), want)


@pytest.mark.parametrize("grid", [0, 1, 2])
@pytest.mark.parametrize("n_h", [16, 32])
def test_nv_invariants(orc, grid, n_h):
    x = synth.normal(64, 256, 21, 0.02)
    q = orc.quantize(x, 0, grid, orc.SCALE_NV, n_h, 0)
    y = rotated_rows(orc, x, n_h, 0).astype(np.float64)
    G = np.abs(y).max()
    qmax = LEVELS[grid][-1]
    S_t = q["tensor_scale"]
    assert abs(S_t * 448 * qmax / G - 1) < 2e-7
    # the block that holds G gets the largest E4M3 scale
    r, c = np.unravel_index(np.argmax(np.abs(y)), y.shape)
    assert q["scales"][r, c // 16] == 0x7E
    d = orc.dequantize(q["codes"], q["scales"], S_t, grid, orc.SCALE_NV)
    assert np.all(np.abs(d) <= qmax * 448 * S_t * (1 + 2 ** -3))
    # without S_t the reconstruction is code * E4M3 scale exactly
    d0 = orc.dequantize(q["codes"], q["scales"], S_t, grid, orc.SCALE_NV, with_tensor_scale=False)
    codes = unpack(q["codes"])
    sb = np.array([orc.e4m3_decode(b) for b in range(256)])[q["scales"]]
    want0 = np.where(codes & 8, -1.0, 1.0) * LEVELS[grid][codes & 7] * np.repeat(sb, 16, axis=1)
    assert np.array_equal(d0.astype(np.float64), want0)
    assert np.allclose(d.astype(np.float64), want0 * S_t, rtol=2 ** -23, atol=0)
    # per-block error: nearest code of y / (sb * S_t) up to the rounding of that step
    err = np.abs(d.astype(np.float64) - y)
    step = np.repeat(sb * S_t, 16, axis=1) * (LEVELS[grid][-1] - LEVELS[grid][-2])
    assert np.all(err <= step / 2 * (1 + 1e-5) + 1e-30)


def test_nv_zero_tensor_and_given_amax(orc):
    z = synth.to_bf16_bits(np.zeros((16, 64), np.float32))
    q = orc.quantize(z, 0, 0, orc.SCALE_NV, 16, 0)
    assert q["tensor_scale"] == 0 and not q["scales"].any() and not (q["codes"] & 0x77).any()
    x = synth.normal(16, 64, 3, 1.0)
    q1 = orc.quantize(x, 0, 0, orc.SCALE_NV, 16, 0)
    G = q1["tensor_scale"] * np.float32(2688.0)
    q2 = orc.quantize(x, 0, 0, orc.SCALE_NV, 16, 0, given_amax=float(np.float32(G)) * 4)
    assert q2["tensor_scale"] > q1["tensor_scale"]
    assert q2["scales"].max() < 0x7E


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_e4m3_bytes_hold_the_code_values(orc, grid):
    x = synth.special_values(32, 128, 5)
    q = orc.quantize(x, 0, grid, orc.SCALE_MX, 16, 0, want_e4m3=True)
    codes = unpack(q["codes"])
    dec = np.array([orc.e4m3_decode(b) for b in range(256)])[q["e4m3"]]
    want = np.where(codes & 8, -1.0, 1.0) * LEVELS[grid][codes & 7]
    assert np.array_equal(dec, want)
    assert np.array_equal(np.signbit(dec), (codes & 8) > 0)


def test_colwise_copy_is_blocks_along_rows(orc):
    """A single outlier row inflates only the row-wise scales of that row but
    the column-wise scales of every column block that contains it."""
    x = np.ones((64, 64), np.float32)
    x[5, :] = 1000.0
    bits = synth.to_bf16_bits(x)
    qr = orc.quantize(bits, 0, 0, orc.SCALE_MX, 0)
    qc = orc.quantize(bits, 1, 0, orc.SCALE_MX, 0)
    assert qr["codes"].shape == (64, 32) and qc["codes"].shape == (64, 32)
    big_r = qr["scales"] > 127
    assert big_r[5].all() and big_r.sum() == 2
    big_c = qc["scales"] > 127
    assert big_c[:, 0].all() and not big_c[:, 1].any()


def test_sr_uses_stored_index(orc):
    """SR on the column-wise copy draws from its own (orient=1) stream: the
    row-wise copy of the transpose has the same blocks and scales but other
    random draws, while under RTNE the two agree code for code."""
    x = synth.student_t(64, 96, 9)
    xt = np.ascontiguousarray(x.T)
    qc = orc.quantize(x, 1, 1, orc.SCALE_MX, 16, 0, orc.SR, 77)
    q_t = orc.quantize(xt, 0, 1, orc.SCALE_MX, 16, 0, orc.SR, 77)
    assert np.array_equal(qc["scales"], q_t["scales"])
    assert not np.array_equal(qc["codes"], q_t["codes"])
    # RTNE does not depend on the stream
    qc0 = orc.quantize(x, 1, 1, orc.SCALE_MX, 16, 0, orc.RTNE)
    qt0 = orc.quantize(xt, 0, 1, orc.SCALE_MX, 16, 0, orc.RTNE)
    assert np.array_equal(qc0["codes"], qt0["codes"])


def test_rejects_nonfinite_and_ragged(orc):
    x = synth.normal(32, 64, 1)
    bad = x.copy()
    bad[3, 7] = 0x7F80  # +inf in bf16
    with pytest.raises(orc.OracleError):
        orc.quantize(bad, 0, 0, orc.SCALE_MX, 16)
    with pytest.raises(orc.OracleError):
        orc.quantize(synth.normal(32, 48, 1), 0, 0, orc.SCALE_MX, 16)
