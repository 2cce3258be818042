"""GPU parity of the tcgen05 block-scaled GEMM against the oracle's fp64 GEMM
of the same (oracle-)quantized operands.

Tolerances: fp32 output within 1e-3 relative Frobenius error of the fp64
result; bf16 output equal to the bf16 rounding of the fp32-accuracy result for
>= 99.9% of entries and within 1 bf16 ulp everywhere (bf16 rounding alone is
~1.6e-3 RMS relative, larger than the fp32 bound)."""
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


def plain_to_mma(plain: np.ndarray) -> np.ndarray:
    rows, nkb = plain.shape
    r = np.arange(rows)[:, None]
    k = np.arange(nkb)[None, :]
    off = ((r // 128) * (nkb // 4) + k // 4) * 512 + 16 * (r % 32) + 4 * ((r // 32) % 4) + k % 4
    out = np.zeros(rows * nkb, np.uint8)
    out[off.reshape(-1)] = plain.reshape(-1)
    return out.reshape(rows, nkb)


def oracle_operand(orc, bits, grid, scale, rot, mask):
    q = orc.quantize(bits, 0, grid, scale, rot, mask)
    deq = orc.dequantize(q["codes"], q["scales"], q["tensor_scale"], grid, scale, with_tensor_scale=False)
    return q, deq


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_gemm(fq, orc, a_bits, b_bits, grid, scale, rot=16, mask=0):
    cfg = fq.Config(grid=grid, scale=scale, rot=rot, sign_mask_row=mask, want_col=False, sf_layout=fq.SF_MMA,
                    emit_e4m3=(grid == fq.GRID_E1M2))
    A, _ = fq.rht_quantize(synth.as_torch(a_bits).cuda(), cfg)
    B, _ = fq.rht_quantize(synth.as_torch(b_bits).cuda(), cfg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Dh, Df = fq.gemm(A, B, grid, scale, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    qa, da = oracle_operand(orc, a_bits, grid, scale, rot, mask)
    qb, db = oracle_operand(orc, b_bits, grid, scale, rot, mask)
    # the operands themselves are bit-exact (the quantizer parity tests), so the
    # oracle GEMM below is the GEMM of exactly what the kernel consumed
    assert np.array_equal(A.codes.cpu().numpy(), qa["codes"])
    alpha = float(np.float64(qa["tensor_scale"]) * np.float64(qb["tensor_scale"])) if scale == fq.SCALE_NV else 1.0
    want = orc.gemm_ref(da, db, alpha)
    got = Df.double().cpu().numpy()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert rel <= 1e-3, f"relative Frobenius error {rel:.3e}"
    # bf16 output: the rounding of the fp32 result
    hb = bf16_bits(Dh).astype(np.int32)
    wb = synth.to_bf16_bits(got.astype(np.float32)).astype(np.int32)
    diff = np.abs(hb - wb)
    assert (diff == 0).mean() >= 0.999 and diff.max() <= 1
    return rel


@pytest.mark.parametrize("grid,scale", [(0, 0), (0, 1), (1, 0), (2, 0), (2, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 384, 512), (128, 128, 640), (384, 256, 1152)])
def test_gemm_small(fq, orc, grid, scale, M, N, K):
    a = synth.normal_channel_outliers(M, K, M + K, 4, 20.0)
    b = synth.normal(N, K, N + 3 * K, 0.05)
    check_gemm(fq, orc, a, b, grid, scale, 16, orc.sign_mask_from_seed(M * N, 16))


@pytest.mark.parametrize("grid", [0, 1])
@pytest.mark.parametrize("M,N,K", [(256, 640, 512), (384, 896, 256), (256, 4096, 1024)])
def test_gemm_exact_tile_edges(fq, orc, grid, M, N, K):
    """Grid-valued operands (unit MX scales, synth.grid_valued) make D = A B^T
    exact in fp32, so the fp32 output equals the oracle's bit for bit and the
    bf16 output is its rounding: every element of every tile, in both row
    groups of the pair and in the 128-column tails of N = 640 and 896
    (kind::mxf4 for E2M1, mxf8f6f4 for E1M2)."""
    a = synth.grid_valued(M, K, 5 * M + K + grid, grid)
    b = synth.grid_valued(N, K, 7 * N + K + grid, grid)
    cfg = fq.Config(grid=grid, rot=0, want_col=False, sf_layout=fq.SF_MMA, emit_e4m3=(grid == fq.GRID_E1M2))
    A, _ = fq.rht_quantize(synth.as_torch(a).cuda(), cfg)
    B, _ = fq.rht_quantize(synth.as_torch(b).cuda(), cfg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Dh, Df = fq.gemm(A, B, grid, fq.SCALE_MX, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _, da = oracle_operand(orc, a, grid, 0, 0, 0)
    _, db = oracle_operand(orc, b, grid, 0, 0, 0)
    D = orc.gemm_ref(da, db)
    D32 = D.astype(np.float32)
    assert np.array_equal(D, D32.astype(np.float64))   # exact in fp32
    got = Df.cpu().numpy()
    bad = np.argwhere(got.view(np.uint32) != D32.view(np.uint32))
    assert bad.size == 0, f"{len(bad)} fp32 entries differ, first at {bad[:4].tolist()}"
    assert np.array_equal(bf16_bits(Dh), synth.to_bf16_bits(D32))


def test_gemm_nv_partial_k_tiles(fq, orc):
    # K = 320: NV-style K tiles of 256 + 64 (one MMA in the last tile)
    a = synth.normal(128, 320, 1)
    b = synth.normal(256, 320, 2)
    check_gemm(fq, orc, a, b, 0, 1, 32, 0x12345678)


def test_gemm_rejects(fq):
    cfg = fq.Config(want_col=False, sf_layout=fq.SF_MMA)
    A, _ = fq.rht_quantize(synth.as_torch(synth.normal(128, 256, 3)).cuda(), cfg)
    with pytest.raises(fq.Fp4qError) as e:
        fq.gemm(A, A, fq.GRID_E1M2, fq.SCALE_NV)
    assert e.value.status == fq.ERR_UNSUPPORTED
    A.rows = 96
    with pytest.raises(fq.Fp4qError):
        fq.gemm(A, A, fq.GRID_E2M1, fq.SCALE_MX)
