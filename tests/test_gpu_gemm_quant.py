"""GPU parity of the GEMM that quantizes its own output (fp4q_gemm_quantize).

Against the oracle: on operands whose entries are grid values with unit
block scales (synth.grid_valued), every product is a multiple of 1/4 (1/16)
and every sum stays exact in fp32 for K <= 4096, so D is exact whatever the
summation order.  The oracle forms D itself (fp64 GEMM of its own quantized
operands), rounds it to bf16 and quantizes that with its own quantizer; the
kernel's bf16 output must equal the oracle's bf16(D) and its output copy the
oracle's copy, bit for bit (codes, scales, E4M3 bytes), for every grid,
rotation and rounding of the output copy, both input kinds with MX scales,
and at the linear layer's Fprop shape (sampled rows, RTNE).

Against the library's own calls (general operands): the output copy equals
fp4q_rht_quantize of the bf16 D the same call stores, and that D equals the
plain GEMM's."""
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


def mma_to_plain(flat, rows, nkb):
    r = np.arange(rows)[:, None]
    k = np.arange(nkb)[None, :]
    off = ((r // 128) * (nkb // 4) + k // 4) * 512 + 16 * (r % 32) + 4 * ((r // 32) % 4) + k % 4
    return flat.reshape(-1)[off]


def exact_case(fq, orc, M, N, K, grid, rows=None):
    """GPU operands of grid-valued inputs, and the oracle's bf16 bits of D = A B^T
    (exact) for the given rows (all by default)."""
    a = synth.grid_valued(M, K, 11 * M + K + grid, grid)
    b = synth.grid_valued(N, K, 13 * N + K + grid, grid)
    cfg = fq.Config(grid=grid, rot=0, want_col=False, sf_layout=fq.SF_MMA, emit_e4m3=(grid == fq.GRID_E1M2))
    A, _ = fq.rht_quantize(synth.as_torch(a).cuda(), cfg)
    B, _ = fq.rht_quantize(synth.as_torch(b).cuda(), cfg)
    sel = slice(None) if rows is None else rows
    qa = orc.quantize(np.ascontiguousarray(a[sel]), 0, grid, 0, 0)
    qb = orc.quantize(b, 0, grid, 0, 0)
    da = orc.dequantize(qa["codes"], qa["scales"], 0.0, grid, 0)
    db = orc.dequantize(qb["codes"], qb["scales"], 0.0, grid, 0)
    D = orc.gemm_ref(da, db)
    assert np.array_equal(D, D.astype(np.float32).astype(np.float64))   # exact in fp32
    return A, B, synth.to_bf16_bits(D.astype(np.float32))


def check_against_oracle(fq, orc, A, B, grid, d_bits, ocfg, rows=None):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    D, q = fq.gemm_quantize(A, B, grid, fq.SCALE_MX, ocfg, want_bf16=True, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    sel = slice(None) if rows is None else rows
    got_d = D.view(torch.int16).cpu().numpy().view(np.uint16)[sel]
    assert np.array_equal(got_d, d_bits), "bf16 D differs from the oracle's exact D"
    ref = orc.quantize(d_bits, 0, ocfg.grid, fq.SCALE_MX, ocfg.rot, ocfg.sign_mask_row, ocfg.round, ocfg.sr_seed,
                       want_e4m3=bool(ocfg.emit_e4m3))
    M, N = D.shape
    codes = q.codes.cpu().numpy()[sel]
    assert np.array_equal(codes, ref["codes"]), f"{int(np.count_nonzero(codes != ref['codes']))} code bytes differ"
    sc = q.scales.cpu().numpy()
    sc = mma_to_plain(sc, M, N // 32) if ocfg.sf_layout == fq.SF_MMA else sc.reshape(M, N // 32)
    assert np.array_equal(sc[sel], ref["scales"])
    if ocfg.emit_e4m3:
        assert np.array_equal(q.e4m3.cpu().numpy()[sel], ref["e4m3"])


@pytest.mark.parametrize("ogrid,rot,rnd", list(itertools.product([0, 1, 2], [0, 16, 32], [0, 1])))
def test_output_copy_matches_oracle(fq, orc, ogrid, rot, rnd):
    M, N, K = 256, 384, 512
    A, B, d_bits = exact_case(fq, orc, M, N, K, 0)
    ocfg = fq.Config(grid=ogrid, rot=rot, round=rnd, sign_mask_row=0x5A3C if rot else 0, sr_seed=777,
                     want_col=False, sf_layout=fq.SF_MMA if rot != 32 else fq.SF_PLAIN, emit_e4m3=(ogrid == 1))
    check_against_oracle(fq, orc, A, B, 0, d_bits, ocfg)


def test_e1m2_inputs_output_copy_matches_oracle(fq, orc):
    """E1M2 operands (kind::mxf8f6f4 on their E4M3 bytes), E1M2 output copy with SR."""
    A, B, d_bits = exact_case(fq, orc, 384, 256, 768, 1)
    ocfg = fq.Config(grid=1, rot=16, round=fq.SR, sign_mask_row=0x0FF0, sr_seed=99, want_col=False,
                     sf_layout=fq.SF_MMA, emit_e4m3=True)
    check_against_oracle(fq, orc, A, B, 1, d_bits, ocfg)


def test_layer_fprop_output_copy_matches_oracle(fq, orc):
    """The linear layer's Fprop shape, 16384 x 4096 x 4096: rows sampled from
    the start, the middle and the end of the output (RTNE; the element index of
    stochastic rounding is that of the whole copy)."""
    M, N, K = 16384, 4096, 4096
    rows = np.r_[0:128, 8192:8320, M - 128:M]
    A, B, d_bits = exact_case(fq, orc, M, N, K, 0, rows)
    ocfg = fq.Config(grid=0, rot=16, sign_mask_row=0x6B2D, want_col=False, sf_layout=fq.SF_MMA)
    check_against_oracle(fq, orc, A, B, 0, d_bits, ocfg, rows)


def operands(fq, M, N, K, grid, scale):
    a = synth.normal_channel_outliers(M, K, M + 7 * K, 4, 20.0)
    b = synth.normal(N, K, N + 5 * K, 0.05)
    cfg = fq.Config(grid=grid, scale=scale, rot=16, sign_mask_row=0x3C5A, want_col=False, sf_layout=fq.SF_MMA,
                    emit_e4m3=(grid == fq.GRID_E1M2))
    A, _ = fq.rht_quantize(synth.as_torch(a).cuda(), cfg)
    B, _ = fq.rht_quantize(synth.as_torch(b).cuda(), cfg)
    return A, B


def check_self(fq, A, B, grid, scale, ocfg, M, N):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    D, q = fq.gemm_quantize(A, B, grid, scale, ocfg, want_bf16=True, status=st)
    Dref, _ = fq.gemm(A, B, grid, scale, want_f32=False)
    ro, _ = fq.rht_quantize(D, ocfg)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(D.view(torch.int16), Dref.view(torch.int16))
    assert torch.equal(q.codes, ro.codes)
    assert torch.equal(q.scales, ro.scales)
    if ocfg.emit_e4m3:
        assert torch.equal(q.e4m3, ro.e4m3)


@pytest.mark.parametrize("ogrid,rot,rnd", list(itertools.product([0, 1, 2], [0, 16, 32], [0, 1])))
def test_output_copy_all_modes(fq, ogrid, rot, rnd):
    M, N, K = 256, 384, 512
    A, B = operands(fq, M, N, K, 0, 0)
    ocfg = fq.Config(grid=ogrid, rot=rot, round=rnd, sign_mask_row=0x9E37 if rot else 0, sr_seed=4242,
                     want_col=False, sf_layout=fq.SF_MMA, emit_e4m3=(ogrid == 1))
    check_self(fq, A, B, 0, 0, ocfg, M, N)


@pytest.mark.parametrize("grid,scale", [(0, 1), (1, 0), (2, 0)])
def test_input_kinds_and_plain_scales(fq, grid, scale):
    M, N, K = 384, 256, 640 if scale == 1 else 768
    A, B = operands(fq, M, N, K, grid, scale)
    ocfg = fq.Config(grid=1 if grid == 1 else 0, rot=16, sign_mask_row=0x1234, want_col=False,
                     sf_layout=fq.SF_PLAIN)
    check_self(fq, A, B, grid, scale, ocfg, M, N)


def test_quantize_only_and_layer_size(fq):
    """No bf16 output requested; the linear layer's Fprop shape (16384x4096x4096)."""
    M, N, K = 16384, 4096, 4096
    X = synth.as_torch(synth.act_x(M, K)).cuda()
    W = synth.as_torch(synth.weight_w(N, K)).cuda()
    cfg = fq.Config(rot=16, sign_mask_row=0x7A1F, want_col=False, sf_layout=fq.SF_MMA)
    A, _ = fq.rht_quantize(X, cfg)
    B, _ = fq.rht_quantize(W, cfg)
    ocfg = fq.Config(rot=16, sign_mask_row=0x0F0F, want_col=False, sf_layout=fq.SF_MMA)
    _, q = fq.gemm_quantize(A, B, 0, 0, ocfg)
    Dref, _ = fq.gemm(A, B, 0, 0, want_f32=False)
    ro, _ = fq.rht_quantize(Dref, ocfg)
    torch.cuda.synchronize()
    assert torch.equal(q.codes, ro.codes) and torch.equal(q.scales, ro.scales)


def test_rejects(fq):
    A, B = operands(fq, 128, 128, 256, 0, 0)
    for bad in (fq.Config(scale=fq.SCALE_NV, want_col=False), fq.Config(want_col=True)):
        with pytest.raises(fq.Fp4qError) as e:
            fq.gemm_quantize(A, B, 0, 0, bad, out=fq.alloc_operand(128, 128, fq.Config(want_col=False), "cuda"))
        assert e.value.status == fq.ERR_UNSUPPORTED
