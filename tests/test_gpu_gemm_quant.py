"""GPU parity of the GEMM that quantizes its own output (fp4q_gemm_quantize):
its row-wise copy must equal, bit for bit, fp4q_rht_quantize of the bf16
output that the same call stores (codes, scales, E4M3 bytes), for every grid,
rotation and rounding mode of the output copy; and the bf16 output must equal
the plain GEMM's.  The plain GEMM and the quantizer are themselves held to the
oracle by test_gpu_gemm.py and test_gpu_quant.py."""
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


def operands(fq, M, N, K, grid, scale):
    a = synth.normal_channel_outliers(M, K, M + 7 * K, 4, 20.0)
    b = synth.normal(N, K, N + 5 * K, 0.05)
    cfg = fq.Config(grid=grid, scale=scale, rot=16, sign_mask_row=0x3C5A, want_col=False, sf_layout=fq.SF_MMA,
                    emit_e4m3=(grid == fq.GRID_E1M2))
    A, _ = fq.rht_quantize(synth.as_torch(a).cuda(), cfg)
    B, _ = fq.rht_quantize(synth.as_torch(b).cuda(), cfg)
    return A, B


def check(fq, A, B, grid, scale, ocfg, M, N):
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
    check(fq, A, B, 0, 0, ocfg, M, N)


@pytest.mark.parametrize("grid,scale", [(0, 1), (1, 0), (2, 0)])
def test_input_kinds_and_plain_scales(fq, grid, scale):
    M, N, K = 384, 256, 640 if scale == 1 else 768
    A, B = operands(fq, M, N, K, grid, scale)
    ocfg = fq.Config(grid=1 if grid == 1 else 0, rot=16, sign_mask_row=0x1234, want_col=False,
                     sf_layout=fq.SF_PLAIN)
    check(fq, A, B, grid, scale, ocfg, M, N)


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
