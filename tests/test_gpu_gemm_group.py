"""fp4q_gemm_group: several GEMMs of one recipe in one launch over a
cost-balanced static tile list.  Every tile is computed by the same kernel code
as in a separate fp4q_gemm call, so the outputs (bf16 and fp32) must equal the
separate calls' bit for bit; fp4q_gemm's own parity against the oracle is in
test_gpu_gemm.py.  Shapes: long-K and short-K GEMMs together (the Dgrad /
Wgrad pattern of a linear layer), ragged N and K, all three MMA kinds, a group
of one, and the linear-layer sizes."""
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


def quantized(fq, rows, cols, seed, grid, scale, std=1.0):
    cfg = fq.Config(grid=grid, scale=scale, rot=16, sign_mask_row=0x2C3B, want_col=False, sf_layout=fq.SF_MMA,
                    emit_e4m3=(grid == fq.GRID_E1M2))
    x = synth.as_torch(synth.normal(rows, cols, seed, std)).cuda()
    if scale == fq.SCALE_NV:
        cfg.global_amax = None
    op, _ = fq.rht_quantize(x, cfg)
    return op


def run_group(fq, shapes, grid, scale, seed=0):
    pairs = []
    for i, (M, N, K) in enumerate(shapes):
        A = quantized(fq, M, K, seed + 10 * i + 1, grid, scale)
        B = quantized(fq, N, K, seed + 10 * i + 2, grid, scale, 0.05)
        pairs.append((A, B))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = fq.gemm_group(pairs, grid, scale, want_bf16=True, want_f32=True, status=st)
    want = [fq.gemm(A, B, grid, scale, want_bf16=True, want_f32=True) for A, B in pairs]
    torch.cuda.synchronize()
    assert st.item() == 0
    for i, ((gb, gf), (wb, wf)) in enumerate(zip(got, want)):
        assert torch.equal(gb.view(torch.int16), wb.view(torch.int16)), f"GEMM {i}: bf16 output differs"
        assert torch.equal(gf.view(torch.int32), wf.view(torch.int32)), f"GEMM {i}: fp32 output differs"


@pytest.mark.parametrize("grid,scale", [(0, 0), (0, 1), (1, 0)])
def test_group_matches_separate_calls(fq, grid, scale):
    shapes = [(1024, 512, 512),      # many short-K tiles (a Dgrad)
              (512, 512, 2048),      # few long-K tiles (a Wgrad)
              (384, 384, 640)]       # ragged N (last block of 128 columns) and K (a partial K tile)
    run_group(fq, shapes, grid, scale)


def test_group_of_one_and_four(fq):
    run_group(fq, [(256, 384, 1152)], 0, 0, seed=5)
    run_group(fq, [(128, 256, 256), (256, 128, 384), (384, 512, 1024), (128, 128, 128)], 0, 0, seed=7)


def test_group_linear_layer_backward(fq):
    """Dgrad (dY W: 16384 x 4096 x 4096) and Wgrad (dY^T X: 4096 x 4096 x 16384) in one launch."""
    grid, scale = 0, 0
    G = quantized(fq, 16384, 4096, 31, grid, scale)
    Wc = quantized(fq, 4096, 4096, 32, grid, scale, 0.02)
    Gc = quantized(fq, 4096, 16384, 33, grid, scale)
    Xc = quantized(fq, 4096, 16384, 34, grid, scale)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = fq.gemm_group([(G, Wc), (Gc, Xc)], grid, scale, want_bf16=True, want_f32=False, status=st)
    want = [fq.gemm(G, Wc, grid, scale, want_bf16=True, want_f32=False)[0],
            fq.gemm(Gc, Xc, grid, scale, want_bf16=True, want_f32=False)[0]]
    torch.cuda.synchronize()
    assert st.item() == 0
    for (gb, _), wb in zip(got, want):
        assert torch.equal(gb.view(torch.int16), wb.view(torch.int16))


def test_group_rejects(fq):
    A = quantized(fq, 128, 256, 1, 0, 0)
    with pytest.raises(fq.Fp4qError) as e:
        fq.gemm_group([], 0, 0)
    assert e.value.status == fq.ERR_INVALID_ARG
    with pytest.raises(fq.Fp4qError) as e:
        fq.gemm_group([(A, A)] * 5, 0, 0)
    assert e.value.status == fq.ERR_INVALID_ARG
    with pytest.raises(fq.Fp4qError) as e:
        fq.gemm_group([(A, A)], 0, 0, want_bf16=False, want_f32=False)
    assert e.value.status == fq.ERR_INVALID_ARG
    with pytest.raises(fq.Fp4qError) as e:
        fq.gemm_group([(A, A)], fq.GRID_E1M2, fq.SCALE_NV)
    assert e.value.status == fq.ERR_UNSUPPORTED
