"""Guard regions around every output: each output tensor is a view into a larger
buffer whose bytes before and after it hold a canary pattern, which must be
intact after the call.  Catches writes that run past an output's ends (the
parity tests compare the bytes inside the outputs)."""
import itertools

import pytest
import torch

from fp4_microscaled_quantization_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096      # canary bytes on each side (keeps the view 16-byte aligned)
CANARY = 0xA5


@pytest.fixture(scope="module")
def fq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp4_microscaled_quantization_gb300 import fp4q
    fp4q.lib()
    return fp4q


class Guarded:
    def __init__(self):
        self.bufs = []

    def tensor(self, shape, dtype):
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        buf = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.bufs.append((buf, nbytes))
        return buf[GUARD:GUARD + nbytes].view(dtype).view(*shape)

    def operand(self, fq, rows, cols, cfg):
        b = cfg.block
        return fq.Operand(
            codes=self.tensor((rows, cols // 2), torch.uint8),
            scales=self.tensor((rows, cols // b), torch.uint8),
            tensor_scale=self.tensor((1,), torch.float32) if cfg.scale == fq.SCALE_NV else None,
            e4m3=self.tensor((rows, cols), torch.uint8) if cfg.emit_e4m3 else None,
            rows=rows, cols=cols, grid=cfg.grid, scale=cfg.scale, sf_layout=cfg.sf_layout)

    def check(self):
        torch.cuda.synchronize()
        for buf, nbytes in self.bufs:
            head, tail = buf[:GUARD], buf[GUARD + nbytes:]
            assert bool((head == CANARY).all()), "bytes before an output were written"
            assert bool((tail == CANARY).all()), "bytes after an output were written"


@pytest.mark.parametrize("grid,scale,rot,rnd", [(0, 0, 16, 0), (1, 0, 32, 1), (2, 1, 16, 1), (1, 1, 0, 0)])
@pytest.mark.parametrize("R,C", [(96, 800), (160, 288), (32, 32)])
def test_quantizer_writes_stay_inside_outputs(fq, grid, scale, rot, rnd, R, C):
    x = synth.as_torch(synth.special_values(R, C, R + C)).cuda()
    cfg = fq.Config(grid=grid, scale=scale, rot=rot, round=rnd, sign_mask_row=0x3C3C if rot else 0,
                    sign_mask_col=0x5A5A if rot else 0, sr_seed=3, emit_e4m3=True)
    g = Guarded()
    row = g.operand(fq, R, C, cfg)
    col = g.operand(fq, C, R, cfg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fq.rht_quantize(x, cfg, row, col, status=st)
    g.check()
    ref_row, ref_col = fq.rht_quantize(x, cfg)
    torch.cuda.synchronize()
    assert torch.equal(row.codes, ref_row.codes) and torch.equal(col.codes, ref_col.codes)


@pytest.mark.parametrize("grid,scale", [(0, 0), (0, 1), (1, 0)])
def test_gemm_writes_stay_inside_outputs(fq, grid, scale):
    M, N, K = 384, 640, 512
    cfg = fq.Config(grid=grid, scale=scale, rot=16, sign_mask_row=0x1111, want_col=False, sf_layout=fq.SF_MMA,
                    emit_e4m3=(grid == fq.GRID_E1M2))
    A, _ = fq.rht_quantize(synth.as_torch(synth.normal(M, K, 1)).cuda(), cfg)
    B, _ = fq.rht_quantize(synth.as_torch(synth.normal(N, K, 2, 0.05)).cuda(), cfg)
    g = Guarded()
    Dh = g.tensor((M, N), torch.bfloat16)
    Df = g.tensor((M, N), torch.float32)
    fq.gemm(A, B, grid, scale, D_bf16=Dh, D_f32=Df)
    g.check()


@pytest.mark.parametrize("ogrid,rnd", list(itertools.product([0, 1], [0, 1])))
def test_fused_gemm_quantize_writes_stay_inside_outputs(fq, ogrid, rnd):
    M, N, K = 256, 384, 512
    cfg = fq.Config(grid=0, rot=16, sign_mask_row=0x2222, want_col=False, sf_layout=fq.SF_MMA)
    A, _ = fq.rht_quantize(synth.as_torch(synth.normal(M, K, 3)).cuda(), cfg)
    B, _ = fq.rht_quantize(synth.as_torch(synth.normal(N, K, 4, 0.05)).cuda(), cfg)
    ocfg = fq.Config(grid=ogrid, rot=16, round=rnd, sign_mask_row=0x0F0F, sr_seed=5, want_col=False,
                     sf_layout=fq.SF_MMA, emit_e4m3=(ogrid == 1))
    g = Guarded()
    out = g.operand(fq, M, N, ocfg)
    Dh = g.tensor((M, N), torch.bfloat16)
    fq.gemm_quantize(A, B, 0, fq.SCALE_MX, ocfg, want_bf16=True, D_bf16=Dh, out=out)
    g.check()
