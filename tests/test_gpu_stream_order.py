"""Stream order across back-to-back launches.

The quantizer and GEMM kernels launch as programmatic dependents of the
stream's previous kernel and wait for it before touching global memory.  The
chain below overwrites buffers the previous launch wrote and reads what the
previous launch produced, with no synchronisation in between, and compares
every stage with the oracle."""
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


def test_overwrite_gemm_requantize_chain(fq, orc):
    M, N, K = 256, 384, 512
    mask = 0x1357
    a1 = synth.normal(M, K, 11)
    a2 = synth.normal_point_outliers(M, K, 12)
    b = synth.normal(N, K, 13, 0.05)
    cfg = fq.Config(grid=0, rot=16, sign_mask_row=mask, want_col=False, sf_layout=fq.SF_MMA)
    ycfg = fq.Config(grid=1, rot=16, sign_mask_row=0x0F0F, want_col=False, round=fq.SR, sr_seed=31)
    x1, x2, xb = (synth.as_torch(v).cuda() for v in (a1, a2, b))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()

    B, _ = fq.rht_quantize(xb, cfg, status=st)
    A, _ = fq.rht_quantize(x1, cfg, status=st)
    fq.rht_quantize(x2, cfg, A, status=st)              # write after write: A now holds a2's copy
    Dh, Df = fq.gemm(A, B, 0, fq.SCALE_MX, status=st)   # read after write
    Yq, _ = fq.rht_quantize(Dh, ycfg, status=st)        # reads the GEMM's output at once
    torch.cuda.synchronize()
    assert st.item() == 0

    qa = orc.quantize(a2, 0, 0, 0, 16, mask)
    assert np.array_equal(A.codes.cpu().numpy(), qa["codes"])
    assert np.array_equal(mma_to_plain(A.scales.cpu().numpy(), M, K // 32), qa["scales"])

    qb = orc.quantize(b, 0, 0, 0, 16, mask)
    da = orc.dequantize(qa["codes"], qa["scales"], 0.0, 0, 0)
    db = orc.dequantize(qb["codes"], qb["scales"], 0.0, 0, 0)
    want = orc.gemm_ref(da, db)
    got = Df.double().cpu().numpy()
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 1e-3

    d_bits = Dh.view(torch.int16).cpu().numpy().view(np.uint16)
    qy = orc.quantize(d_bits, 0, 1, 0, 16, 0x0F0F, 1, 31)
    assert np.array_equal(Yq.codes.cpu().numpy(), qy["codes"])
    assert np.array_equal(Yq.scales.cpu().numpy(), qy["scales"])


def test_cuda_graph_capture_and_replay(fq):
    """The quantizer and GEMM launches (programmatic dependents, no host
    synchronisation or allocation inside a call) can be captured in a CUDA
    graph; a replay on new inputs gives the bits an eager run gives."""
    M, N, K = 256, 384, 512
    cfg = fq.Config(grid=0, rot=16, sign_mask_row=0x2468, want_col=False, sf_layout=fq.SF_MMA)
    X = synth.as_torch(synth.normal(M, K, 21)).cuda()
    W = synth.as_torch(synth.normal(N, K, 22, 0.05)).cuda()
    Xr, _ = fq.rht_quantize(X, cfg)
    Wr, _ = fq.rht_quantize(W, cfg)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up outside the capture
        fq.rht_quantize(X, cfg, Xr, status=st)
        fq.gemm(Xr, Wr, 0, fq.SCALE_MX, want_f32=False, D_bf16=D, status=st)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fq.rht_quantize(X, cfg, Xr, status=st)
        fq.rht_quantize(W, cfg, Wr, status=st)
        fq.gemm(Xr, Wr, 0, fq.SCALE_MX, want_f32=False, D_bf16=D, status=st)
    X.copy_(synth.as_torch(synth.normal_point_outliers(M, K, 23)).cuda())
    W.copy_(synth.as_torch(synth.normal(N, K, 24, 0.05)).cuda())
    graph.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    got = (Xr.codes.clone(), Wr.codes.clone(), D.clone())
    Xe, _ = fq.rht_quantize(X, cfg)
    We, _ = fq.rht_quantize(W, cfg)
    De, _ = fq.gemm(Xe, We, 0, fq.SCALE_MX, want_f32=False)
    torch.cuda.synchronize()
    assert torch.equal(got[0], Xe.codes) and torch.equal(got[1], We.codes)
    assert torch.equal(got[2], De)
