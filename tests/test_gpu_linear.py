"""The linear-layer recipe driver (fp4_microscaled_quantization_gb300.linear):
every GEMM of both recipes against the oracle composed the same way (same
grid, rotation per copy, masks along each contraction axis, SR on dY), fp32
output within 1e-3 relative Frobenius error; and a report of the output SQNR
and attenuation of each recipe against the unquantized GEMMs."""
import numpy as np
import pytest
import torch

from fp4_microscaled_quantization_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lin():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp4_microscaled_quantization_gb300 import fp4q, linear
    fp4q.lib()
    return linear


def oracle_copy(orc, bits, orient, grid, rotate, mask, sr, seed):
    q = orc.quantize(bits, orient, grid, 0, 16 if rotate else 0, mask if rotate else 0, orc.SR if sr else orc.RTNE,
                     seed)
    return orc.dequantize(q["codes"], q["scales"], 0, grid, 0)


@pytest.mark.parametrize("recipe", ["ufp4", "e2m1"])
def test_recipe_gemms_match_oracle(lin, orc, recipe):
    M, K, N = 256, 384, 256
    X = synth.normal_channel_outliers(M, K, 11, 4, 30.0)
    W = synth.normal(N, K, 12, 0.02)
    dY = synth.student_t(M, N, 13)
    layer = lin.Fp4Linear(recipe, seed=77, out_f32=True)
    res = layer(synth.as_torch(X).cuda(), synth.as_torch(W).cuda(), synth.as_torch(dY).cuda())
    torch.cuda.synchronize()
    grid = 1 if recipe == "ufp4" else 0
    every = recipe == "ufp4"
    s = layer.sr_seed
    Xr = oracle_copy(orc, X, 0, grid, every, layer.mask_K, False, s)
    Xc = oracle_copy(orc, X, 1, grid, True, layer.mask_M, False, s)
    Wr = oracle_copy(orc, W, 0, grid, every, layer.mask_K, False, s)
    Wc = oracle_copy(orc, W, 1, grid, every, layer.mask_N, False, s)
    Gr = oracle_copy(orc, dY, 0, grid, every, layer.mask_N, True, s)
    Gc = oracle_copy(orc, dY, 1, grid, True, layer.mask_M, True, s)
    for name, got, (A, B) in (("fprop", res.Y, (Xr, Wr)), ("dgrad", res.dX, (Gr, Wc)), ("wgrad", res.dW, (Gc, Xc))):
        want = orc.gemm_ref(A, B)
        g = got.double().cpu().numpy()
        rel = np.linalg.norm(g - want) / np.linalg.norm(want)
        assert rel <= 1e-3, f"{recipe} {name}: {rel:.3e}"
    ref = lin.reference_gemms(synth.as_torch(X).cuda(), synth.as_torch(W).cuda(), synth.as_torch(dY).cuda())
    q = lin.output_quality(res, ref)
    print(recipe, {k: (round(v["sqnr_db"], 2), round(v["alpha"], 5)) for k, v in q.items()})
    assert all(v["sqnr_db"] > 5.0 for v in q.values())
