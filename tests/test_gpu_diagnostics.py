"""GPU parity of the diagnostics (fp4_microscaled_quantization_gb300.diagnostics)
against the same measurements composed from the oracle: the code histogram
bit-exact, the fp64 sums within 1e-9 relative (both sides sum in fp64, only the
order differs), the bucket ratio from the oracle's own formula; each layer of
the depth chain within 1e-3 relative Frobenius error of the oracle's fp64 GEMM
of the oracle-quantized operands of that layer's (device) input."""
import numpy as np
import pytest
import torch

from fp4_microscaled_quantization_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp4_microscaled_quantization_gb300 import diagnostics, fp4q
    fp4q.lib()
    return diagnostics


def oracle_report(orc, bits, grid, rot, mask):
    q = orc.quantize(bits, 0, grid, orc.SCALE_MX, rot, mask if rot else 0)
    deq = orc.dequantize(q["codes"], q["scales"], 0, grid, orc.SCALE_MX, True, rot, mask if rot else 0, bool(rot))
    st = orc.bias_stats(synth.bf16_bits_to_f32(bits).ravel(), deq.ravel(), q["codes"])
    st["bucket_ratio"] = orc.effective_bucket_ratio(st["hist"], grid)
    st["mean_rel_error"] = orc.rel_error(synth.bf16_bits_to_f32(bits).ravel(), deq.ravel())["mean"]
    st["grid_error"] = orc.grid_error(bits, grid, orc.SCALE_MX, rot, mask if rot else 0, q["codes"], q["scales"])
    return st


@pytest.mark.parametrize("grid", [0, 1, 2])
@pytest.mark.parametrize("rot", [0, 16, 32])
def test_quantizer_report_matches_oracle(dg, orc, grid, rot):
    bits = synth.normal_channel_outliers(96, 640, 41, 8, 40.0)
    mask = orc.sign_mask_from_seed(5, rot) if rot else 0
    got = dg.quantizer_report(synth.as_torch(bits).cuda(), grid, rot, mask)
    want = oracle_report(orc, bits, grid, rot, mask)
    assert np.array_equal(np.asarray(got["hist"], dtype=np.uint64), want["hist"])
    assert np.allclose(got["sums"], want["sums"], rtol=1e-9, atol=0)
    assert got["bucket_ratio"] == pytest.approx(want["bucket_ratio"], rel=1e-12)
    assert got["sqnr_db"] == pytest.approx(want["sqnr_db"], rel=1e-9)
    assert got["mean_rel_error"] == pytest.approx(want["mean_rel_error"], rel=1e-9)
    assert np.array_equal(got["grid_error"]["counts"], want["grid_error"]["counts"])
    assert got["grid_error"]["mean"] == pytest.approx(want["grid_error"]["mean"], abs=1e-6)


def test_delta_sqnr_sweep(dg, orc):
    rows = dg.delta_sqnr_sweep(128, 1024, [1.0, 10.0, 100.0])
    assert len(rows) == 9
    for r in rows:
        print(r["strength"], r["grid"], round(r["sqnr_plain_db"], 2), round(r["sqnr_rht_db"], 2),
              round(r["delta_sqnr_db"], 2), round(r["bucket_ratio_plain"], 3), round(r["bucket_ratio_rht"], 3))
        assert np.isfinite(r["delta_sqnr_db"])
        assert 0 < r["bucket_ratio_plain"] <= 1 and 0 < r["bucket_ratio_rht"] <= 1
    # one row recomputed from the oracle end to end
    seed, n_h = 2024, 16
    mask = orc.sign_mask_from_seed(seed, n_h)
    bits = synth.normal_channel_outliers(128, 1024, seed + 2, 8, 100.0)
    plain = oracle_report(orc, bits, 1, 0, 0)
    rht = oracle_report(orc, bits, 1, n_h, mask)
    row = [r for r in rows if r["strength"] == 100.0 and r["grid"] == "e1m2"][0]
    assert row["delta_sqnr_db"] == pytest.approx(rht["sqnr_db"] - plain["sqnr_db"], rel=1e-9, abs=1e-9)
    assert row["bucket_ratio_rht"] == pytest.approx(rht["bucket_ratio"], rel=1e-12)


@pytest.mark.parametrize("grid", [0, 1, 2])
def test_depth_chain_layers_match_oracle(dg, orc, grid):
    M, d, depth = 256, 512, 3
    x = synth.normal(M, d, 61)
    ws = dg.chain_weights(d, depth, 70)
    res = dg.depth_chain(x, ws, grid, rot=16, keep=True)
    for k, layer in enumerate(res["kept"]):
        hb = layer["input_bf16"].view(torch.int16).cpu().numpy().view(np.uint16)
        mask = layer["mask"]
        qa = orc.quantize(hb, 0, grid, orc.SCALE_MX, 16, mask)
        qb = orc.quantize(ws[k], 0, grid, orc.SCALE_MX, 16, mask)
        da = orc.dequantize(qa["codes"], qa["scales"], 0, grid, orc.SCALE_MX)
        db = orc.dequantize(qb["codes"], qb["scales"], 0, grid, orc.SCALE_MX)
        want = orc.gemm_ref(da, db)
        got = layer["out_f32"].double().cpu().numpy()
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert rel <= 1e-3, f"layer {k}: {rel:.3e}"
        # this layer's attenuation against the exact product of its own input
        exact = synth.bf16_bits_to_f32(hb).astype(np.float64) @ synth.bf16_bits_to_f32(ws[k]).astype(np.float64).T
        a_orc = orc.bias_stats(exact.astype(np.float32).ravel(), got.astype(np.float32).ravel())["alpha"]
        assert res["layers"][k]["alpha"] == pytest.approx(a_orc, abs=1e-5)
    a = [l["alpha"] for l in res["layers"]]
    assert res["prod_alpha"] == pytest.approx(float(np.prod(a)), rel=1e-12)
    print(res["grid"], [round(v, 5) for v in a], round(res["prod_alpha"], 5), round(res["exp_minus_sum_delta"], 5),
          round(res["end_to_end_alpha"], 5))
    assert 0.5 < res["end_to_end_alpha"] < 1.5
