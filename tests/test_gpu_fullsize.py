"""Parity at the full workload sizes, in the launch configuration the benchmark
times (32 x 256 quantizer tiles, 128 x 256 GEMM tiles):

  tiny    X 256x512, row-wise, H16 + seeded signs, MX E2M1 and E1M2, RTNE, with
          SQNR / shrinkage of the reconstruction
  act     X 8192x4096, both copies, deterministic H16, MX E2M1 and E1M2, RTNE
  grad    dY 8192x14336, both copies, random H16, MX E1M2, Philox SR
  weight  W 14336x4096, both copies, H32, NVFP4-style E2M1 and E1M2, RTNE,
          two-pass (amax pre-pass) and one-pass (caller's amax)
  layer   X 16384x4096, W 4096^2, dY 16384x4096: all six copies bit-exact, and
          the Fprop / Dgrad / Wgrad GEMMs (Dgrad and Wgrad in one grouped launch)
          on 4096 sampled outputs per GEMM, for each of the three MMA kinds

Every quantized copy is compared in full, bit for bit.  The oracle runs in
threads (its C calls release the GIL)."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

from fp4_microscaled_quantization_gb300 import synth

pytestmark = pytest.mark.gpu

POOL = cf.ThreadPoolExecutor(max_workers=8)


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


def quantize_both(fq, orc, bits, cfg, given=None):
    """GPU copies and oracle futures for the requested orientations."""
    x = synth.as_torch(bits).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ro, co = fq.rht_quantize(x, cfg, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    futs = {}
    for orient, want in ((0, cfg.want_row), (1, cfg.want_col)):
        if want:
            mask = cfg.sign_mask_row if orient == 0 else cfg.sign_mask_col
            g = None if given is None else given[orient]
            futs[orient] = POOL.submit(orc.quantize, bits, orient, cfg.grid, cfg.scale, cfg.rot, mask, cfg.round,
                                       cfg.sr_seed, g, cfg.emit_e4m3)
    return {0: ro, 1: co}, futs


def assert_same(cfg, op, ref):
    codes = op.codes.cpu().numpy()
    n_bad = int(np.count_nonzero(codes != ref["codes"]))
    assert n_bad == 0, f"{n_bad} code bytes differ"
    sc = op.scales.cpu().numpy()
    if cfg.sf_layout == 1:
        sc = mma_to_plain(sc, *ref["scales"].shape)
    assert np.array_equal(sc, ref["scales"])
    if cfg.scale == 1:
        assert op.tensor_scale.cpu().numpy()[0].view(np.uint32) == np.float32(ref["tensor_scale"]).view(np.uint32)
    if cfg.emit_e4m3:
        assert np.array_equal(op.e4m3.cpu().numpy(), ref["e4m3"])


def test_tiny_rowwise_with_stats(fq, orc):
    x = synth.tiny_x()
    mask = orc.sign_mask_from_seed(1001, 16)
    for grid in (0, 1):
        cfg = fq.Config(grid=grid, rot=16, sign_mask_row=mask, want_col=False)
        ops, futs = quantize_both(fq, orc, x, cfg)
        ref = futs[0].result()
        assert_same(cfg, ops[0], ref)
        # reconstruction statistics in the original domain, GPU vs oracle
        deq = fq.dequantize(ops[0], cfg, orient=0, unrotate=True)
        xf = torch.from_numpy(synth.bf16_bits_to_f32(x)).cuda()
        got = fq.bias_stats(xf, deq, ops[0].codes)
        want_deq = orc.dequantize(ref["codes"], ref["scales"], 0, grid, 0, True, 16, mask, True)
        want = orc.bias_stats(synth.bf16_bits_to_f32(x), want_deq, ref["codes"])
        for k in ("sqnr_db", "alpha", "shrinkage"):
            assert abs(got[k] - want[k]) <= 1e-4 * max(1.0, abs(want[k])), k
        assert np.array_equal(got["hist"], want["hist"])
        print(f"tiny grid={grid}: SQNR {got['sqnr_db']:.3f} dB alpha {got['alpha']:.6f} "
              f"shrinkage {got['shrinkage']:.6f}")


@pytest.mark.parametrize("grid", [0, 1])
def test_act_both_copies(fq, orc, grid):
    x = synth.act_x()
    cfg = fq.Config(grid=grid, rot=16)
    ops, futs = quantize_both(fq, orc, x, cfg)
    for o in (0, 1):
        assert_same(cfg, ops[o], futs[o].result())


def test_grad_sr_both_copies(fq, orc):
    x = synth.grad_dy()
    mr, mc = orc.sign_mask_from_seed(1003, 16), orc.sign_mask_from_seed(1013, 16)
    cfg = fq.Config(grid=1, rot=16, round=fq.SR, sign_mask_row=mr, sign_mask_col=mc, sr_seed=1004)
    ops, futs = quantize_both(fq, orc, x, cfg)
    for o in (0, 1):
        assert_same(cfg, ops[o], futs[o].result())


@pytest.mark.parametrize("grid", [0, 1])
def test_weight_nv_two_and_one_pass(fq, orc, grid):
    w = synth.weight_w()
    cfg = fq.Config(grid=grid, scale=fq.SCALE_NV, rot=32)
    ops, futs = quantize_both(fq, orc, w, cfg)
    refs = {o: futs[o].result() for o in (0, 1)}
    for o in (0, 1):
        assert_same(cfg, ops[o], refs[o])
    # one pass with the caller's amax: identical copies
    G = fq.rotated_amax(synth.as_torch(w).cuda(), cfg)
    cfg1 = fq.Config(grid=grid, scale=fq.SCALE_NV, rot=32, global_amax=G)
    r1, c1 = fq.rht_quantize(synth.as_torch(w).cuda(), cfg1)
    torch.cuda.synchronize()
    assert_same(cfg1, r1, refs[0])
    assert_same(cfg1, c1, refs[1])


@pytest.mark.parametrize("kind", ["mxf4", "nvf4", "mxf8f6f4"])
def test_layer_operands_and_gemms(fq, orc, kind):
    """All six copies of the layer's operands bit-exact, then Fprop (fp4q_gemm)
    and Dgrad + Wgrad in one grouped launch (fp4q_gemm_group, as the benchmark
    runs them) on 4096 sampled outputs each against the oracle's fp64 GEMM of
    the oracle's own copies, for each MMA kind: E2M1 with MX scales
    (kind::mxf4), E2M1 with NVFP4-style scales (kind::mxf4nvf4, alpha =
    S_t(A) S_t(B)) and E1M2 through its E4M3 bytes (kind::mxf8f6f4)."""
    X, W, dY = synth.layer()
    grid = 1 if kind == "mxf8f6f4" else 0
    scale = fq.SCALE_NV if kind == "nvf4" else fq.SCALE_MX
    e4 = grid == 1
    mK, mN, mM = (orc.sign_mask_from_seed(1005 + i, 16) for i in range(3))
    cfg_x = fq.Config(grid=grid, scale=scale, rot=16, sign_mask_row=mK, sign_mask_col=mM, sf_layout=fq.SF_MMA,
                      emit_e4m3=e4)
    cfg_w = fq.Config(grid=grid, scale=scale, rot=16, sign_mask_row=mK, sign_mask_col=mN, sf_layout=fq.SF_MMA,
                      emit_e4m3=e4)
    cfg_g = fq.Config(grid=grid, scale=scale, rot=16, sign_mask_row=mN, sign_mask_col=mM, round=fq.SR, sr_seed=1008,
                      sf_layout=fq.SF_MMA, emit_e4m3=e4)
    ox, fx = quantize_both(fq, orc, X, cfg_x)
    ow, fw = quantize_both(fq, orc, W, cfg_w)
    og, fg = quantize_both(fq, orc, dY, cfg_g)
    refs = {}
    for name, cfg, ops, futs in (("x", cfg_x, ox, fx), ("w", cfg_w, ow, fw), ("g", cfg_g, og, fg)):
        for o in (0, 1):
            refs[(name, o)] = futs[o].result()
            assert_same(cfg, ops[o], refs[(name, o)])
    deq = {k: orc.dequantize(v["codes"], v["scales"], v["tensor_scale"], grid, scale, with_tensor_scale=False)
           for k, v in refs.items()}
    ts = {k: v["tensor_scale"] for k, v in refs.items()}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, Yf = fq.gemm(ox[0], ow[0], grid, scale, want_bf16=False, status=st)
    (_, dXf), (_, dWf) = fq.gemm_group([(og[0], ow[1]), (og[1], ox[1])], grid, scale, want_bf16=False,
                                       want_f32=True, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rng = np.random.default_rng(0)
    cases = {"fprop": (Yf, ("x", 0), ("w", 0)), "dgrad": (dXf, ("g", 0), ("w", 1)),
             "wgrad": (dWf, ("g", 1), ("x", 1))}
    for name, (Df, ka, kb) in cases.items():
        ii = rng.integers(0, Df.shape[0], 4096)
        jj = rng.integers(0, Df.shape[1], 4096)
        alpha = float(np.float64(ts[ka]) * np.float64(ts[kb])) if scale == fq.SCALE_NV else 1.0
        want = orc.gemm_entries(deq[ka], deq[kb], ii, jj, alpha)
        got = Df[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].double().cpu().numpy()
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert rel <= 1e-3, f"{kind} {name}: sampled relative Frobenius error {rel:.3e}"
        print(f"{kind} {name}: sampled rel err {rel:.2e}")
