"""The quantizer's bounded pipeline waits, exercised without any fault: CTA 0
is made to wait for one of its tiles on a barrier that nothing arrives at
(fp4q_test_quantize_wait_expiry), with a 20 ms limit.  The call must come back
with FP4Q_DEV_TIMEOUT in the status word (CTA 0 stopped, drained its own tile
loads and returned), every tile of the other CTAs must be quantized as usual,
and the next ordinary call must again be bit-exact against the oracle: the
context stays usable."""
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


@pytest.mark.parametrize("stall_tile", [0, 1])
def test_wait_expiry_raises_timeout_and_context_survives(fq, orc, stall_tile):
    R, C = 4096, 4096                         # 2048 tiles of 32 x 256: several per CTA
    bits = synth.normal(R, C, 4711 + stall_tile)
    x = synth.as_torch(bits).cuda()
    cfg = fq.Config(rot=16, sign_mask_row=0x1357, want_col=False)
    ref = orc.quantize(bits, 0, 0, 0, 16, 0x1357)
    ro = fq.alloc_operand(R, C, cfg, "cuda")
    ro.codes.fill_(0xAA)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fq.test_quantize_wait_expiry(x, cfg, ro, None, st, stall_tile, 20000)
    torch.cuda.synchronize()
    assert st.item() & fq.DEV_TIMEOUT, f"status {st.item():#x}"
    # CTA 0 walks tiles 0, G, 2G, ... (G = three persistent CTAs per SM for
    # RTNE, at most one per tile); from the stalled one on its tiles keep the
    # fill, every other tile is quantized
    codes = ro.codes.cpu().numpy()
    tiles_per_row = C // 256
    n_tiles = R // 32 * tiles_per_row
    G = min(n_tiles, 3 * torch.cuda.get_device_properties(0).multi_processor_count)
    unwritten = set()
    for t in range(n_tiles):
        r0, c0 = (t // tiles_per_row) * 32, (t % tiles_per_row) * 128
        if not np.array_equal(codes[r0:r0 + 32, c0:c0 + 128], ref["codes"][r0:r0 + 32, c0:c0 + 128]):
            unwritten.add(t)
    assert unwritten == set(range(G * stall_tile, n_tiles, G)), sorted(unwritten)[:10]
    # the context is still usable: an ordinary call is bit-exact again
    st.zero_()
    ro2, _ = fq.rht_quantize(x, cfg, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(ro2.codes.cpu().numpy(), ref["codes"])
    assert np.array_equal(ro2.scales.cpu().numpy(), ref["scales"])


def test_wait_expiry_rejects_bad_arguments(fq):
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    cfg = fq.Config(want_col=False)
    ro = fq.alloc_operand(128, 256, cfg, "cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for tile, us in ((-1, 1000), (0, 0), (0, 3000000)):
        with pytest.raises(fq.Fp4qError) as e:
            fq.test_quantize_wait_expiry(x, cfg, ro, None, st, tile, us)
        assert e.value.status == fq.ERR_INVALID_ARG
