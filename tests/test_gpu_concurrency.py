"""Concurrent callers: two host threads, each on its own CUDA stream, run the
quantizer and grouped GEMMs of different shapes at the same time (the
library's host-side caches: per-device occupancy, per-thread grouped-launch
schedules).  Every result equals the one a single serial run gives."""
import threading

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


def work(fq, shape, seed, stream):
    """Quantize X, W, dY of one layer shape and run Dgrad + Wgrad grouped; returns the outputs."""
    T, D = shape
    with torch.cuda.stream(stream):
        X = synth.as_torch(synth.normal(T, D, seed)).cuda()
        W = synth.as_torch(synth.normal(D, D, seed + 1, 0.05)).cuda()
        G = synth.as_torch(synth.student_t(T, D, seed + 2)).cuda()
        cx = fq.Config(rot=16, sign_mask_row=0x1234, sign_mask_col=0x4321, sf_layout=fq.SF_MMA)
        cw = fq.Config(rot=16, sign_mask_row=0x1234, sign_mask_col=0x5555, sf_layout=fq.SF_MMA)
        cg = fq.Config(rot=16, sign_mask_row=0x5555, sign_mask_col=0x4321, round=fq.SR, sr_seed=seed,
                       sf_layout=fq.SF_MMA)
        Xr, Xc = fq.rht_quantize(X, cx, stream=stream)
        Wr, Wc = fq.rht_quantize(W, cw, stream=stream)
        Gr, Gc = fq.rht_quantize(G, cg, stream=stream)
        outs = fq.gemm_group([(Gr, Wc), (Gc, Xc)], 0, fq.SCALE_MX, want_bf16=True, want_f32=False, stream=stream)
        Y, _ = fq.gemm(Xr, Wr, 0, fq.SCALE_MX, want_f32=False, stream=stream)
    return [Xr.codes, Wc.codes, Gc.codes, outs[0][0], outs[1][0], Y]


def test_two_threads_two_streams(fq):
    shapes = [((1024, 512), 100), ((512, 768), 200)]
    serial = []
    for shape, seed in shapes:
        serial.append(work(fq, shape, seed, torch.cuda.current_stream()))
    torch.cuda.synchronize()
    results, errors = [None, None], []

    def run(i):
        try:
            s = torch.cuda.Stream()
            for _ in range(4):
                r = work(fq, shapes[i][0], shapes[i][1], s)
            s.synchronize()
            results[i] = r
        except Exception as e:   # reported below, from the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i in range(2):
        for got, want in zip(results[i], serial[i]):
            assert torch.equal(got, want)
