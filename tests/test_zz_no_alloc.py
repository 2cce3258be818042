"""The allocation-free statistics entry point, for callers that cannot
allocate device memory (frameworks that own every device byte through their
own pool, plugins inside a fixed memory budget, paths that must not pay for
cudaMalloc's implicit synchronisation).  It is called here through the C ABI
directly and must reproduce the workspace-taking fp4q_bias_stats, call after
call, although both share the library's one built-in scratch array.

Kept in a file that sorts last so that a run stopping at its first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp4_microscaled_quantization_gb300 import fp4q
    fp4q.lib()
    return fp4q


def _noalloc(fq, ref, approx, codes):
    out = torch.full((22,), float("nan"), dtype=torch.float64, device=ref.device)
    s = fq.lib().fp4q_bias_stats_noalloc(ref.data_ptr(), approx.data_ptr(), ref.numel(),
                                         None if codes is None else codes.data_ptr(), out.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert s == fq.OK, fq.status_str(s)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("n", [1000, 1 << 21])
def test_noalloc_matches_workspace_entry_point(fq, n):
    rng = np.random.default_rng(n)
    ref = torch.from_numpy(rng.standard_normal(n).astype(np.float32)).cuda()
    approx = torch.from_numpy((rng.standard_normal(n) * 0.1).astype(np.float32)).cuda() + ref * 0.95
    codes = torch.from_numpy(rng.integers(0, 256, n // 2, dtype=np.uint8)).cuda()
    want = fq.bias_stats(ref, approx, codes, sync=False).cpu()
    for _ in range(2):   # two calls in a row share (and must clear) the built-in scratch
        got = _noalloc(fq, ref, approx, codes)
        assert np.allclose(got[:5].numpy(), want[:5].numpy(), rtol=1e-9, atol=0)
        assert np.array_equal(got.view(torch.int64)[5:].numpy(), want.view(torch.int64)[5:].numpy())
