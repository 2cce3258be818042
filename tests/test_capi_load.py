"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports
every function include/fp4q.h declares, and its host-only logic (status text,
sign masks, workspace sizes, statistics finalisation, argument validation)
behaves as documented.  No compute call is made here."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fq():
    from fp4_microscaled_quantization_gb300 import build, fp4q
    if not os.path.exists(fp4q.LIB_PATH):
        build.build()
    return fp4q


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fp4q.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4q_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(fq):
    names = declared_functions()
    assert len(names) >= 12
    L = ctypes.CDLL(fq.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(fq):
    assert fq.status_str(0) == "ok"
    assert "workspace" in fq.status_str(fq.ERR_WORKSPACE)
    assert fq.lib().fp4q_version() % 10000 == 1031


def test_sign_mask_matches_oracle(fq, orc):
    for seed in (0, 1, 7, 2 ** 40 + 3, 2 ** 64 - 1):
        for n in (16, 32):
            assert fq.sign_mask_from_seed(seed, n) == orc.sign_mask_from_seed(seed, n)


def test_workspace_sizes(fq):
    assert fq.workspace_bytes(128, 128, fq.Config(scale=fq.SCALE_MX)) == 0
    assert fq.workspace_bytes(128, 128, fq.Config(scale=fq.SCALE_NV)) >= 8
    assert fq.bias_stats_workspace_bytes(1000) > 0


def test_stats_finalize_hand_example(fq):
    import numpy as np
    s = np.array([5.0, 1.0, 3.0, 3.0, -1.0])     # ref [1,2], approx [1,1]
    a, b, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    fq.lib().fp4q_stats_finalize(s.ctypes.data_as(ctypes.c_void_p), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    assert abs(a.value - 10 * math.log10(5)) < 1e-12 and b.value == 0.6 and abs(c.value + 1 / 3) < 1e-15


def _quant(fq, x_ptr, rows, cols, ld, cfg, ro=None, co=None):
    cc = cfg.c()
    return fq.lib().fp4q_rht_quantize(x_ptr, rows, cols, ld, ctypes.byref(cc),
                                      ctypes.byref(ro) if ro else None, ctypes.byref(co) if co else None,
                                      None, 0, None, None)


def test_validation_rejects_before_launch(fq):
    L = fq.lib()
    fake = 1 << 20   # never dereferenced: every call below fails validation first
    op = fq.COperand(fake, fake, fake, fake)
    cfg = fq.Config()
    assert L.fp4q_rht_quantize(fake, 64, 64, 64, None, None, None, None, 0, None, None) == fq.ERR_INVALID_ARG
    assert _quant(fq, fake, 64, 48, 64, cfg, op, op) == fq.ERR_INVALID_ARG            # cols % 32
    assert _quant(fq, fake, 48, 64, 64, cfg, op, op) == fq.ERR_INVALID_ARG            # rows % 32 with col copy
    assert _quant(fq, fake, 64, 64, 60, cfg, op, op) == fq.ERR_INVALID_ARG            # ld < cols
    assert _quant(fq, fake, 64, 64, 68, cfg, op, op) == fq.ERR_ALIGNMENT              # ld % 8
    assert _quant(fq, fake + 2, 64, 64, 64, cfg, op, op) == fq.ERR_ALIGNMENT          # x alignment
    assert _quant(fq, fake, 64, 64, 64, fq.Config(grid=7), op, op) == fq.ERR_INVALID_ARG
    assert _quant(fq, fake, 64, 64, 64, fq.Config(rot=8), op, op) == fq.ERR_INVALID_ARG
    assert _quant(fq, fake, 64, 64, 64, fq.Config(want_row=False, want_col=False)) == fq.ERR_INVALID_ARG
    assert _quant(fq, fake, 64, 64, 64, cfg, None, op) == fq.ERR_INVALID_ARG          # missing row copy
    assert _quant(fq, fake, 64, 64, 64, fq.Config(sf_layout=fq.SF_MMA), op, op) == fq.ERR_INVALID_ARG  # rows % 128
    assert _quant(fq, fake, 65535 * 64 + 32, 64, 64, cfg, op, op) == fq.ERR_INVALID_ARG  # (rows + 63) / 64 > 65535
    assert _quant(fq, fake, 128, 128, 128, fq.Config(scale=fq.SCALE_NV), op, op) == fq.ERR_WORKSPACE
    nots = fq.COperand(fake, fake, None, None)
    assert _quant(fq, fake, 128, 128, 128, fq.Config(scale=fq.SCALE_NV), nots, nots) == fq.ERR_INVALID_ARG
    assert _quant(fq, fake, 0, 64, 64, cfg, op, op) == fq.OK                          # empty: nothing to do
    assert _quant(fq, None, 64, 0, 64, cfg, op, op) == fq.OK
    assert L.fp4q_bias_stats(fake, fake, 100, None, None, 0, fake, None) == fq.ERR_WORKSPACE
    assert L.fp4q_bias_stats(fake, fake, 101, fake, fake, 1 << 30, fake, None) == fq.ERR_INVALID_ARG
    assert L.fp4q_hadamard_rotate_bf16(fake, 64, 64, 64, 0, 0, 0, fake, None, None) == fq.ERR_INVALID_ARG
    # GEMM shape limits: M / 128 <= 65535, N and K <= INT32_MAX
    for M, N, K in ((65536 * 128, 128, 128), (128, 1 << 31, 128), (128, 128, 1 << 31)):
        assert L.fp4q_gemm(ctypes.byref(op), ctypes.byref(op), M, N, K, 0, 0, fake, None, None,
                           None) == fq.ERR_INVALID_ARG
