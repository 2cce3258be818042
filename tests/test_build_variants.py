"""The GEMM's build options that are off by default still compile for sm_103a:
the cta_group::2 pair form (-DFP4Q_GEMM_CLUSTER=1) and sixteen epilogue warps
(-DFP4Q_GEMM_EPI_WARPS=16).  Compile only (no GPU); the two run in parallel."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GEMM = os.path.join(ROOT, "fp4_microscaled_quantization_gb300", "csrc", "gemm.cu")
VARIANTS = {"pair": "-DFP4Q_GEMM_CLUSTER=1", "epi16": "-DFP4Q_GEMM_EPI_WARPS=16"}


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return path if os.path.exists(path) else None


def test_gemm_build_options_compile():
    exe = nvcc()
    if exe is None:
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as tmp:
        procs = {}
        for name, flag in VARIANTS.items():
            cmd = [exe, flag, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                   "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-c", GEMM, "-o", os.path.join(tmp, name + ".o")]
            procs[name] = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        failed = {}
        for name, p in procs.items():
            out, _ = p.communicate(timeout=600)
            if p.returncode != 0:
                failed[name] = out[-2000:]
        assert not failed, failed
