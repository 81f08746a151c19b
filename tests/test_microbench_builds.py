"""The standalone tcgen05 MMA instruction-rate microbenchmark (the measurement
behind the verify pass's tile analysis) compiles for sm_103a; no GPU needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "decode_attention_kv_dattn_gb300")


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_mma_rate_microbench_compiles(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    src = os.path.join(PKG, "microbench", "tcgen05_mma_rate.cu")
    out = tmp_path / "tcgen05_mma_rate"
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "--expt-relaxed-constexpr", "-I", os.path.join(PKG, "csrc"), "-o", str(out), src],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-4000:]
    assert out.exists()
