"""The group-scale arithmetic of the quantiser (csrc/quant.cuh) against the
IEEE operations it stands for, exhaustively on the GPU: the scale
fp16_rn(amax / Q) for every non-negative finite fp32 amax (Q = 7 and 127) and
the reciprocal fl(1/s) for every positive finite fp16 scale s.  The check is
compiled from tests/scale_math_check.cu against the library's own header."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_scale_and_reciprocal_equal_ieee_everywhere(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "scale_math_check")
    csrc = os.path.join(ROOT, "serving_tcgen05_streamed_gb300", "csrc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", f"-I{csrc}",
                    f"-I{os.path.join(ROOT, 'include')}", "-o", exe, os.path.join(ROOT, "tests", "scale_math_check.cu")],
                   check=True, timeout=300)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0; Q=127 mismatches 0; scale_reciprocal mismatches 0" in r.stdout
