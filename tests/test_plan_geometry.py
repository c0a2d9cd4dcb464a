"""Host-side check of the tensor-core plans (no GPU): compiles
tests/plan_check.cu against the kernel source with nvcc and runs it.  It
replays the producers' stores and the MMA operand addresses of every plan
shape the kernels use and compares each against the input pixel the
convolution definition reads."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _nvcc():
    return os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"


@pytest.mark.skipif(not os.path.exists(_nvcc()), reason="nvcc not available")
def test_plan_geometry_host_replay():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "plan_check")
        # PTX only: the device code is not run here, only the host planner is
        cmd = [_nvcc(), "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=compute_103a",
               "-I", os.path.join(ROOT, "include"), "-x", "cu",
               os.path.join(HERE, "plan_check.cu"), "-o", exe]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
        out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert "CHECK OK" in out.stdout, out.stdout[-3000:]
        assert out.returncode == 0
