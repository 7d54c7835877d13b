"""The single-CTA GEMM kernels (used where no CTA pair fits, and for GroupedLinear 2 when
H % 256 != 0) keep their own parity coverage: the grouped-MLP parity cases rerun in a child
process with MXFP8MOE_SINGLE_CTA=1, which makes the library choose them for both GEMMs."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_single_cta_kernels_parity():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    env = dict(os.environ, MXFP8MOE_SINGLE_CTA="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_gpu_grouped_mlp.py"), "-k", "tiny or ragged or single or empty or mixtral"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
