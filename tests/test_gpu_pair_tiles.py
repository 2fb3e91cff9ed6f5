"""The CTA-pair GEMM tiles (tcgen05 cta_group::2) are not the default, so the
GEMM, grouped and linear parity tests are re-run here, in a fresh process with
MXQ_GEMM_CTA_GROUP=2, against the same oracle and tolerances."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_on_pair_tiles(mxq):
    cmd = [sys.executable, "-m", "pytest", "tests/test_gpu_gemm.py", "tests/test_gpu_grouped.py",
           "tests/test_gpu_linear.py", "tests/test_gpu_grouped_linear.py", "-m", "gpu", "-q", "-x", "-k", "not full_size", "-p", "no:cacheprovider"]
    env = dict(os.environ, MXQ_GEMM_CTA_GROUP="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
