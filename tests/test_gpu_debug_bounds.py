"""The parity suites again, on the debug build of the library.

compute-sanitizer is not available on this GPU pool, so the library has its
own bounds checking: built with MXQ_DEBUG (libmxq_debug.so), every kernel
checks the address of each plain global load and store it computes against
the extent of the buffer it belongs to, skips an access outside it and sets
bit 3 of the device error word.  Every test below ends with
mxq_poll_device_error() == 0, so running them on the debug build shows that
no kernel computed an address outside its buffers on any of their shapes --
ragged tails, empty and many groups, strided views, unaligned fallbacks --
and that the checks do not change a single result.  The full-size cases are
left out (they take minutes on the slower debug build)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_quant.py", "tests/test_gpu_gemm.py", "tests/test_gpu_grouped.py", "tests/test_gpu_ste.py",
          "tests/test_gpu_qat.py", "tests/test_gpu_linear.py", "tests/test_gpu_weight_reuse.py",
          "tests/test_gpu_group_offsets.py", "tests/test_gpu_grouped_linear.py"]


def test_parity_suites_pass_on_the_bounds_checking_build(mxq):
    env = dict(os.environ, MXQ_LIBRARY="debug")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", "not full_size", "-p", "no:cacheprovider",
           *SUITES]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = "\n".join((res.stdout + res.stderr).splitlines()[-25:])
    assert res.returncode == 0, tail
    assert " passed" in res.stdout, tail
