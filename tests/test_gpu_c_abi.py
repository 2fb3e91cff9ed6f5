"""The C ABI from a plain C program (tests/c_abi/mxq_c_smoke.c): no Python,
no torch in that process. It quantizes two operands with mxq_quantize,
multiplies them with mxq_gemm and compares with the exact integer product
(operands in {-1, 0, 1}, so every step is exact)."""
import os
import shutil
import subprocess

import pytest

import mx_block_scaled_mxq_gb300 as m

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_c_program_quantizes_and_multiplies(tmp_path, mxq):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(m.library_path())
    exe = str(tmp_path / "mxq_c_smoke")
    build = [cc, "-O2", "-std=c11", "-Wall", "-Werror", f"-I{CUDA}/include", f"-I{ROOT}/include",
             os.path.join(ROOT, "tests", "c_abi", "mxq_c_smoke.c"), f"-L{lib_dir}", "-lmxq", f"-L{CUDA}/lib64",
             "-lcudart", f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{CUDA}/lib64", "-o", exe]
    r = subprocess.run(build, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout[-2000:] + r.stderr[-2000:]
