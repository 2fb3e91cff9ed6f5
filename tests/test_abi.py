"""The C ABI library: builds, loads without a GPU, exports every symbol its
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import mx_block_scaled_mxq_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mxq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mxq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return m.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 15
    raw = ctypes.CDLL(m.library_path())
    for n in names:
        assert hasattr(raw, n), n
        assert n in m.__all__, f"binding lacks {n}"


def test_size_queries(lib):
    assert m.mxq_scale_bytes(128, 4) == 512
    assert m.mxq_scale_bytes(130, 5) == 256 * 8
    assert m.mxq_scale_bytes(0, 4) == 0
    assert m.mxq_grouped_padded_rows(32768, 32) == 128 * (256 + 32)
    M, N, K = 8192, 14336, 4096
    saved = m.mxq_linear_saved_bytes(M, N, K, m.SAVE_QUANT)
    # (M*K + N*K) codes + their scales, each rounded to 256 bytes
    assert saved == M * K + K * (M // 32) + N * K + K * (N // 32)
    assert m.mxq_linear_saved_bytes(M, N, K, m.RECOMPUTE) == 0
    assert m.mxq_linear_ctx_bytes(M, N, K, m.RECOMPUTE) == N * M + N * (M // 32)
    assert m.mxq_linear_workspace_bytes(M, N, K, m.RECOMPUTE) >= m.mxq_linear_workspace_bytes(M, N, K, m.SAVE_QUANT)
    # weight cache: row(W) + colT(W); the cached path's ctx has no colT(W)
    assert m.mxq_linear_weight_cache_bytes(N, K) == 2 * (N * K + K * (N // 32))
    colTW = N * K + N * (K // 32)
    assert m.mxq_linear_wq_ctx_bytes(M, N, K, m.SAVE_QUANT) == m.mxq_linear_ctx_bytes(M, N, K, m.SAVE_QUANT) - colTW
    assert m.mxq_linear_wq_ctx_bytes(M, N, K, m.RECOMPUTE) == m.mxq_linear_ctx_bytes(M, N, K, m.RECOMPUTE)


def _status(fn, *args):
    try:
        fn(*args)
    except m.MXQError as e:
        return e.status
    return 0


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced by a rejected call


def test_host_validation_rejects_before_launch(lib):
    INV, UNS = 1, 2
    # GEMM: K must be a positive multiple of 32, ldc >= N, pointers aligned
    assert _status(m.mxq_gemm, FAKE, FAKE, FAKE, FAKE, 128, 128, 33, FAKE, 128, 0) == INV
    assert _status(m.mxq_gemm, FAKE, FAKE, FAKE, FAKE, 128, 128, 64, FAKE, 64, 0) == INV
    assert _status(m.mxq_gemm, FAKE + 4, FAKE, FAKE, FAKE, 128, 128, 64, FAKE, 128, 0) == INV
    assert _status(m.mxq_gemm, None, FAKE, FAKE, FAKE, 128, 128, 64, FAKE, 128, 0) == INV
    # MXFP4 QDQ: block size 32 only, scale_factor > 0 (AMCT wrapper / config checks)
    assert _status(m.mxq_qdq_mxfp4, FAKE, FAKE, 4, 64, 16, 6.0, 0) == UNS
    assert _status(m.mxq_qdq_mxfp4, FAKE, FAKE, 4, 64, 32, 0.0, 0) == INV
    assert _status(m.mxq_qdq_mxfp4, FAKE, FAKE, 4, 64, 32, -1.0, 0) == INV
    assert _status(m.mxq_qdq_mxfp4, FAKE, FAKE, 4, 64, 32, float("nan"), 0) == INV
    # clipped STE: same checks as the QDQ plus a non-null, aligned mask
    assert _status(m.mxq_mxfp4_ste_forward, FAKE, FAKE, FAKE, 4, 64, 16, 6.0, 0) == UNS
    assert _status(m.mxq_mxfp4_ste_forward, FAKE, FAKE, None, 4, 64, 32, 6.0, 0) == INV
    assert _status(m.mxq_mxfp4_ste_forward, FAKE, FAKE, FAKE + 2, 4, 64, 32, 6.0, 0) == INV
    assert _status(m.mxq_mxfp4_ste_forward, FAKE, FAKE, FAKE, 4, 64, 32, 0.0, 0) == INV
    assert _status(m.mxq_mxfp4_ste_backward, FAKE, None, 4, 64, FAKE, 0) == INV
    assert _status(m.mxq_mxfp4_ste_backward, None, FAKE, 4, 64, FAKE, 0) == INV
    assert _status(m.mxq_mxfp4_ste_backward, FAKE, FAKE, -1, 64, FAKE, 0) == INV
    assert _status(m.mxq_mxfp4_ste_backward, None, None, 0, 64, None, 0) == 0
    # QAT linear forward: dims multiple of 32, sf > 0, workspace, aligned bias
    assert _status(m.mxq_qat_linear_fwd, FAKE, FAKE, None, 64, 64, 48, 1, 6.0, FAKE, FAKE, 1 << 30, 0) == INV
    assert _status(m.mxq_qat_linear_fwd, FAKE, FAKE, None, 64, 64, 64, 1, 0.0, FAKE, FAKE, 1 << 30, 0) == INV
    assert _status(m.mxq_qat_linear_fwd, FAKE, FAKE, FAKE + 2, 64, 64, 64, 1, 6.0, FAKE, FAKE, 1 << 30, 0) == INV
    assert _status(m.mxq_qat_linear_fwd, FAKE, FAKE, None, 64, 64, 64, 1, 6.0, FAKE, FAKE, 16, 0) == INV
    assert m.mxq_qat_linear_workspace_bytes(64, 64, 64, 1) == 2 * (64 * 64 + 512)
    assert m.mxq_qat_linear_workspace_bytes(64, 64, 64, 0) == 2 * 64 * 64
    # bf16 quant-dequant: cols % 32, aligned pointers
    assert _status(m.mxq_qdq_mxfp4_bf16, FAKE, FAKE, 4, 48, 32, 6.0, 0) == UNS
    assert _status(m.mxq_qdq_mxfp4_bf16, FAKE + 8, FAKE, 4, 64, 32, 6.0, 0) == INV
    # weight cache: size and dims checked before launch
    assert _status(m.mxq_linear_quantize_weight, FAKE, 64, 64, FAKE, 16, 0) == INV
    assert _status(m.mxq_linear_quantize_weight, FAKE, 64, 48, FAKE, 1 << 30, 0) == INV
    assert _status(m.mxq_linear_fwd_wq, FAKE, FAKE, 64, 64, 64, m.SAVE_QUANT, FAKE, FAKE, FAKE, 16, 0) == INV
    # failure-detection self-test: bounded timeout, device flag required
    assert _status(m.mxq_selftest_wait_timeout, 0, FAKE, 0) == INV
    assert _status(m.mxq_selftest_wait_timeout, 20000, FAKE, 0) == INV
    assert _status(m.mxq_selftest_wait_timeout, 50, None, 0) == INV
    # quantize: MXFP8 needs bf16, E2M1 is last-axis only, block axis multiple of 32
    assert _status(m.mxq_quantize, FAKE, m.F32, 64, 64, 64, -1, m.E4M3, 0, FAKE, FAKE, None, None, 0) == UNS
    assert _status(m.mxq_quantize, FAKE, m.BF16, 64, 64, 64, -2, m.E2M1, 0, None, None, FAKE, FAKE, 0) == UNS
    assert _status(m.mxq_quantize, FAKE, m.BF16, 64, 48, 48, -1, m.E4M3, 0, FAKE, FAKE, None, None, 0) == INV
    assert _status(m.mxq_quantize, FAKE, m.BF16, 64, 64, 64, 0, m.E4M3, 0, FAKE, FAKE, None, None, 0) == INV
    assert _status(m.mxq_quantize, FAKE, m.BF16, 64, 64, 64, -1, m.E4M3, 0, None, FAKE, None, None, 0) == INV
    # empty input is a no-op that succeeds without touching the device
    assert _status(m.mxq_quantize, None, m.BF16, 0, 64, 64, -1, m.E4M3, 0, None, None, None, None, 0) == 0
    assert _status(m.mxq_gemm, None, None, None, None, 0, 0, 64, None, 0, 0) == 0
    # grouped: E range, t_pad capacity, N multiple of 128 for FWD/DX
    assert _status(m.mxq_quantize_grouped_col, FAKE, 100, 64, FAKE, 0, 1024, FAKE, FAKE, 0) == INV
    assert _status(m.mxq_quantize_grouped_col, FAKE, 1000, 64, FAKE, 4, 1024, FAKE, FAKE, 0) == INV
    # grouped dual: row outputs both or neither, and cols % 32 == 0 for them
    assert _status(m.mxq_quantize_grouped_dual, FAKE, 100, 64, FAKE, 2, 512, FAKE, None, FAKE, FAKE, 0) == INV
    assert _status(m.mxq_quantize_grouped_dual, FAKE, 100, 72, FAKE, 2, 512, FAKE, FAKE, FAKE, FAKE, 0) == INV
    assert _status(m.mxq_quantize_grouped_dual, FAKE, 100, 64, FAKE, 2, 128, FAKE, FAKE, FAKE, FAKE, 0) == INV
    assert "t_pad" in m.mxq_last_error_string()
    assert _status(m.mxq_grouped_gemm, m.GG_FWD, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 100, 192, 64, 0, FAKE, 0) == INV
    assert _status(m.mxq_grouped_gemm, m.GG_DW, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 100, 128, 64, 100, FAKE, 0) == INV
    # the per-group padded row scales: the row outputs are required, and the
    # forward / dX take t_pad = 0 or a valid padded length
    assert _status(m.mxq_quantize_grouped_dual_padded, FAKE, 100, 64, FAKE, 2, 512, None, None, FAKE, FAKE,
                   0) == INV
    assert _status(m.mxq_quantize_grouped_dual_padded, FAKE, 100, 64, FAKE, 2, 128, FAKE, FAKE, FAKE, FAKE,
                   0) == INV
    assert _status(m.mxq_grouped_gemm, m.GG_FWD, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 100, 128, 64, 200, FAKE, 0) == INV
    assert "t_pad" in m.mxq_last_error_string()
    assert _status(m.mxq_grouped_gemm, m.GG_DX, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 100, 128, 64, -128, FAKE, 0) == INV
    # grouped QAT forward: N multiple of 128, finite positive scale factor, workspace size
    ws = m.mxq_qat_grouped_fwd_workspace_bytes(100, 4, 128, 64, 1)
    assert ws > 0 and m.mxq_qat_grouped_fwd_workspace_bytes(100, 4, 128, 64, 0) == 2 * 4 * 128 * 64
    assert _status(m.mxq_qat_grouped_fwd, FAKE, FAKE, FAKE, 4, 100, 96, 64, 1, 6.0, FAKE, FAKE, ws, 0) == INV
    assert _status(m.mxq_qat_grouped_fwd, FAKE, FAKE, FAKE, 4, 100, 128, 64, 1, 0.0, FAKE, FAKE, ws, 0) == INV
    assert _status(m.mxq_qat_grouped_fwd, FAKE, FAKE, FAKE, 4, 100, 128, 64, 1, 6.0, FAKE, FAKE, ws - 1, 0) == INV
    assert "workspace" in m.mxq_last_error_string()
    assert _status(m.mxq_qat_grouped_fwd, None, FAKE, FAKE, 4, 0, 128, 64, 1, 6.0, None, FAKE, ws, 0) == 0
    # grouped linear layer: N multiple of 128, T > 0, mode, workspace
    gws = m.mxq_grouped_linear_workspace_bytes(100, 4, 128, 64, m.RECOMPUTE)
    assert gws >= m.mxq_grouped_linear_workspace_bytes(100, 4, 128, 64, m.SAVE_QUANT) > 0
    assert _status(m.mxq_grouped_linear_fwd, FAKE, FAKE, FAKE, 4, 100, 96, 64, m.SAVE_QUANT, FAKE, FAKE, FAKE, gws,
                   0) == INV
    assert _status(m.mxq_grouped_linear_fwd, FAKE, FAKE, FAKE, 4, 0, 128, 64, m.SAVE_QUANT, FAKE, FAKE, FAKE, gws,
                   0) == INV
    assert _status(m.mxq_grouped_linear_bwd_dx, FAKE, FAKE, FAKE, 4, 100, 128, 64, 7, FAKE, FAKE, FAKE, gws, 0) == INV
    assert _status(m.mxq_grouped_linear_bwd_dw, FAKE, FAKE, FAKE, 4, 100, 128, 64, m.RECOMPUTE, FAKE, FAKE, FAKE, 16,
                   0) == INV
    assert "workspace" in m.mxq_last_error_string()
    assert m.mxq_grouped_linear_saved_bytes(100, 4, 128, 64, m.RECOMPUTE) == 0
    # linear: dimensions multiple of 32, workspace large enough
    assert _status(m.mxq_linear_fwd, FAKE, FAKE, 100, 64, 64, m.SAVE_QUANT, FAKE, FAKE, FAKE, 1 << 30, 0) == INV
    assert _status(m.mxq_linear_fwd, FAKE, FAKE, 64, 64, 64, m.SAVE_QUANT, FAKE, FAKE, FAKE, 16, 0) == INV
    assert _status(m.mxq_linear_fwd, FAKE, FAKE, 64, 64, 64, 7, FAKE, FAKE, FAKE, 1 << 30, 0) == INV
    assert "workspace" in m.mxq_last_error_string() or "mode" in m.mxq_last_error_string()


def test_group_offsets_validated_on_the_host(lib):
    """The rule every grouped kernel applies to its device offsets, checked
    here on host arrays: off[0] = 0, non-decreasing, off[E] = T."""
    INV = 1
    ok = [0, 10, 10, 300, 300]
    assert _status(m.mxq_validate_group_offsets, ok, 4, 300) == 0
    assert _status(m.mxq_validate_group_offsets, [0, 0], 1, 0) == 0            # one empty group
    bad = {
        "off[0]": ([5, 10, 10, 300, 300], 300),                                 # does not start at 0
        "decrease": ([0, 200, 100, 300, 300], 300),                             # non-monotone
        "negative": ([0, -8, 10, 300, 300], 300),                               # negative (and decreasing)
        "must equal T": ([0, 10, 10, 300, 299], 300),                           # off[E] != T
        "past T": ([0, 10, 400, 500, 600], 300),                                # rows past the tensor
    }
    for what, (off, T) in bad.items():
        assert _status(m.mxq_validate_group_offsets, off, 4, T) == INV, what
    assert _status(m.mxq_validate_group_offsets, [0, 2, 1], 2, 1) == INV
    assert "must not decrease" in m.mxq_last_error_string()
    assert _status(m.mxq_validate_group_offsets, ok, 0, 300) == INV           # E out of range
    assert _status(m.mxq_validate_group_offsets, ok, 4, -1) == INV            # negative T
    # the device checker rejects bad arguments on the host, before any launch
    assert _status(m.mxq_check_group_offsets, None, 4, 300, 0) == INV
    assert _status(m.mxq_check_group_offsets, FAKE + 4, 4, 300, 0) == INV
    assert _status(m.mxq_check_group_offsets, FAKE, 0, 300, 0) == INV


def test_debug_build_exports_every_symbol_and_loads_under_the_switch():
    """libmxq_debug.so (MXQ_DEBUG: bounds checks on every computed global
    access) builds, exports the same entry points, and is what the binding
    loads when MXQ_LIBRARY=debug."""
    import subprocess
    import sys
    from mx_block_scaled_mxq_gb300 import build as b
    path = b.build(debug=True)
    raw = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(raw, n), n
    env = dict(os.environ, MXQ_LIBRARY="debug")
    code = "import mx_block_scaled_mxq_gb300 as m; m.load(); import os; print(os.path.basename(m.library_path()))"
    res = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip().endswith("libmxq_debug.so")
