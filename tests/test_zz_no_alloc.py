"""mxq_linear_fwd_noalloc: the linear forward for callers that cannot allocate
device memory (for example a plug-in inside a framework that owns the whole
memory pool and forbids cudaMalloc).  It keeps its scratch in a fixed array
inside the library, so the caller passes only x, w and y.

It runs the same quant and GEMM kernels as the regular mxq_linear_fwd (which
takes a workspace from the caller), so its output must equal that one bit for
bit, and lie within the GEMM tolerance of the other tests from the oracle's
binary64 product -- on calls in a row, where each later call reuses the
scratch an earlier, larger one left behind.  This file is collected last so
that a run stopping at its first failure has already run every other test."""
import numpy as np
import pytest
import torch

import mxq_inputs
import oracle
from test_gpu_gemm import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _regular_forward(mxq, x, w, M, N, K):
    mode = mxq.RECOMPUTE
    ctx = torch.empty(max(mxq.mxq_linear_ctx_bytes(M, N, K, mode), 1), dtype=torch.uint8, device=DEV)
    wsb = mxq.mxq_linear_workspace_bytes(M, N, K, mode)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_linear_fwd(x, w, M, N, K, mode, ctx, y, ws, wsb)
    return y


def test_no_alloc_forward_matches_regular_forward_and_oracle(mxq):
    # calls in a row with different sizes and inputs: the largest first, then
    # sizes whose scale tiles are only partly used (M and N not multiples of
    # 128), so anything the scratch kept from an earlier call would show up
    for (M, N, K), seed in (((1024, 2048, 4096), 1), ((256, 512, 512), 2), ((96, 160, 64), 3),
                            ((1024, 2048, 4096), 4)):
        x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=seed)
        xg, wg = x.to(DEV), w.to(DEV)
        ref = _regular_forward(mxq, xg, wg, M, N, K)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        mxq.mxq_linear_fwd_noalloc(xg, wg, M, N, K, y)
        torch.cuda.synchronize()
        assert mxq.mxq_poll_device_error() == 0
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), (M, N, K)
        qx, sx = oracle.mxfp8_quant_rows(x)
        qw, sw = oracle.mxfp8_quant_rows(w)
        check_close(y, oracle.gemm_ref(qx, sx, qw, sw))


def test_no_alloc_forward_allocates_nothing(mxq):
    M, N, K = 512, 1024, 2048
    x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=5)
    xg, wg = x.to(DEV), w.to(DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_linear_fwd_noalloc(xg, wg, M, N, K, y)       # loads the module, looks up the scratch
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        mxq.mxq_linear_fwd_noalloc(xg, wg, M, N, K, y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert mxq.mxq_poll_device_error() == 0


def test_no_alloc_forward_rejects_sizes_beyond_its_scratch(mxq):
    M, N, K = 8192, 14336, 4096          # needs ~92 MB of quantized operands
    x = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    w = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mxq.MXQError) as err:
        mxq.mxq_linear_fwd_noalloc(x, w, M, N, K, y)
    assert err.value.status == 1 and "MXQ_NOALLOC_SCRATCH_BYTES" in str(err.value)
