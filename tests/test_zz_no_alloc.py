"""mxq_linear_fwd_noalloc: the linear forward for callers that cannot allocate
device memory (for example a plug-in inside a framework that owns the whole
memory pool and forbids cudaMalloc).  It keeps its scratch in a fixed array
inside the library, so the caller passes only x, w and y.

Its output must match the regular mxq_linear_fwd (which takes a workspace
from the caller) within the GEMM tolerance of the other tests, on two calls in
a row -- the second call reuses the scratch the first one left behind.  This
file is collected last so that a run stopping at its first failure has
already run every other test."""
import numpy as np
import pytest
import torch

import mxq_inputs
from test_gpu_gemm import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _regular_forward(mxq, x, w, M, N, K):
    mode = mxq.RECOMPUTE
    ctx = torch.empty(mxq.mxq_linear_ctx_bytes(M, N, K, mode), dtype=torch.uint8, device=DEV)
    wsb = mxq.mxq_linear_workspace_bytes(M, N, K, mode)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_linear_fwd(x, w, M, N, K, mode, ctx, y, ws, wsb)
    return y


def test_no_alloc_forward_matches_regular_forward_twice(mxq):
    # two calls in a row, the second with different sizes and inputs, so that
    # anything left in the shared scratch by the first would show up
    for (M, N, K), seed in (((1024, 2048, 4096), 1), ((256, 512, 512), 2)):
        x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=seed)
        xg, wg = x.to(DEV), w.to(DEV)
        ref = _regular_forward(mxq, xg, wg, M, N, K)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        mxq.mxq_linear_fwd_noalloc(xg, wg, M, N, K, y)
        torch.cuda.synchronize()
        assert mxq.mxq_poll_device_error() == 0
        check_close(y, ref.float().cpu().numpy().astype(np.float64))


def test_no_alloc_forward_rejects_sizes_beyond_its_scratch(mxq):
    M, N, K = 8192, 14336, 4096          # needs ~92 MB of quantized operands
    x = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    w = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mxq.MXQError) as err:
        mxq.mxq_linear_fwd_noalloc(x, w, M, N, K, y)
    assert err.value.status == 1 and "MXQ_NOALLOC_SCRATCH_BYTES" in str(err.value)
