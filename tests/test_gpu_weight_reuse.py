"""GPU parity of quantized-weight reuse (the reuse flags of the MindSpeed
MXFP8 matmul path): W quantized once into a cache and reused by several
micro-batches' forward and input-gradient calls gives results bitwise equal
to quantizing W on every call, in both modes."""
import pytest
import torch

import mxq_inputs
import oracle
from test_gpu_gemm import check_close
from test_gpu_linear import run_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_cached(mxq, xs, w, dys, mode):
    """One optimizer step over micro-batches (x_i, dy_i) with a weight cache."""
    N, K = w.shape
    wg = w.to(DEV)
    cb = mxq.mxq_linear_weight_cache_bytes(N, K)
    cache = torch.empty(cb, dtype=torch.uint8, device=DEV)
    mxq.mxq_linear_quantize_weight(wg, N, K, cache, cb)
    outs = []
    for x, dy in zip(xs, dys):
        M = x.shape[0]
        xg, dyg = x.to(DEV), dy.to(DEV)
        ctx = torch.full((mxq.mxq_linear_wq_ctx_bytes(M, N, K, mode),), 0xAB, dtype=torch.uint8, device=DEV)
        wsb = mxq.mxq_linear_workspace_bytes(M, N, K, mode)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=DEV)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        dx = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
        dw = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device=DEV)
        mxq.mxq_linear_fwd_wq(xg, cache, M, N, K, mode, ctx, y, ws, wsb)
        ws.fill_(0xCD)
        mxq.mxq_linear_bwd_dx_wq(dyg, cache, M, N, K, mode, ctx, dx, ws, wsb)
        ws.fill_(0xCD)
        mxq.mxq_linear_bwd_dw(dyg, xg, M, N, K, mode, ctx, dw, ws, wsb)
        torch.cuda.synchronize()
        assert mxq.mxq_poll_device_error() == 0
        outs.append((y, dx, dw))
    return outs


@pytest.mark.parametrize("mode_name", ["SAVE_QUANT", "RECOMPUTE"])
@pytest.mark.parametrize("N,K", [(512, 512), (640, 256), (160, 2048)])
def test_cached_weight_is_bitwise_equal_to_per_call(mxq, mode_name, N, K):
    mode = getattr(mxq, mode_name)
    micro = [mxq_inputs.linear_inputs(M, N, K, seed=i) for i, M in enumerate([256, 96, 384])]
    w = micro[0][1]
    xs, dys = [mb[0] for mb in micro], [mb[2] for mb in micro]
    got = run_cached(mxq, xs, w, dys, mode)
    for (x, dy), outs in zip(zip(xs, dys), got):
        ref = run_layer(mxq, x, w, dy, mode)
        for a, b in zip(outs, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ry, rdx, rdw = oracle.linear_ref(xs[1], w, dys[1])
    check_close(got[1][0], ry)
    check_close(got[1][1], rdx)
    check_close(got[1][2], rdw)
