"""GPU parity of the MXFP8 linear layer (forward, input gradient, weight
gradient) in saved-quant and recompute modes.  The two modes must agree bit for
bit (the fb-split PR's flag path shipped broken because nothing compared them),
and both must match the binary64 oracle within tolerance."""
import numpy as np
import pytest
import torch

import mxq_inputs
import oracle
from test_gpu_gemm import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_layer(mxq, x, w, dy, mode):
    M, K = x.shape
    N = w.shape[0]
    xg, wg, dyg = x.to(DEV), w.to(DEV), dy.to(DEV)
    ctx = torch.empty(mxq.mxq_linear_ctx_bytes(M, N, K, mode), dtype=torch.uint8, device=DEV)
    wsb = mxq.mxq_linear_workspace_bytes(M, N, K, mode)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=DEV)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    dx = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    dw = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_linear_fwd(xg, wg, M, N, K, mode, ctx, y, ws, wsb)
    ws.fill_(0xCD)  # workspace is scratch: nothing may depend on it surviving between calls
    mxq.mxq_linear_bwd_dx(dyg, wg, M, N, K, mode, ctx, dx, ws, wsb)
    ws.fill_(0xCD)
    mxq.mxq_linear_bwd_dw(dyg, xg, M, N, K, mode, ctx, dw, ws, wsb)
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    return y, dx, dw


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (384, 640, 256), (96, 160, 2048), (32, 32, 32)])
def test_modes_agree_and_match_oracle(mxq, M, N, K):
    x, w, dy = mxq_inputs.linear_inputs(M, N, K, seed=M + N)
    save = run_layer(mxq, x, w, dy, mxq.SAVE_QUANT)
    rec = run_layer(mxq, x, w, dy, mxq.RECOMPUTE)
    for a, b in zip(save, rec):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ry, rdx, rdw = oracle.linear_ref(x, w, dy)
    check_close(save[0], ry)
    check_close(save[1], rdx)
    check_close(save[2], rdw)


def test_saved_bytes_are_the_column_quants():
    import mx_block_scaled_mxq_gb300 as m
    M, N, K = 8192, 14336, 4096
    assert m.mxq_linear_saved_bytes(M, N, K, m.SAVE_QUANT) == (M * K + N * K) * 33 // 32
    assert m.mxq_linear_saved_bytes(M, N, K, m.RECOMPUTE) == 0


def test_full_size_layer_sampled(mxq):
    """M=8192, N=14336, K=4096 in both modes: bitwise-equal outputs, and each of
    Y, dX, dW checked against the oracle on sampled rows."""
    M, N, K = 8192, 14336, 4096
    x, w, dy = mxq_inputs.linear_inputs(M, N, K, seed=0)
    save = run_layer(mxq, x, w, dy, mxq.SAVE_QUANT)
    rec = run_layer(mxq, x, w, dy, mxq.RECOMPUTE)
    for a, b in zip(save, rec):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    del rec
    y, dx, dw = save
    rng = np.random.default_rng(1)
    rm = np.unique(np.concatenate([rng.choice(M, 48, replace=False), [0, M - 1]]))
    rn = np.unique(np.concatenate([rng.choice(N, 48, replace=False), [0, N - 1]]))
    tm, tn = torch.from_numpy(rm), torch.from_numpy(rn)
    # Y rows: row-quant X rows, row-quant W
    qx, sx = oracle.mxfp8_quant_rows(x[tm])
    qw, sw = oracle.mxfp8_quant_rows(w)
    check_close(y[tm.to(DEV)], oracle.gemm_ref(qx, sx, qw, sw))
    del qw, sw
    # dX rows: row-quant dY rows, column-quant W (blocks along N)
    qdy, sdy = oracle.mxfp8_quant_rows(dy[tm])
    qwT, swT = oracle.mxfp8_quant_cols(w)
    check_close(dx[tm.to(DEV)], oracle.gemm_ref(qdy, sdy, qwT, swT))
    del qwT, swT
    # dW rows n: column-quant of dY's columns n (blocks along M), column-quant X
    qdyT, sdyT = oracle.mxfp8_quant_cols(dy[:, tn].contiguous())
    qxT, sxT = oracle.mxfp8_quant_cols(x)
    check_close(dw[tn.to(DEV)], oracle.gemm_ref(qdyT, sdyT, qxT, sxT))
