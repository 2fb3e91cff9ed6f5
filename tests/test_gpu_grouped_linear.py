"""The MoE expert layer's forward and backward through mxq_grouped_linear_*,
in both modes ([FB]: saved-quant vs recompute-in-backward): the two modes must
be bitwise identical, equal bit for bit the grouped GEMMs called on the same
quantized operands, and within the GEMM tolerance of the binary64 oracle."""
import numpy as np
import pytest
import torch

import mxq_inputs
import oracle
from test_gpu_gemm import check_close
from test_gpu_grouped import MoE, _oracle_w

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_layer(mxq, off, x, w, dy, mode):
    """y, dx, dw of one step (fwd, bwd_dx, bwd_dw) through the C ABI."""
    E, N, K = w.shape
    T = x.shape[0]
    d_off = torch.from_numpy(np.asarray(off, dtype=np.int64)).to(DEV)
    xg, wg, dyg = x.to(DEV), w.to(DEV), dy.to(DEV)
    ctx = torch.empty(max(mxq.mxq_grouped_linear_ctx_bytes(T, E, N, K, mode), 1), dtype=torch.uint8, device=DEV)
    wsb = mxq.mxq_grouped_linear_workspace_bytes(T, E, N, K, mode)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=DEV)
    y = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    dx = torch.full((T, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    dw = torch.full((E, N, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_grouped_linear_fwd(xg, wg, d_off, E, T, N, K, mode, ctx, y, ws, wsb)
    mxq.mxq_grouped_linear_bwd_dx(dyg, wg, d_off, E, T, N, K, mode, ctx, dx, ws, wsb)
    mxq.mxq_grouped_linear_bwd_dw(dyg, xg, d_off, E, T, N, K, mode, ctx, dw, ws, wsb)
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    return y, dx, dw


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("sizes,K,N", [([3, 0, 200, 0, 97], 256, 256), ([128, 128], 160, 384),
                                       ([0, 0, 1], 1024, 1024), ([129, 127, 0, 3, 255, 1], 224, 256)])
def test_modes_agree_and_match_oracle(mxq, sizes, K, N):
    off, x, w, dy = mxq_inputs.moe_inputs(len(sizes), sum(sizes), K, N, seed=len(sizes) + 3 * K, sizes=sizes)
    save = run_layer(mxq, off, x, w, dy, mxq.SAVE_QUANT)
    rec = run_layer(mxq, off, x, w, dy, mxq.RECOMPUTE)
    for a, b in zip(save, rec):
        assert _same(a, b)
    y, dx, dw = save
    qx, sx = oracle.mxfp8_quant_rows(x)
    qw, sw, qwT, swT = _oracle_w(w)
    qdy, sdy = oracle.mxfp8_quant_rows(dy)
    check_close(y, oracle.grouped_fwd_ref(qx, sx, qw, sw, off))
    check_close(dx, oracle.grouped_fwd_ref(qdy, sdy, qwT, swT, off))
    qdyT, sdyT = oracle.mxfp8_quant_cols_grouped(dy, off)
    qxT, sxT = oracle.mxfp8_quant_cols_grouped(x, off)
    ref_dw = oracle.grouped_dw_ref(qdyT, sdyT, qxT, sxT, off)
    for e in range(len(sizes)):
        if sizes[e] == 0:
            assert not torch.any(dw[e].float() != 0)
        else:
            check_close(dw[e], ref_dw[e])


def test_saved_bytes_are_the_column_quants(mxq):
    T, E, N, K = 32768, 32, 4096, 7168
    t_pad = mxq.mxq_grouped_padded_rows(T, E)
    xT = K * t_pad + mxq.mxq_scale_bytes(K, t_pad // 32)
    wT = K * E * N + mxq.mxq_scale_bytes(K, E * N // 32)
    assert mxq.mxq_grouped_linear_saved_bytes(T, E, N, K, mxq.SAVE_QUANT) == xT + wT
    assert mxq.mxq_grouped_linear_saved_bytes(T, E, N, K, mxq.RECOMPUTE) == 0
    dyT = N * t_pad + mxq.mxq_scale_bytes(N, t_pad // 32)
    assert mxq.mxq_grouped_linear_ctx_bytes(T, E, N, K, mxq.RECOMPUTE) == dyT


def test_many_experts(mxq):
    """300 experts (tiles decoded from the device offsets): modes agree, and
    equal the grouped GEMMs on the same operands bit for bit."""
    E, T, K, N = 300, 1200, 64, 128
    sizes = mxq_inputs.dirichlet_group_sizes(E, T, alpha=0.5, seed=3)
    off, x, w, dy = mxq_inputs.moe_inputs(E, T, K, N, seed=5, sizes=sizes)
    save = run_layer(mxq, off, x, w, dy, mxq.SAVE_QUANT)
    rec = run_layer(mxq, off, x, w, dy, mxq.RECOMPUTE)
    ref = MoE(mxq, off, x, w, dy, padded=True)
    for a, b, r in zip(save, rec, (ref.fwd(), ref.dx(), ref.dw())):
        assert _same(a, b) and _same(a, r)


def test_full_size_modes_and_grouped_gemms(mxq):
    """32 experts, 32768 Dirichlet-routed rows, K = 7168, N = 4096: both modes
    bitwise identical, and bit for bit the grouped GEMMs whose outputs the
    full-size grouped test checks against the oracle."""
    E, T, K, N = 32, 32768, 7168, 4096
    off, x, w, dy = mxq_inputs.moe_inputs(E, T, K, N, seed=0)
    save = run_layer(mxq, off, x, w, dy, mxq.SAVE_QUANT)
    ref = MoE(mxq, off, x, w, dy, padded=True)
    for a, r in zip(save, (ref.fwd(), ref.dx(), ref.dw())):
        assert _same(a, r)
    del ref
    rec = run_layer(mxq, off, x, w, dy, mxq.RECOMPUTE)
    for a, b in zip(save, rec):
        assert _same(a, b)
