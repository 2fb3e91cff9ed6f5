"""Every entry point runs on the stream it is given.

The caller's stream first sleeps (a spin kernel of about 50 ms), then writes
the call's inputs, then makes the call with that stream passed explicitly
while the current stream is the default one.  A call that launched anywhere
else would run during the sleep and read the inputs' old contents (zeros);
on the right stream it sees the new ones and must equal, bit for bit, the
same call made on the default stream with the new inputs in place."""
import numpy as np
import pytest
import torch

import mxq_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
SLEEP_CYCLES = 100_000_000


def _poison(t):
    if t.dtype in (torch.bfloat16, torch.float32):
        t.fill_(float("nan"))
    else:
        t.fill_(0xAB)


def check_on_side_stream(inputs, outputs, call):
    """inputs: {tensor: new value}; outputs: tensors the call writes;
    call(stream) makes the call on `stream` (None: the current stream)."""
    for dst, new in inputs.items():
        dst.copy_(new)
    for o in outputs:
        _poison(o)
    call(None)
    torch.cuda.synchronize()
    ref = [o.clone() for o in outputs]

    for dst in inputs:
        dst.zero_()
    for o in outputs:
        _poison(o)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(SLEEP_CYCLES)
        for dst, new in inputs.items():
            dst.copy_(new)
    call(s)  # the current stream is the default one here
    s.synchronize()
    for o, r in zip(outputs, ref):
        assert torch.equal(o.view(torch.uint8), r.view(torch.uint8))


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (scale * torch.randn(*shape, generator=g)).bfloat16().to(DEV)


def _u8(n):
    return torch.empty(n, dtype=torch.uint8, device=DEV)


def test_dual_quant(mxq):
    R, C = 1024, 2048
    x_new, x = _bf16((R, C), 1), torch.empty(R, C, dtype=torch.bfloat16, device=DEV)
    q, s = _u8(R * C), _u8(mxq.mxq_scale_bytes(R, C // 32))
    qT, sT = _u8(R * C), _u8(mxq.mxq_scale_bytes(C, R // 32))
    check_on_side_stream({x: x_new}, [q, s, qT, sT],
                         lambda st: mxq.mxq_quantize(x, mxq.BF16, R, C, C, -1, mxq.E4M3, 1, q, s, qT, sT, st))


def test_grouped_dual_quant_padded(mxq):
    sizes = [3, 0, 600, 97, 300]
    E, T, C = len(sizes), sum(sizes), 256
    off = torch.from_numpy(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)).to(DEV)
    tp = mxq.mxq_grouped_padded_rows(T, E)
    x_new, x = _bf16((T, C), 2), torch.empty(T, C, dtype=torch.bfloat16, device=DEV)
    q, s = _u8(T * C), _u8(mxq.mxq_scale_bytes(tp, C // 32))
    qT, sT = _u8(C * tp), _u8(mxq.mxq_scale_bytes(C, tp // 32))
    check_on_side_stream({x: x_new}, [q, s, qT, sT],
                         lambda st: mxq.mxq_quantize_grouped_dual_padded(x, T, C, off, E, tp, q, s, qT, sT, st))


def test_qdq_mxfp4(mxq):
    R, C = 512, 1024
    g = torch.Generator().manual_seed(3)
    x_new = torch.randn(R, C, generator=g).to(DEV)
    x, y = torch.empty_like(x_new), torch.empty_like(x_new)
    check_on_side_stream({x: x_new}, [y], lambda st: mxq.mxq_qdq_mxfp4(x, y, R, C, 32, 6.0, st))


def test_gemm(mxq):
    M, N, K = 384, 512, 640
    xq, xs = mxq.quantize_mxfp8(_bf16((M, K), 4))[:2]
    wq, ws = mxq.quantize_mxfp8(_bf16((N, K), 5, 0.02))[:2]
    a, sa, b, sb = (torch.empty_like(t) for t in (xq, xs, wq, ws))
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    check_on_side_stream({a: xq, sa: xs, b: wq, sb: ws}, [y],
                         lambda st: mxq.mxq_gemm(a, sa, b, sb, M, N, K, y, N, st))


def test_grouped_gemm_forward(mxq):
    sizes = [129, 0, 255, 40]
    E, T, K, N = len(sizes), sum(sizes), 256, 256
    off_np, xm, wm, _ = mxq_inputs.moe_inputs(E, T, K, N, seed=6, sizes=sizes)
    off = torch.from_numpy(np.asarray(off_np, dtype=np.int64)).to(DEV)
    xq, xs = mxq.quantize_mxfp8(xm.to(DEV))[:2]
    wq, ws = mxq.quantize_mxfp8(wm.reshape(E * N, K).to(DEV))[:2]
    a, sa, b, sb = (torch.empty_like(t) for t in (xq, xs, wq, ws))
    y = torch.empty(T, N, dtype=torch.bfloat16, device=DEV)
    check_on_side_stream({a: xq, sa: xs, b: wq, sb: ws}, [y],
                         lambda st: mxq.mxq_grouped_gemm(mxq.GG_FWD, a, sa, b, sb, off, E, T, N, K, 0, y, st))


@pytest.mark.parametrize("mode_name", ["SAVE_QUANT", "RECOMPUTE"])
def test_linear_forward(mxq, mode_name):
    mode = getattr(mxq, mode_name)
    M, N, K = 256, 512, 512
    x_new, w_new = _bf16((M, K), 7), _bf16((N, K), 8, 0.02)
    x, w = torch.empty_like(x_new), torch.empty_like(w_new)
    ctx = _u8(max(mxq.mxq_linear_ctx_bytes(M, N, K, mode), 1))
    wsb = mxq.mxq_linear_workspace_bytes(M, N, K, mode)
    ws = _u8(max(wsb, 1))
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    check_on_side_stream({x: x_new, w: w_new}, [y],
                         lambda st: mxq.mxq_linear_fwd(x, w, M, N, K, mode, ctx, y, ws, wsb, st))


def test_grouped_linear_forward(mxq):
    sizes = [100, 0, 300, 5]
    E, T, K, N = len(sizes), sum(sizes), 256, 256
    off_np, xm, wm, _ = mxq_inputs.moe_inputs(E, T, K, N, seed=9, sizes=sizes)
    off = torch.from_numpy(np.asarray(off_np, dtype=np.int64)).to(DEV)
    x_new, w_new = xm.to(DEV), wm.to(DEV)
    x, w = torch.empty_like(x_new), torch.empty_like(w_new)
    mode = mxq.SAVE_QUANT
    ctx = _u8(mxq.mxq_grouped_linear_ctx_bytes(T, E, N, K, mode))
    wsb = mxq.mxq_grouped_linear_workspace_bytes(T, E, N, K, mode)
    ws = _u8(wsb)
    y = torch.empty(T, N, dtype=torch.bfloat16, device=DEV)
    check_on_side_stream({x: x_new, w: w_new}, [y],
                         lambda st: mxq.mxq_grouped_linear_fwd(x, w, off, E, T, N, K, mode, ctx, y, ws, wsb, st))


def test_qat_linear_forward(mxq):
    M, N, K = 256, 384, 512
    x_new, w_new = _bf16((M, K), 10), _bf16((N, K), 11, 0.02)
    x, w = torch.empty_like(x_new), torch.empty_like(w_new)
    wsb = mxq.mxq_qat_linear_workspace_bytes(M, N, K, 1)
    ws = _u8(wsb)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    check_on_side_stream({x: x_new, w: w_new}, [y],
                         lambda st: mxq.mxq_qat_linear_fwd(x, w, None, M, N, K, 1, 6.0, y, ws, wsb, st))


@pytest.mark.parametrize("mode_name", ["SAVE_QUANT", "RECOMPUTE"])
def test_linear_backward(mxq, mode_name):
    """bwd_dx then bwd_dw on the side stream, after a forward on the default one."""
    mode = getattr(mxq, mode_name)
    M, N, K = 256, 512, 384
    x, w = _bf16((M, K), 12), _bf16((N, K), 13, 0.02)
    dy_new, dy = _bf16((M, N), 14, 1e-3), torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    ctx = _u8(max(mxq.mxq_linear_ctx_bytes(M, N, K, mode), 1))
    wsb = mxq.mxq_linear_workspace_bytes(M, N, K, mode)
    ws = _u8(max(wsb, 1))
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    mxq.mxq_linear_fwd(x, w, M, N, K, mode, ctx, y, ws, wsb)
    torch.cuda.synchronize()
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    dw = torch.empty(N, K, dtype=torch.bfloat16, device=DEV)

    def call(st):
        mxq.mxq_linear_bwd_dx(dy, w, M, N, K, mode, ctx, dx, ws, wsb, st)
        mxq.mxq_linear_bwd_dw(dy, x, M, N, K, mode, ctx, dw, ws, wsb, st)
    check_on_side_stream({dy: dy_new}, [dx, dw], call)


def test_grouped_linear_backward(mxq):
    sizes = [100, 0, 300, 5]
    E, T, K, N = len(sizes), sum(sizes), 256, 256
    off_np, xm, wm, dym = mxq_inputs.moe_inputs(E, T, K, N, seed=15, sizes=sizes)
    off = torch.from_numpy(np.asarray(off_np, dtype=np.int64)).to(DEV)
    x, w = xm.to(DEV), wm.to(DEV)
    dy_new = dym.to(DEV)
    dy = torch.empty_like(dy_new)
    mode = mxq.RECOMPUTE
    ctx = _u8(mxq.mxq_grouped_linear_ctx_bytes(T, E, N, K, mode))
    wsb = mxq.mxq_grouped_linear_workspace_bytes(T, E, N, K, mode)
    ws = _u8(wsb)
    dx = torch.empty(T, K, dtype=torch.bfloat16, device=DEV)
    dw = torch.empty(E, N, K, dtype=torch.bfloat16, device=DEV)

    def call(st):
        mxq.mxq_grouped_linear_bwd_dx(dy, w, off, E, T, N, K, mode, ctx, dx, ws, wsb, st)
        mxq.mxq_grouped_linear_bwd_dw(dy, x, off, E, T, N, K, mode, ctx, dw, ws, wsb, st)
    check_on_side_stream({dy: dy_new}, [dx, dw], call)
