"""GPU parity of the MoE grouped GEMMs (forward, input gradient, weight
gradient) against the binary64 oracle, with ragged and empty groups."""
import numpy as np
import pytest
import torch

import mxq_inputs
import oracle
from test_gpu_gemm import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


class MoE:
    """Quantized operands of one MoE expert layer, built through the C ABI.
    padded=True takes X's and dY's row quants from the grouped dual quant with
    per-group padded row scales, and passes t_pad to the forward and dX."""

    def __init__(self, mxq, off, x, w, dy, padded=False):
        self.mxq = mxq
        self.off = off
        self.E = len(off) - 1
        self.T, self.K = x.shape
        self.N = w.shape[1]
        E, T, K, N = self.E, self.T, self.K, self.N
        self.d_off = torch.from_numpy(off).to(DEV)
        xg, wg, dyg = x.to(DEV), w.reshape(E * N, K).to(DEV), dy.to(DEV)
        self.wq, self.ws, self.wqT, self.wsT = mxq.quantize_mxfp8(wg, dual=True)  # forward B, dX B
        self.t_pad = mxq.mxq_grouped_padded_rows(T, E)
        self.row_pad = self.t_pad if padded else 0
        if padded:
            self.xq, self.xs, self.xqT, self.xsT = self._gdual_padded(xg, K)     # forward A, dW B
            self.dyq, self.dys, self.dyqT, self.dysT = self._gdual_padded(dyg, N)  # dX A, dW A
        else:
            self.xq, self.xs, _, _ = mxq.quantize_mxfp8(xg)                   # forward A
            self.dyq, self.dys, _, _ = mxq.quantize_mxfp8(dyg)                # dX A
            self.dyqT, self.dysT = self._gcol(dyg, N)                         # dW A
            self.xqT, self.xsT = self._gcol(xg, K)                            # dW B

    def _gdual_padded(self, t, C):
        u8 = lambda n: torch.empty((n,), dtype=torch.uint8, device=DEV)  # noqa: E731
        q, s = u8(max(self.T, 1) * C), u8(self.mxq.mxq_scale_bytes(self.t_pad, C // 32))
        qT, sT = u8(C * self.t_pad), u8(self.mxq.mxq_scale_bytes(C, self.t_pad // 32))
        self.mxq.mxq_quantize_grouped_dual_padded(t, self.T, C, self.d_off, self.E, self.t_pad, q, s, qT, sT)
        return q, s, qT, sT

    def _gcol(self, t, C):
        qT = torch.empty((C, self.t_pad), dtype=torch.uint8, device=DEV)
        sT = torch.empty((self.mxq.mxq_scale_bytes(C, self.t_pad // 32),), dtype=torch.uint8, device=DEV)
        self.mxq.mxq_quantize_grouped_col(t, self.T, C, self.d_off, self.E, self.t_pad, qT, sT)
        return qT, sT

    def fwd(self):
        y = torch.full((self.T, self.N), float("nan"), dtype=torch.bfloat16, device=DEV)
        self.mxq.mxq_grouped_gemm(self.mxq.GG_FWD, self.xq, self.xs, self.wq, self.ws, self.d_off, self.E, self.T,
                                  self.N, self.K, self.row_pad, y)
        return y

    def dx(self):
        dx = torch.full((self.T, self.K), float("nan"), dtype=torch.bfloat16, device=DEV)
        self.mxq.mxq_grouped_gemm(self.mxq.GG_DX, self.dyq, self.dys, self.wqT, self.wsT, self.d_off, self.E,
                                  self.T, self.N, self.K, self.row_pad, dx)
        return dx

    def dw(self):
        dw = torch.full((self.E, self.N, self.K), float("nan"), dtype=torch.bfloat16, device=DEV)
        self.mxq.mxq_grouped_gemm(self.mxq.GG_DW, self.dyqT, self.dysT, self.xqT, self.xsT, self.d_off, self.E,
                                  self.T, self.N, self.K, self.t_pad, dw)
        return dw


def _oracle_w(w):
    E = w.shape[0]
    rows = [oracle.mxfp8_quant_rows(w[e]) for e in range(E)]
    cols = [oracle.mxfp8_quant_cols(w[e]) for e in range(E)]
    return (np.stack([r[0] for r in rows]), np.stack([r[1] for r in rows]),
            np.stack([c[0] for c in cols]), np.stack([c[1] for c in cols]))


# The Frobenius bound is a statistic over the output: bf16 output rounding alone
# contributes ~1.1e-3 on average, and over a handful of elements it can exceed
# 2e-3, so every case keeps >= 1024 elements per checked output (the one-row
# group below has 1 x 1024 outputs).
@pytest.mark.parametrize("sizes,K,N", [([3, 0, 200, 0, 97], 256, 256), ([128, 128], 160, 384),
                                       ([0, 0, 1], 1024, 1024), ([700], 512, 128)])
def test_grouped_fwd_dx_dw(mxq, sizes, K, N):
    off, x, w, dy = mxq_inputs.moe_inputs(len(sizes), sum(sizes), K, N, seed=len(sizes) + K, sizes=sizes)
    moe = MoE(mxq, off, x, w, dy)
    y, dx, dw = moe.fwd(), moe.dx(), moe.dw()
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    qx, sx = oracle.mxfp8_quant_rows(x)
    qw, sw, qwT, swT = _oracle_w(w)
    qdy, sdy = oracle.mxfp8_quant_rows(dy)
    check_close(y, oracle.grouped_fwd_ref(qx, sx, qw, sw, off))
    check_close(dx, oracle.grouped_fwd_ref(qdy, sdy, qwT, swT, off))
    qdyT, sdyT = oracle.mxfp8_quant_cols_grouped(dy, off)
    qxT, sxT = oracle.mxfp8_quant_cols_grouped(x, off)
    ref_dw = oracle.grouped_dw_ref(qdyT, sdyT, qxT, sxT, off)
    got_dw = dw.float().cpu().numpy()
    for e in range(len(sizes)):
        if sizes[e] == 0:
            assert not np.any(got_dw[e]), "an empty group must give an all-zero weight gradient"
        else:
            check_close(dw[e], ref_dw[e])


def test_grouped_dirichlet_32_experts(mxq):
    off, x, w, dy = mxq_inputs.moe_inputs(32, 4096, 512, 256, seed=0)
    moe = MoE(mxq, off, x, w, dy)
    y, dx, dw = moe.fwd(), moe.dx(), moe.dw()
    qx, sx = oracle.mxfp8_quant_rows(x)
    qw, sw, qwT, swT = _oracle_w(w)
    qdy, sdy = oracle.mxfp8_quant_rows(dy)
    check_close(y, oracle.grouped_fwd_ref(qx, sx, qw, sw, off))
    check_close(dx, oracle.grouped_fwd_ref(qdy, sdy, qwT, swT, off))
    qdyT, sdyT = oracle.mxfp8_quant_cols_grouped(dy, off)
    qxT, sxT = oracle.mxfp8_quant_cols_grouped(x, off)
    ref_dw = oracle.grouped_dw_ref(qdyT, sdyT, qxT, sxT, off)
    n = np.diff(off)
    for e in range(32):
        if n[e] == 0:
            assert not torch.any(dw[e].float() != 0)
        else:
            check_close(dw[e], ref_dw[e])


def test_full_size_moe_sampled(mxq):
    """32 experts, 32768 routed rows (Dirichlet(0.5) sizes), K=7168, N=4096:
    forward and input gradient on sampled rows, weight gradient of the three
    smallest non-empty experts in full, of the two largest on sampled rows
    (their contractions run over 4415 and 4740 rows: the most k-blocks and
    stage-ring wraps of the launch), and the empty ones exactly zero."""
    E, T, K, N = 32, 32768, 7168, 4096
    off, x, w, dy = mxq_inputs.moe_inputs(E, T, K, N, seed=0)
    moe = MoE(mxq, off, x, w, dy)
    y, dx, dw = moe.fwd(), moe.dx(), moe.dw()
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    # the per-group padded row scales give the same forward and dX bit for bit
    pm = MoE(mxq, off, x, w, dy, padded=True)
    assert torch.equal(pm.fwd().view(torch.int16), y.view(torch.int16))
    assert torch.equal(pm.dx().view(torch.int16), dx.view(torch.int16))
    del pm
    n = np.diff(off)
    rng = np.random.default_rng(0)
    # six non-empty experts (the oracle re-quantizes each one's full weight):
    # their first and last rows plus random rows inside them
    experts = rng.choice(np.nonzero(n > 0)[0], 6, replace=False)
    picks = []
    for e in experts:
        r0, r1 = int(off[e]), int(off[e + 1])
        picks += [r0, r1 - 1] + list(rng.integers(r0, r1, size=6))
    rows = np.unique(np.array(picks, dtype=np.int64))
    expert_of = np.searchsorted(off, rows, side="right") - 1
    qx, sx = oracle.mxfp8_quant_rows(x[torch.from_numpy(rows)])
    qdy, sdy = oracle.mxfp8_quant_rows(dy[torch.from_numpy(rows)])
    ref_y = np.zeros((len(rows), N))
    ref_dx = np.zeros((len(rows), K))
    for e in np.unique(expert_of):
        sel = expert_of == e
        qw, sw = oracle.mxfp8_quant_rows(w[e])
        qwT, swT = oracle.mxfp8_quant_cols(w[e])
        ref_y[sel] = oracle.gemm_ref(qx[sel], sx[sel], qw, sw)
        ref_dx[sel] = oracle.gemm_ref(qdy[sel], sdy[sel], qwT, swT)
    idx = torch.from_numpy(rows).to(DEV)
    check_close(y[idx], ref_y)
    check_close(dx[idx], ref_dx)
    nonempty = [e for e in np.argsort(n) if n[e] > 0][:3]
    for e in nonempty:
        r0, r1 = off[e], off[e + 1]
        a, sa = oracle.mxfp8_quant_cols(dy[r0:r1])
        b, sb = oracle.mxfp8_quant_cols(x[r0:r1])
        check_close(dw[e], oracle.gemm_ref(a, sa, b, sb))
    for e in np.argsort(n)[-2:]:
        r0, r1 = int(off[e]), int(off[e + 1])
        a, sa = oracle.mxfp8_quant_cols(dy[r0:r1])
        b, sb = oracle.mxfp8_quant_cols(x[r0:r1])
        rows_n = np.unique(np.concatenate([rng.choice(N, 46, replace=False), [0, N - 1]]))
        check_close(dw[int(e)][torch.from_numpy(rows_n).to(DEV)], oracle.gemm_ref(a[rows_n], sa[rows_n], b, sb))
    for e in np.nonzero(n == 0)[0]:
        assert not torch.any(dw[int(e)].float() != 0)


def test_grouped_many_experts_decode_without_tables(mxq):
    """300 experts: more than the kernel keeps in its shared-memory group tables,
    so tiles are decoded from the device offsets (and the per-group column
    quant scans 300 groups)."""
    E, T, K, N = 300, 1200, 64, 128
    sizes = mxq_inputs.dirichlet_group_sizes(E, T, alpha=0.5, seed=3)
    assert (sizes == 0).any() and (sizes > 0).sum() > 100
    off, x, w, dy = mxq_inputs.moe_inputs(E, T, K, N, seed=5, sizes=sizes)
    moe = MoE(mxq, off, x, w, dy)
    y, dx, dw = moe.fwd(), moe.dx(), moe.dw()
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    qx, sx = oracle.mxfp8_quant_rows(x)
    qw, sw, qwT, swT = _oracle_w(w)
    qdy, sdy = oracle.mxfp8_quant_rows(dy)
    check_close(y, oracle.grouped_fwd_ref(qx, sx, qw, sw, off))
    check_close(dx, oracle.grouped_fwd_ref(qdy, sdy, qwT, swT, off))
    qdyT, sdyT = oracle.mxfp8_quant_cols_grouped(dy, off)
    qxT, sxT = oracle.mxfp8_quant_cols_grouped(x, off)
    ref_dw = oracle.grouped_dw_ref(qdyT, sdyT, qxT, sxT, off)
    got_dw = dw.float().cpu().numpy()
    for e in range(E):
        if sizes[e] == 0:
            assert not np.any(got_dw[e])
        else:
            check_close(dw[e], ref_dw[e])


@pytest.mark.parametrize("sizes,K,N", [([3, 0, 200, 0, 97], 256, 256), ([128, 128], 160, 384), ([0, 0, 1], 1024, 1024),
                                       ([129, 127, 0, 3, 255, 1], 224, 256), ([1] * 40, 64, 128)])
def test_grouped_padded_row_scales(mxq, sizes, K, N):
    """Forward and dX from the per-group padded row scales (tiles start at
    each group's first row): bit for bit the result of the matrix-aligned row
    tiles, and within tolerance of the oracle; the weight gradient from the
    same padded quant's column outputs likewise."""
    off, x, w, dy = mxq_inputs.moe_inputs(len(sizes), sum(sizes), K, N, seed=len(sizes) + K + 7, sizes=sizes)
    ref, pad = MoE(mxq, off, x, w, dy), MoE(mxq, off, x, w, dy, padded=True)
    y, dx, dw = pad.fwd(), pad.dx(), pad.dw()
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    assert torch.equal(y.view(torch.int16), ref.fwd().view(torch.int16))
    assert torch.equal(dx.view(torch.int16), ref.dx().view(torch.int16))
    assert torch.equal(dw.view(torch.int16), ref.dw().view(torch.int16))
    qx, sx = oracle.mxfp8_quant_rows(x)
    qw, sw, qwT, swT = _oracle_w(w)
    qdy, sdy = oracle.mxfp8_quant_rows(dy)
    check_close(y, oracle.grouped_fwd_ref(qx, sx, qw, sw, off))
    check_close(dx, oracle.grouped_fwd_ref(qdy, sdy, qwT, swT, off))


def test_grouped_padded_row_scales_many_experts(mxq):
    """300 experts (tiles decoded from the device offsets, no shared-memory
    tables): padded and matrix-aligned row tiles agree bit for bit."""
    E, T, K, N = 300, 1200, 64, 128
    sizes = mxq_inputs.dirichlet_group_sizes(E, T, alpha=0.5, seed=3)
    off, x, w, dy = mxq_inputs.moe_inputs(E, T, K, N, seed=5, sizes=sizes)
    ref, pad = MoE(mxq, off, x, w, dy), MoE(mxq, off, x, w, dy, padded=True)
    assert torch.equal(pad.fwd().view(torch.int16), ref.fwd().view(torch.int16))
    assert torch.equal(pad.dx().view(torch.int16), ref.dx().view(torch.int16))
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
