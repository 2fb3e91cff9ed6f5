"""Malformed group offsets are caught on the device.

Every grouped kernel checks off[0..E] (off[0] = 0, non-decreasing, off[E] = T)
before it does anything that depends on an offset; a malformed array makes it
skip all of its work and set the bad-offsets bit that mxq_poll_device_error
reports as MXQ_ERR_INVALID_ARG.  Offsets feed the experts' grouped matmul
("低精度训练特性（MXFP8 / HiFloat8）", section "MoE 专家层低精度").

The arrays given to the grouped kernels here keep every row inside the
buffers even if the check were missing (decreasing offsets give empty groups,
and a wrong start or end stays within [0, T]), so no run can touch memory
outside them.  Arrays with negative or out-of-range offsets go only to the
stand-alone checker, which reads the offsets and nothing else."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"
E, T, K, N = 4, 300, 64, 128
BAD_IN_BOUNDS = {
    "decreasing": [0, 200, 100, 300, 300],
    "start not 0": [10, 50, 100, 300, 300],
    "end below T": [0, 50, 100, 200, 250],
}
GOOD = [0, 10, 10, 290, 300]


def _dev(off):
    return torch.tensor(off, dtype=torch.int64, device=DEV)


def _expect_bad(mxq):
    w = mxq.mxq_poll_device_error()
    assert w & 4, f"bad-offsets bit not set (error word {w:#x})"
    assert mxq.mxq_poll_device_error() == 0, "the error word is cleared by the poll"


def test_checker_flags_every_kind_of_malformed_offsets(mxq):
    bad = dict(BAD_IN_BOUNDS)
    bad["negative"] = [0, -8, 10, 300, 300]
    bad["past T"] = [0, 10, 400, 500, 300]
    bad["all past T"] = [0, 1 << 40, 1 << 41, 1 << 42, 300]
    for what, off in bad.items():
        mxq.mxq_check_group_offsets(_dev(off), E, T)
        torch.cuda.synchronize()
        w = mxq.mxq_poll_device_error()
        assert w == 4, (what, w)
    for off, t in ((GOOD, T), ([0, 0, 0, 0, 0], 0), ([0, 300, 300, 300, 300], 300)):
        mxq.mxq_check_group_offsets(_dev(off), E, t)
        assert mxq.mxq_poll_device_error() == 0, off
    # the status the C poll returns for the bit
    mxq.mxq_check_group_offsets(_dev(BAD_IN_BOUNDS["decreasing"]), E, T)
    torch.cuda.synchronize()
    with pytest.raises(mxq.MXQError) as err:
        mxq._check(mxq.load().mxq_poll_device_error(None), "poll")
    assert err.value.status == 1 and "group offsets" in str(err.value)


def _sentinel(n):
    return torch.full((n,), 0xA5, dtype=torch.uint8, device=DEV)


def test_grouped_kernels_skip_all_work_on_malformed_offsets(mxq):
    x = torch.randn(T, K, device=DEV).to(torch.bfloat16)
    t_pad = mxq.mxq_grouped_padded_rows(T, E)
    q = _sentinel(T * K)
    s = _sentinel(mxq.mxq_scale_bytes(T, K // 32))
    qT = _sentinel(K * t_pad)
    sT = _sentinel(mxq.mxq_scale_bytes(K, t_pad // 32))
    # GEMM operands (contents do not matter: nothing is computed)
    a = torch.zeros(T * N, dtype=torch.uint8, device=DEV)
    sa = torch.zeros(mxq.mxq_scale_bytes(T, N // 32), dtype=torch.uint8, device=DEV)
    wq = torch.zeros(E * N * K, dtype=torch.uint8, device=DEV)
    ws = torch.zeros(mxq.mxq_scale_bytes(E * N, K // 32), dtype=torch.uint8, device=DEV)
    aT = torch.zeros(N * t_pad, dtype=torch.uint8, device=DEV)
    saT = torch.zeros(mxq.mxq_scale_bytes(N, t_pad // 32), dtype=torch.uint8, device=DEV)
    bT = torch.zeros(K * t_pad, dtype=torch.uint8, device=DEV)
    sbT = torch.zeros(mxq.mxq_scale_bytes(K, t_pad // 32), dtype=torch.uint8, device=DEV)
    wqT = torch.zeros(K * E * N, dtype=torch.uint8, device=DEV)
    wsT = torch.zeros(mxq.mxq_scale_bytes(K, E * N // 32), dtype=torch.uint8, device=DEV)
    xq = torch.zeros(T * K, dtype=torch.uint8, device=DEV)
    xs = torch.zeros(mxq.mxq_scale_bytes(T, K // 32), dtype=torch.uint8, device=DEV)
    y = _sentinel(T * N * 2)
    dx = _sentinel(T * K * 2)
    dw = _sentinel(E * N * K * 2)
    for what, off in BAD_IN_BOUNDS.items():
        d = _dev(off)
        mxq.mxq_quantize_grouped_dual(x, T, K, d, E, t_pad, q, s, qT, sT)
        torch.cuda.synchronize()
        _expect_bad(mxq)
        mxq.mxq_quantize_grouped_col(x, T, K, d, E, t_pad, qT, sT)
        torch.cuda.synchronize()
        _expect_bad(mxq)
        mxq.mxq_grouped_gemm(mxq.GG_FWD, xq, xs, wq, ws, d, E, T, N, K, 0, y)
        torch.cuda.synchronize()
        _expect_bad(mxq)
        mxq.mxq_grouped_gemm(mxq.GG_DX, a, sa, wqT, wsT, d, E, T, N, K, 0, dx)
        torch.cuda.synchronize()
        _expect_bad(mxq)
        mxq.mxq_grouped_gemm(mxq.GG_DW, aT, saT, bT, sbT, d, E, T, N, K, t_pad, dw)
        torch.cuda.synchronize()
        _expect_bad(mxq)
        for name, buf in (("q_row", q), ("s_row", s), ("q_colT", qT), ("s_colT", sT), ("fwd", y), ("dx", dx),
                          ("dw", dw)):
            assert bool((buf == 0xA5).all()), f"{what}: {name} was written"
    # well-formed offsets afterwards: the kernels run and report nothing
    d = _dev(GOOD)
    mxq.mxq_quantize_grouped_dual(x, T, K, d, E, t_pad, q, s, qT, sT)
    mxq.mxq_grouped_gemm(mxq.GG_FWD, xq, xs, wq, ws, d, E, T, N, K, 0, y)
    mxq.mxq_grouped_gemm(mxq.GG_DW, aT, saT, bT, sbT, d, E, T, N, K, t_pad, dw)
    assert mxq.mxq_poll_device_error() == 0
    assert not bool((q == 0xA5).all())
    assert bool((y.view(torch.bfloat16) == 0).all())           # zero operands give zero outputs
    assert bool((dw.view(torch.bfloat16) == 0).all())
