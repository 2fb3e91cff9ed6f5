"""Failure detection without a GPU fault: every wait in the library's kernels is
bounded; a wait that runs out sets a device error word that the host reads
(mxq_poll_device_error) while the context stays usable.  The self-test kernel
waits on an mbarrier that nothing arrives on, so its wait runs out."""
import time

import numpy as np
import pytest
import torch

import oracle
from test_gpu_gemm import _bf16_rne, _exact_operands

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _exact_gemm(mxq, c):
    rng = np.random.default_rng(7)
    qa, la = _exact_operands(256, 512, rng)
    qb, lb = _exact_operands(384, 512, rng)
    mxq.mxq_gemm(torch.from_numpy(qa).to(DEV), torch.from_numpy(oracle.swizzle_scales(la)).to(DEV),
                 torch.from_numpy(qb).to(DEV), torch.from_numpy(oracle.swizzle_scales(lb)).to(DEV),
                 256, 384, 512, c, 384)
    torch.cuda.synchronize()
    return _bf16_rne(oracle.gemm_ref(qa, la, qb, lb))


def _time_out(mxq, ms=50):
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    mxq.mxq_selftest_wait_timeout(ms, flag)
    torch.cuda.synchronize()
    return flag.item(), time.perf_counter() - t0


def test_wait_runs_out_and_is_reported(mxq):
    assert mxq.mxq_poll_device_error() == 0
    gave_up, dt = _time_out(mxq, 50)
    assert gave_up == 1
    assert 0.045 <= dt < 5.0, dt
    assert mxq.mxq_poll_device_error() == 1  # bit 0: a wait timed out
    assert mxq.mxq_poll_device_error() == 0  # reading clears it


def test_context_stays_usable_and_pending_error_stops_gemms(mxq):
    assert mxq.mxq_poll_device_error() == 0
    assert _time_out(mxq, 20)[0] == 1
    # while the error is pending, GEMM launches skip their tiles: C keeps its fill
    c = torch.full((256, 384), float("nan"), dtype=torch.bfloat16, device=DEV)
    _exact_gemm(mxq, c)
    assert torch.isnan(c.float()).all()
    assert mxq.mxq_poll_device_error() == 1
    # once read and cleared, the same context computes again, bit for bit
    c = torch.full((256, 384), float("nan"), dtype=torch.bfloat16, device=DEV)
    ref = _exact_gemm(mxq, c)
    assert np.array_equal(c.cpu().view(torch.int16).numpy(), ref)
    assert mxq.mxq_poll_device_error() == 0
