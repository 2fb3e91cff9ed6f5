"""The end-to-end measurement computes the real step: the outputs that the
pipelined host-buffer steps copy back (both device slots, both copy streams)
equal, bit for bit, those of one step on the device-resident inputs."""
import os
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_pipelined_host_steps_match_the_device_step(mxq):
    import bench
    dev = torch.device("cuda", 0)
    wl = bench.Workload(dev, mxq.SAVE_QUANT, bench.make_host_inputs())
    wl.step()
    torch.cuda.synchronize()
    ref = {k: getattr(wl, k).cpu() for k in bench.E2EPipeline.OUT}
    e2e = bench.E2EPipeline(wl)
    for k in bench.E2EPipeline.OUT:  # the host result buffers start out different
        for h in e2e.h_out:
            h[k].zero_()
    for _ in range(4):  # two steps per device slot
        e2e.step()
    torch.cuda.synchronize()
    e2e.restore()
    for slot in range(2):
        for k, r in ref.items():
            got = e2e.h_out[slot][k]
            assert got.shape == r.shape and got.dtype == r.dtype, k
            assert torch.equal(got.view(torch.uint8), r.view(torch.uint8)), (slot, k)
