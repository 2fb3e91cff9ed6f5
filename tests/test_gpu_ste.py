"""GPU parity of the clipped straight-through estimator ("AMCT FakeQuant"
article, section 4.1): the forward's quant-dequant output and packed
saturation mask, and the backward's masked gradient, bit for bit against the
oracle."""
import numpy as np
import pytest
import torch

import mxq_inputs
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _forward(mxq, a: np.ndarray, sf: float):
    y, m = mxq.mxfp4_ste_forward(torch.from_numpy(a).to(DEV), float(np.float32(sf)))
    torch.cuda.synchronize()
    return y.cpu().numpy(), m.cpu().numpy().view(np.uint32)


def _check_forward(mxq, a, sf):
    y, m = _forward(mxq, a, sf)
    cols = a.shape[-1]
    assert np.array_equal(y.view(np.uint32), oracle.mxfp4_qdq(a, np.float32(sf)).view(np.uint32))
    assert np.array_equal(m, oracle.mxfp4_saturation_mask(a, np.float32(sf)).reshape(-1, (cols + 31) // 32))
    return m


# ragged shapes use the one-warp-per-block kernel; multiples of 32 the vector one
SHAPES = [(2, 33), (3, 17), (4, 48, 33), (1, 32), (37, 96), (256, 512), (5, 1000), (129, 4128)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("sf", [6.0, 7.0, 12.0, 4.0, 9.0])
def test_forward_bit_exact(mxq, shape, sf):
    a = mxq_inputs.mxfp4_small(shape, seed=sum(shape)) * np.float32(3.0)
    _check_forward(mxq, a, sf)


def test_forward_full_size_heavy_tail(mxq):
    """4096 x 4096 fp32, t(3) tails with x100 outliers and zeroed blocks."""
    a = mxq_inputs.mxfp4_large(4096, 4096, seed=0)
    m = _check_forward(mxq, a, 6.0)
    assert m.any()


def test_forward_unaligned_uses_general_path(mxq):
    """A 4-byte but not 16-byte aligned view takes the per-block kernel."""
    a = mxq_inputs.mxfp4_large(64, 256, seed=4)
    buf = torch.zeros(a.size + 1, dtype=torch.float32, device=DEV)
    x = buf[1:].view(64, 256)
    x.copy_(torch.from_numpy(a))
    y = torch.empty(a.size + 1, dtype=torch.float32, device=DEV)[1:].view(64, 256)
    m = torch.empty((64, 8), dtype=torch.int32, device=DEV)
    mxq.mxq_mxfp4_ste_forward(x, y, m, 64, 256, 32, 6.0)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), oracle.mxfp4_qdq(a).view(np.uint32))
    assert np.array_equal(m.cpu().numpy().view(np.uint32), oracle.mxfp4_saturation_mask(a))


def test_forward_nonfinite_block(mxq):
    a = mxq_inputs.mxfp4_small((4, 64), seed=3) * np.float32(10.0)
    a[1, 5] = np.inf
    a[2, 40] = np.nan
    y, m = _forward(mxq, a, 6.0)
    ref_m = oracle.mxfp4_saturation_mask(a)
    assert np.array_equal(m, ref_m)
    assert ref_m[1, 0] == 0 and ref_m[2, 1] == 0
    assert np.isnan(y[1, :32]).all() and np.isnan(y[2, 32:]).all()


def test_plain_qdq_unchanged_by_mask_output(mxq):
    a = mxq_inputs.mxfp4_large(512, 1024, seed=8)
    y0 = mxq.qdq_mxfp4(torch.from_numpy(a).to(DEV)).cpu().numpy()
    y1, _ = _forward(mxq, a, 6.0)
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))


@pytest.mark.parametrize("shape", [(2, 33), (4, 48, 33), (37, 96), (4096, 4096)])
def test_backward_bit_exact(mxq, shape):
    a = (mxq_inputs.mxfp4_large(int(np.prod(shape[:-1])), shape[-1], seed=6)).reshape(shape)
    gy = mxq_inputs.mxfp4_small(shape, seed=7)
    flat = gy.reshape(-1, shape[-1])
    flat[0, :3] = [np.inf, -0.0, np.nan]
    _, m = _forward(mxq, a, 6.0)
    gx = mxq.mxfp4_ste_backward(torch.from_numpy(gy).to(DEV), torch.from_numpy(m.view(np.int32)).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.mxfp4_ste_backward(gy, oracle.mxfp4_saturation_mask(a))
    assert np.array_equal(gx.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_backward_in_place(mxq):
    a = mxq_inputs.mxfp4_large(64, 128, seed=10)
    gy = mxq_inputs.mxfp4_small((64, 128), seed=11)
    _, m = _forward(mxq, a, 6.0)
    t = torch.from_numpy(gy.copy()).to(DEV)
    mxq.mxq_mxfp4_ste_backward(t, torch.from_numpy(m.view(np.int32)).to(DEV), 64, 128, t)
    torch.cuda.synchronize()
    ref = oracle.mxfp4_ste_backward(gy, oracle.mxfp4_saturation_mask(a))
    assert np.array_equal(t.cpu().numpy().view(np.uint32), ref.view(np.uint32))
