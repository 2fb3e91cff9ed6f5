"""GPU parity of the quantization kernels against the CPU oracle: codes and
scales must be bit-identical (every byte of the padded scale buffers too)."""
import numpy as np
import pytest
import torch

import mxq_inputs
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(R, C, kind, seed):
    if kind == "normal":
        return mxq_inputs.normal_bf16((R, C), 1.0, seed=seed)
    x = mxq_inputs.sweep_bf16(R, C, seed=seed)            # heavy tail, 1000x outliers
    if R >= 4 and C >= 64:
        x[1, :32] = 0                                      # an all-zero row block
        x[2, 32:64] = -0.0                                 # negative zeros
        x[:32, 3] = 0                                      # an all-zero column block
        x[0, 0] = 3.0e38                                   # near the bf16 maximum
        x[3, 5] = 1e-40                                    # a bf16 subnormal
    return x


ROW_SHAPES = [(256, 512), (512, 512), (100, 96), (1, 32), (129, 160), (384, 4096), (128, 128)]


@pytest.mark.parametrize("R,C", ROW_SHAPES)
@pytest.mark.parametrize("kind", ["normal", "heavy"])
def test_row_quant_bit_exact(mxq, R, C, kind):
    x = _inputs(R, C, kind, seed=R + C)
    q, s, _, _ = mxq.quantize_mxfp8(x.to(DEV), axis=-1)
    oq, os_ = oracle.mxfp8_quant_rows(x)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))


# (80, 256) and (144, 96): a transposed-code row pitch that is a multiple of 16
# bytes but not of 32 (the 16-byte store path of the column pass)
COL_SHAPES = [(256, 512), (96, 64), (100, 64), (130, 136), (33, 8), (1, 32), (4096, 384), (200, 1024), (80, 256),
              (144, 96)]


@pytest.mark.parametrize("R,C", COL_SHAPES)
@pytest.mark.parametrize("dual", [False, True])
def test_col_and_dual_quant_bit_exact(mxq, R, C, dual):
    if dual and C % 32:
        pytest.skip("row axis needs cols % 32 == 0")
    x = _inputs(R, C, "heavy", seed=3 * R + C)
    q, s, qT, sT = mxq.quantize_mxfp8(x.to(DEV), axis=-2, dual=dual)
    oqT, osT = oracle.mxfp8_quant_cols(x)
    assert np.array_equal(qT.cpu().numpy(), oqT)
    assert np.array_equal(sT.cpu().numpy(), oracle.swizzle_scales(osT))
    if dual:
        oq, os_ = oracle.mxfp8_quant_rows(x)
        assert np.array_equal(q.cpu().numpy(), oq)
        assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))


def _grouped(mxq, x, off):
    T, C = x.shape
    E = len(off) - 1
    t_pad = mxq.mxq_grouped_padded_rows(T, E)
    qT = torch.full((C, t_pad), 0xAB, dtype=torch.uint8, device=DEV)     # poison: every byte must be written
    sT = torch.full((mxq.mxq_scale_bytes(C, t_pad // 32),), 0xAB, dtype=torch.uint8, device=DEV)
    d_off = torch.from_numpy(off).to(DEV)
    mxq.mxq_quantize_grouped_col(x.to(DEV), T, C, d_off, E, t_pad, qT, sT)
    return qT.cpu().numpy(), sT.cpu().numpy(), t_pad


@pytest.mark.parametrize("sizes", [[0, 5, 128, 33, 0, 200, 1], [300], [0, 0, 64], [1] * 40])
def test_grouped_col_quant_bit_exact(mxq, sizes):
    off = mxq_inputs.offsets_from_sizes(sizes)
    x = _inputs(int(off[-1]), 136, "heavy", seed=len(sizes))
    qT, sT, t_pad = _grouped(mxq, x, off)
    oqT, osT = oracle.mxfp8_quant_cols_grouped(x, off, t_pad)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(sT, oracle.swizzle_scales(osT))


def test_grouped_col_quant_dirichlet(mxq):
    n = mxq_inputs.dirichlet_group_sizes(32, 4096, 0.5, seed=0)
    assert (n == 0).any() or n.min() < 40         # the recipe gives tiny / empty groups
    off = mxq_inputs.offsets_from_sizes(n)
    x = mxq_inputs.normal_bf16((4096, 512), 1e-3, seed=2)
    qT, sT, t_pad = _grouped(mxq, x, off)
    oqT, osT = oracle.mxfp8_quant_cols_grouped(x, off, t_pad)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(sT, oracle.swizzle_scales(osT))


# ------------------------------------------------------------------ MXFP4

def _read_shapes():
    import os
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "mxfp4_ragged_shapes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(tuple(int(v) for v in line.split()))
    return rows


@pytest.mark.parametrize("shape", _read_shapes() + [(5, 64), (7, 1), (3, 95)])
@pytest.mark.parametrize("sf", [6.0, 4.0, 6.0 / 1.3])
def test_qdq_mxfp4_ragged_bit_exact(mxq, shape, sf):
    a = mxq_inputs.mxfp4_small(shape, seed=sum(shape))
    got = mxq.qdq_mxfp4(torch.from_numpy(a).to(DEV), np.float32(sf)).cpu().numpy()
    ref = oracle.mxfp4_qdq(a, np.float32(sf))
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_qdq_mxfp4_large_bit_exact(mxq):
    a = mxq_inputs.mxfp4_large(4096, 4096, seed=0)   # t(3) tails, x100 outliers, zero blocks
    got = mxq.qdq_mxfp4(torch.from_numpy(a).to(DEV)).cpu().numpy()
    ref = oracle.mxfp4_qdq(a)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_qdq_mxfp4_in_place(mxq):
    a = mxq_inputs.mxfp4_small((64, 96), seed=9)
    t = torch.from_numpy(a).to(DEV)
    mxq.mxq_qdq_mxfp4(t, t, 64, 96, 32, 6.0)
    assert np.array_equal(t.cpu().numpy().view(np.uint32), oracle.mxfp4_qdq(a).view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("R,C", [(48, 160), (128, 128), (300, 4096), (512, 4096), (4096, 4096)])
def test_packed_mxfp4_bit_exact(mxq, dtype, R, C):
    a = mxq_inputs.mxfp4_large(R, C, seed=R)
    t = torch.from_numpy(a).to(dtype)
    q, s = mxq.quantize_mxfp4(t.to(DEV))
    oq, os_ = oracle.mxfp4_quant(t.to(torch.float32).numpy())
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))


def _f32_at16(a: np.ndarray) -> torch.Tensor:
    """a copy of `a` on the GPU whose data starts 16 bytes past a 32-byte boundary"""
    buf = torch.empty(a.size + 12, dtype=torch.float32, device=DEV)
    o = ((-buf.data_ptr()) % 32 + 16) // 4
    t = buf[o:o + a.size].view(a.shape)
    t.copy_(torch.from_numpy(a))
    assert t.data_ptr() % 32 == 16
    return t


def test_fp32_vector_paths_16_but_not_32_byte_aligned(mxq):
    """fp32 MXFP4 QDQ, clipped-STE forward/backward and packed quant on
    buffers 16 bytes past a 32-byte boundary take the 16-byte access path;
    results unchanged."""
    R, C = 64, 256
    a = mxq_inputs.mxfp4_large(R, C, seed=21)
    x = _f32_at16(a)
    y = _f32_at16(np.zeros_like(a))
    mxq.mxq_qdq_mxfp4(x, y, R, C, 32, 6.0)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), oracle.mxfp4_qdq(a).view(np.uint32))
    m = torch.empty((R, C // 32), dtype=torch.int32, device=DEV)
    mxq.mxq_mxfp4_ste_forward(x, y, m, R, C, 32, 6.0)
    ref_m = oracle.mxfp4_saturation_mask(a)
    assert np.array_equal(m.cpu().numpy().view(np.uint32), ref_m)
    gy = mxq_inputs.mxfp4_small((R, C), seed=22)
    g = _f32_at16(gy)
    gx = _f32_at16(np.zeros_like(gy))
    mxq.mxq_mxfp4_ste_backward(g, m, R, C, gx)
    assert np.array_equal(gx.cpu().numpy().view(np.uint32), oracle.mxfp4_ste_backward(gy, ref_m).view(np.uint32))
    q, s = mxq.quantize_mxfp4(x)
    oq, os_ = oracle.mxfp4_quant(a)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))


# ------------------------------------------------------------------ full sizes

def test_full_size_linear_operands_dual_quant(mxq):
    """X[8192x4096], W[14336x4096], dY[8192x14336]: dual quant bit-exact in full."""
    x, w, dy = mxq_inputs.linear_inputs(8192, 14336, 4096, seed=0)
    for t in (x, w, dy):
        q, s, qT, sT = mxq.quantize_mxfp8(t.to(DEV), dual=True)
        oq, os_ = oracle.mxfp8_quant_rows(t)
        assert np.array_equal(q.cpu().numpy(), oq)
        assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))
        oqT, osT = oracle.mxfp8_quant_cols(t)
        assert np.array_equal(qT.cpu().numpy(), oqT)
        assert np.array_equal(sT.cpu().numpy(), oracle.swizzle_scales(osT))
        del q, s, qT, sT


def _sweep_rows(C, p):
    """The bandwidth sweep's row count for 2^p elements of width C."""
    return ((1 << p) // C + 127) // 128 * 128


@pytest.mark.parametrize("C", [2048, 7168, 14336])
@pytest.mark.parametrize("p", [22, 24])
def test_sweep_shapes_dual_quant_bit_exact(mxq, C, p):
    """The dual-quant sweep's shapes up to 2^24 elements, heavy-tailed with
    1000x outliers: all four outputs in full against the oracle."""
    x = mxq_inputs.sweep_bf16(_sweep_rows(C, p), C, seed=p * C)
    q, s, qT, sT = mxq.quantize_mxfp8(x.to(DEV), dual=True)
    oq, os_ = oracle.mxfp8_quant_rows(x)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))
    oqT, osT = oracle.mxfp8_quant_cols(x)
    assert np.array_equal(qT.cpu().numpy(), oqT)
    assert np.array_equal(sT.cpu().numpy(), oracle.swizzle_scales(osT))


@pytest.mark.parametrize("C", [2048, 7168, 14336])
def test_sweep_largest_size_dual_quant_sampled(mxq, C):
    """The sweep's largest size, 2^30 elements drawn on the device as the
    sweep draws them: three 128-row slabs of the row outputs and two
    128-column slabs of the column outputs (every block of those columns)
    against the oracle, scale tiles included (a slab of 128 rows or columns
    starting at a multiple of 128 is one row of 512-byte scale tiles)."""
    R = _sweep_rows(C, 30)
    x = mxq_inputs.sweep_bf16_device(R, C, seed=C, device=DEV)
    q, s, qT, sT = mxq.quantize_mxfp8(x, dual=True)
    torch.cuda.synchronize()
    kp = (C // 32 + 3) // 4 * 4                    # row-scale tile columns x 4
    for r0 in (0, (R // 256) * 128, R - 128):
        xs = x[r0:r0 + 128].cpu()
        oq, os_ = oracle.mxfp8_quant_rows(xs)
        assert np.array_equal(q[r0:r0 + 128].cpu().numpy(), oq), r0
        tiles = s[r0 * kp:(r0 + 128) * kp].cpu().numpy()
        assert np.array_equal(tiles, oracle.swizzle_scales(os_)), r0
    kpT = (R // 32 + 3) // 4 * 4
    for c0 in (0, C - 128):
        xs = x[:, c0:c0 + 128].contiguous().cpu()
        oqT, osT = oracle.mxfp8_quant_cols(xs)
        assert np.array_equal(qT[c0:c0 + 128].cpu().numpy(), oqT), c0
        tiles = sT[c0 * kpT:(c0 + 128) * kpT].cpu().numpy()
        assert np.array_equal(tiles, oracle.swizzle_scales(osT)), c0


@pytest.mark.parametrize("R,C,pad,shift", [(256, 64, 8, 0), (130, 96, 16, 8), (64, 128, 8, 24)])
def test_dual_quant_strided_views(mxq, R, C, pad, shift):
    """A row stride larger than the row (ldx = C + pad + shift elements) and a
    base 16-byte aligned but not tile aligned (shift elements in): the staged
    tiles follow the stride, so codes and scales are those of the contiguous
    tensor."""
    x = _inputs(R, C, "heavy", seed=R + C + pad)
    wide = torch.zeros((R, C + pad + shift), dtype=torch.bfloat16)
    wide[:, shift:shift + C] = x
    view = wide.to(DEV)[:, shift:shift + C]
    assert view.stride(0) == C + pad + shift
    q, s, qT, sT = mxq.quantize_mxfp8(view, dual=True)
    oq, os_ = oracle.mxfp8_quant_rows(x)
    oqT, osT = oracle.mxfp8_quant_cols(x)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))
    assert np.array_equal(qT.cpu().numpy(), oqT)
    assert np.array_equal(sT.cpu().numpy(), oracle.swizzle_scales(osT))


@pytest.mark.parametrize("grouped", [False, True])
def test_dual_quant_outputs_16_but_not_32_byte_aligned(mxq, grouped):
    """Output buffers that start 16 bytes past a 32-byte boundary take the
    16-byte store path; codes and scales are unchanged."""
    R, C = 384, 256
    x = _inputs(R, C, "heavy", seed=9)
    off = mxq_inputs.offsets_from_sizes([100, 0, 284])
    t_pad = mxq.mxq_grouped_padded_rows(R, 3) if grouped else R
    def at16(n):  # a buffer of n bytes at 16 mod 32
        buf = torch.full((n + 48,), 0xAB, dtype=torch.uint8, device=DEV)
        o = (-buf.data_ptr()) % 32 + 16
        return buf[o:o + n]
    q, s = at16(R * C), at16(mxq.mxq_scale_bytes(R, C // 32))
    qT, sT = at16(C * t_pad), at16(mxq.mxq_scale_bytes(C, t_pad // 32))
    assert q.data_ptr() % 32 == 16 and qT.data_ptr() % 32 == 16
    xd = x.to(DEV)
    if grouped:
        mxq.mxq_quantize_grouped_dual(xd, R, C, torch.from_numpy(off).to(DEV), 3, t_pad, q, s, qT, sT)
        oqT, osT = oracle.mxfp8_quant_cols_grouped(x, off, t_pad)
    else:
        mxq.mxq_quantize(xd, mxq.BF16, R, C, C, -1, mxq.E4M3, 1, q, s, qT, sT)
        oqT, osT = oracle.mxfp8_quant_cols(x)
    oq, os_ = oracle.mxfp8_quant_rows(x)
    assert np.array_equal(q.cpu().numpy().reshape(R, C), oq)
    assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))
    assert np.array_equal(qT.cpu().numpy().reshape(C, t_pad), oqT)
    assert np.array_equal(sT.cpu().numpy(), oracle.swizzle_scales(osT))


def _grouped_dual(mxq, x, off):
    T, C = x.shape
    E = len(off) - 1
    t_pad = mxq.mxq_grouped_padded_rows(T, E)
    poison = lambda *shape: torch.full(shape, 0xAB, dtype=torch.uint8, device=DEV)  # noqa: E731
    q, s = poison(max(T, 1), C), poison(mxq.mxq_scale_bytes(T, C // 32))
    qT, sT = poison(C, t_pad), poison(mxq.mxq_scale_bytes(C, t_pad // 32))
    mxq.mxq_quantize_grouped_dual(x.to(DEV), T, C, torch.from_numpy(off).to(DEV), E, t_pad, q, s, qT, sT)
    return q.cpu().numpy()[:T], s.cpu().numpy(), qT.cpu().numpy(), sT.cpu().numpy(), t_pad


@pytest.mark.parametrize("sizes", [[0, 5, 128, 33, 0, 200, 1], [300], [0, 0, 64], [1] * 40, [129, 127, 0, 3]])
@pytest.mark.parametrize("C", [160, 256])
def test_grouped_dual_quant_bit_exact(mxq, sizes, C):
    """Row quant and per-group column quant from one read: both equal the
    oracle's separate quants byte for byte, padding included (outputs are
    poisoned first; rows past T in the last row-scale tile must read 0)."""
    off = mxq_inputs.offsets_from_sizes(sizes)
    x = _inputs(int(off[-1]), C, "heavy", seed=len(sizes) + C)
    q, s, qT, sT, t_pad = _grouped_dual(mxq, x, off)
    oq, os_ = oracle.mxfp8_quant_rows(x)
    assert np.array_equal(q, oq)
    assert np.array_equal(s, oracle.swizzle_scales(os_))
    oqT, osT = oracle.mxfp8_quant_cols_grouped(x, off, t_pad)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(sT, oracle.swizzle_scales(osT))


def test_grouped_dual_quant_300_groups(mxq):
    """More groups than the kernel keeps in shared-memory tables (256): the
    per-tile group lookup scans the offsets in global memory instead."""
    sizes = np.random.default_rng(300).integers(0, 40, size=300)
    off = mxq_inputs.offsets_from_sizes(sizes)
    x = _inputs(int(off[-1]), 64, "heavy", seed=300)
    q, s, qT, sT, t_pad = _grouped_dual(mxq, x, off)
    oq, os_ = oracle.mxfp8_quant_rows(x)
    assert np.array_equal(q, oq)
    assert np.array_equal(s, oracle.swizzle_scales(os_))
    oqT, osT = oracle.mxfp8_quant_cols_grouped(x, off, t_pad)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(sT, oracle.swizzle_scales(osT))


def _grouped_dual_padded(mxq, x, off):
    T, C = x.shape
    E = len(off) - 1
    t_pad = mxq.mxq_grouped_padded_rows(T, E)
    poison = lambda *shape: torch.full(shape, 0xAB, dtype=torch.uint8, device=DEV)  # noqa: E731
    q, s = poison(max(T, 1), C), poison(mxq.mxq_scale_bytes(t_pad, C // 32))
    qT, sT = poison(C, t_pad), poison(mxq.mxq_scale_bytes(C, t_pad // 32))
    mxq.mxq_quantize_grouped_dual_padded(x.to(DEV), T, C, torch.from_numpy(off).to(DEV), E, t_pad, q, s, qT, sT)
    return q.cpu().numpy()[:T], s.cpu().numpy(), qT.cpu().numpy(), sT.cpu().numpy(), t_pad


def _padded_row_scales(os_, off, t_pad):
    """The oracle's row scales laid out per group: group e's rows from padded
    row P_e = sum of ceil128 of the earlier groups' lengths, zeros elsewhere."""
    L = np.zeros((t_pad, os_.shape[1]), np.uint8)
    p = 0
    for e in range(len(off) - 1):
        n = int(off[e + 1] - off[e])
        L[p:p + n] = os_[int(off[e]):int(off[e + 1])]
        p += (n + 127) // 128 * 128
    return oracle.swizzle_scales(L)


@pytest.mark.parametrize("sizes", [[0, 5, 128, 33, 0, 200, 1], [300], [0, 0, 64], [1] * 40, [129, 127, 0, 3],
                                   [0, 0]])
@pytest.mark.parametrize("C", [160, 256])
def test_grouped_dual_quant_padded_row_scales(mxq, sizes, C):
    """The per-group padded row-scale layout: row codes as the plain row
    quant, row scales placed per group (every padding byte zero, outputs
    poisoned first), column outputs as the per-group column quant."""
    off = mxq_inputs.offsets_from_sizes(sizes)
    T = int(off[-1])
    x = _inputs(T, C, "heavy", seed=len(sizes) + C + 1) if T else torch.zeros((0, C), dtype=torch.bfloat16)
    q, s, qT, sT, t_pad = _grouped_dual_padded(mxq, x, off)
    oq, os_ = oracle.mxfp8_quant_rows(x) if T else (np.zeros((0, C), np.uint8), np.zeros((0, C // 32), np.uint8))
    assert np.array_equal(q, oq)
    assert np.array_equal(s, _padded_row_scales(os_, off, t_pad))
    oqT, osT = oracle.mxfp8_quant_cols_grouped(x, off, t_pad)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(sT, oracle.swizzle_scales(osT))


def test_grouped_dual_quant_full_size_moe_dy(mxq):
    """The MoE layer's dY, 32768 x 4096 bf16 in 32 Dirichlet(0.5) groups: every
    byte of the four outputs against the oracle."""
    E, T, C = 32, 32768, 4096
    off = mxq_inputs.offsets_from_sizes(mxq_inputs.dirichlet_group_sizes(E, T, seed=0))
    x = mxq_inputs.normal_bf16((T, C), 1e-3, seed=5)
    q, s, qT, sT, t_pad = _grouped_dual(mxq, x, off)
    oq, os_ = oracle.mxfp8_quant_rows(x)
    assert np.array_equal(q, oq)
    assert np.array_equal(s, oracle.swizzle_scales(os_))
    oqT, osT = oracle.mxfp8_quant_cols_grouped(x, off, t_pad)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(sT, oracle.swizzle_scales(osT))
    # the per-group padded row scales of the same tensor
    qp, sp, qTp, sTp, _ = _grouped_dual_padded(mxq, x, off)
    assert np.array_equal(qp, oq)
    assert np.array_equal(sp, _padded_row_scales(os_, off, t_pad))
    assert np.array_equal(qTp, oqT) and np.array_equal(sTp, sT)


def test_grouped_dual_quant_without_row_outputs_is_the_column_quant(mxq):
    off = mxq_inputs.offsets_from_sizes([7, 0, 250, 64])
    x = _inputs(int(off[-1]), 96, "heavy", seed=3)
    T, C, E = x.shape[0], x.shape[1], len(off) - 1
    t_pad = mxq.mxq_grouped_padded_rows(T, E)
    qT = torch.full((C, t_pad), 0xAB, dtype=torch.uint8, device=DEV)
    sT = torch.full((mxq.mxq_scale_bytes(C, t_pad // 32),), 0xAB, dtype=torch.uint8, device=DEV)
    mxq.mxq_quantize_grouped_dual(x.to(DEV), T, C, torch.from_numpy(off).to(DEV), E, t_pad, None, None, qT, sT)
    oqT, osT = oracle.mxfp8_quant_cols_grouped(x, off, t_pad)
    assert np.array_equal(qT.cpu().numpy(), oqT)
    assert np.array_equal(sT.cpu().numpy(), oracle.swizzle_scales(osT))


def test_grouped_col_quant_with_no_rows_writes_zero_padding(mxq):
    """Every group empty (T = 0): each byte of the t_pad-wide outputs is padding
    and must be written as 0 (the codes and the E8M0 scale bytes)."""
    E, C = 3, 64
    t_pad = mxq.mxq_grouped_padded_rows(0, E)
    assert t_pad == 128 * E
    d_off = torch.zeros(E + 1, dtype=torch.int64, device=DEV)
    qT = torch.full((C, t_pad), 0xFF, dtype=torch.uint8, device=DEV)
    sT = torch.full((mxq.mxq_scale_bytes(C, t_pad // 32),), 0xFF, dtype=torch.uint8, device=DEV)
    mxq.mxq_quantize_grouped_col(None, 0, C, d_off, E, t_pad, qT, sT)
    torch.cuda.synchronize()
    assert not qT.any() and not sT.any()


def test_every_bf16_pattern_alone_in_a_block(mxq):
    """Each of the 65,536 bf16 bit patterns (zeros, subnormals, normals, Inf,
    NaN) as the only nonzero element of its 32-element block, in both the row
    and the column direction: codes and scales bit for bit."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = np.zeros((65536, 32), dtype=np.uint16)
    x[:, 7] = bits
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    q, s, _, _ = mxq.quantize_mxfp8(xt.to(DEV))
    oq, os_ = oracle.mxfp8_quant_rows(x)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))
    # column direction: the transpose, column j holding pattern j alone
    xc = np.ascontiguousarray(x.T)
    xc_t = torch.from_numpy(xc.view(np.int16)).view(torch.bfloat16)
    _, _, qT, sT = mxq.quantize_mxfp8(xc_t.to(DEV), axis=-2)
    oqT, osT = oracle.mxfp8_quant_cols(xc)
    assert np.array_equal(qT.cpu().numpy(), oqT)
    assert np.array_equal(sT.cpu().numpy(), oracle.swizzle_scales(osT))
