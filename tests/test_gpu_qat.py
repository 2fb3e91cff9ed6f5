"""GPU parity of the MXFP4 QAT linear forward ("AMCT FakeQuant" article,
section 4.3): y = F.linear(Q(x), Q(W), b) against the binary64 oracle.

Tolerance as for the MXFP8 GEMMs (max-rel 1e-2, Frobenius 2e-3 against the
binary64 product of the quant-dequantized operands plus bias); where every
partial sum is exact in fp32 the bf16 result must match bit for bit."""
import numpy as np
import pytest
import torch

import mxq_inputs
import oracle
from test_gpu_gemm import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _rne_bits(ref: np.ndarray) -> np.ndarray:
    return torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy()


def _on_grid(R, K, seed, emin=-2, emax=2):
    """Blocks of codebook values x 2^e, each holding +-6 * 2^e: fixed points of
    the MXFP4 quant-dequant along K."""
    rng = np.random.default_rng(seed)
    book = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    v = rng.choice(book, size=(R, K)) * rng.choice([-1.0, 1.0], size=(R, K))
    v[:, ::32] = 6.0 * rng.choice([-1.0, 1.0], size=(R, K // 32))
    e = rng.integers(emin, emax + 1, size=(R, K // 32))
    return v * np.repeat(np.exp2(e), 32, axis=1)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (96, 352, 96), (256, 512, 256)])
def test_exact_sums_bit_exact(mxq, M, N, K):
    """Operands on the MXFP4 grid with exponents in [-2, 2] and a bias on a
    2^-2 grid: every partial sum is exact in fp32, so y = bf16(exact)."""
    x, w = _on_grid(M, K, 1), _on_grid(N, K, 2)
    b = np.random.default_rng(3).integers(-64, 64, size=N) * 0.25
    y = mxq.qat_linear_fwd(_bf16(x).to(DEV), _bf16(w).to(DEV), _bf16(b).to(DEV))
    ref = oracle.qat_linear_ref(_bf16(x), _bf16(w), _bf16(b))
    assert np.array_equal(ref, x @ w.T + b[None, :])
    assert np.array_equal(y.cpu().view(torch.int16).numpy(), _rne_bits(ref))


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (1024, 768, 1024), (224, 352, 160)])
@pytest.mark.parametrize("sf", [6.0, 7.5])
@pytest.mark.parametrize("with_bias", [False, True])
def test_random_within_tolerance(mxq, M, N, K, sf, with_bias):
    x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=M + N)
    b = _bf16(0.05 * np.random.default_rng(N).standard_normal(N)) if with_bias else None
    y = mxq.qat_linear_fwd(x.to(DEV), w.to(DEV), None if b is None else b.to(DEV), scale_factor=sf)
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    check_close(y, oracle.qat_linear_ref(x, w, b, scale_factor=sf))


def test_full_size_sampled_rows(mxq):
    """8192 x 14336 x 4096 (the dense layer's shape), 64 sampled rows."""
    M, N, K = 8192, 14336, 4096
    x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=0)
    b = _bf16(0.05 * np.random.default_rng(1).standard_normal(N))
    y = mxq.qat_linear_fwd(x.to(DEV), w.to(DEV), b.to(DEV))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.random.default_rng(2).choice(M, 60, replace=False), [0, 127, 128, M - 1]]))
    ref = oracle.qat_linear_ref(x[torch.from_numpy(rows)], w, b)
    check_close(y[torch.from_numpy(rows).to(DEV)], ref)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (96, 352, 512)])
def test_w4a16_exact_sums_bit_exact(mxq, M, N, K):
    """x on a 2^-4 grid (|x| <= 8), W on the MXFP4 grid: every partial sum of
    x Q(W)^T is exact in fp32, so y = bf16(exact)."""
    rng = np.random.default_rng(M + K)
    x = rng.integers(-128, 129, size=(M, K)) / 16.0
    w = _on_grid(N, K, 5)
    y = mxq.qat_linear_fwd(_bf16(x).to(DEV), _bf16(w).to(DEV), quantize_input=False)
    ref = oracle.qat_linear_ref(_bf16(x), _bf16(w), quantize_input=False)
    assert np.array_equal(ref, x @ w.T)
    assert np.array_equal(y.cpu().view(torch.int16).numpy(), _rne_bits(ref))


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (224, 352, 160), (1024, 768, 1024)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_w4a16_random_within_tolerance(mxq, M, N, K, with_bias):
    x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=3 * M + N)
    b = _bf16(0.05 * np.random.default_rng(K).standard_normal(N)) if with_bias else None
    y = mxq.qat_linear_fwd(x.to(DEV), w.to(DEV), None if b is None else b.to(DEV), quantize_input=False)
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    check_close(y, oracle.qat_linear_ref(x, w, b, quantize_input=False))


def test_w4a16_full_size_sampled_rows(mxq):
    M, N, K = 8192, 14336, 4096
    x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=0)
    y = mxq.qat_linear_fwd(x.to(DEV), w.to(DEV), quantize_input=False)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.random.default_rng(4).choice(M, 60, replace=False), [0, M - 1]]))
    check_close(y[torch.from_numpy(rows).to(DEV)],
                oracle.qat_linear_ref(x[torch.from_numpy(rows)], w, quantize_input=False))


def _r256(n: int) -> int:
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("M,N,K", [(96, 160, 352), (256, 128, 512)])
@pytest.mark.parametrize("sf", [6.0, 7.5])
def test_w4a4_operands_are_the_mxfp4_quant_as_e4m3(mxq, M, N, K, sf):
    """The W4A4 forward holds Q(x) and Q(w) in its workspace as E4M3 codes under
    the MXFP4 E8M0 scales (codes, then scales, each from a 256-byte boundary,
    x first).  Every code must be the E4M3 code of the oracle's E2M1 value
    (sign kept) and every scale byte the oracle's, padding included."""
    x = _bf16(mxq_inputs.mxfp4_large(M, K, seed=M + K))
    w = _bf16(mxq_inputs.mxfp4_large(N, K, seed=N + K + 1))
    ws_bytes = mxq.mxq_qat_linear_workspace_bytes(M, N, K, 1)
    ws = torch.full((ws_bytes,), 0xAB, dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mxq.mxq_qat_linear_fwd(x.to(DEV), w.to(DEV), None, M, N, K, 1, sf, y, ws, ws_bytes)
    wsh = ws.cpu().numpy()
    # E4M3 code of each E2M1 codebook value, looked up in the E4M3 decode table
    t8, t4 = oracle.e4m3_decode_table(), oracle.e2m1_decode_table()
    as_e4m3 = np.array([int(np.flatnonzero(t8 == t4[i])[0]) for i in range(8)], dtype=np.uint8)
    off = 0
    for t, R in ((x, M), (w, N)):
        nib, sc = oracle.mxfp4_quant(t.to(torch.float32).numpy(), sf)
        codes = np.empty((R, K), np.uint8)
        codes[:, 0::2], codes[:, 1::2] = nib & 0xF, nib >> 4
        want = as_e4m3[codes & 7] | np.where(codes & 8, 0x80, 0).astype(np.uint8)
        got = wsh[off:off + R * K].reshape(R, K)
        assert np.array_equal(got, want)
        off += _r256(R * K)
        nsb = mxq.mxq_scale_bytes(R, K // 32)
        assert np.array_equal(wsh[off:off + nsb], oracle.swizzle_scales(sc))
        off += _r256(nsb)


@pytest.mark.parametrize("shape", [(64, 256), (4096, 4096), (3, 96)])
@pytest.mark.parametrize("sf", [6.0, 7.5])
def test_bf16_qdq_bit_exact(mxq, shape, sf):
    """bf16 -> bf16 quant-dequant equals the fp32 oracle on the widened values,
    narrowed back to bf16 (exact)."""
    a = mxq_inputs.mxfp4_large(shape[0], shape[1], seed=shape[0])
    xb = _bf16(a)
    y = mxq.qdq_mxfp4(xb.to(DEV), sf).cpu()
    ref = oracle.mxfp4_qdq(xb.to(torch.float32).numpy(), np.float32(sf))
    assert np.array_equal(torch.from_numpy(ref).to(torch.bfloat16).to(torch.float32).numpy().view(np.uint32),
                          ref.view(np.uint32))  # exact in bf16
    assert np.array_equal(y.view(torch.int16).numpy(), torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy())


def test_bf16_qdq_every_bf16_pattern_under_six_scales(mxq):
    """Every finite bf16 pattern p, each in its own block of 32 whose maximum
    is an anchor 1.5 * 2^(E_p + j), j = 0..5, so that p / scale falls in every
    codebook interval and on every midpoint of the MXFP4 rule ("AMCT FakeQuant
    模拟伪量化工具包", section 2): the bf16 quant-dequant equals the fp32 oracle
    on the widened values, bit for bit."""
    pats = np.arange(1 << 16, dtype=np.uint32)
    f = (pats << 16).view(np.float32)
    p = f[np.isfinite(f) & (f != 0)]
    e_p = np.floor(np.log2(np.abs(p).astype(np.float64))).astype(np.int64)
    rows = []
    for j in range(6):
        blk = np.zeros((p.size, 32), np.float32)
        blk[:, 0] = (1.5 * np.exp2(np.minimum(e_p + j, 127))).astype(np.float32)
        blk[:, 1] = p
        rows.append(blk)
    a = np.concatenate(rows)
    a = a[np.isfinite(a).all(axis=1)]
    # keep the blocks whose anchor bf16 holds exactly (not the deepest subnormal ones)
    a = a[torch.from_numpy(a[:, 0]).to(torch.bfloat16).to(torch.float32).numpy() == a[:, 0]]
    xb = torch.from_numpy(a).to(torch.bfloat16)
    assert torch.equal(xb.to(torch.float32), torch.from_numpy(a))
    y = mxq.qdq_mxfp4(xb.to(DEV), 6.0).cpu()
    ref = oracle.mxfp4_qdq(a, np.float32(6.0))
    assert np.array_equal(y.view(torch.int16).numpy(), torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy())


# ------------------------------------------------------------------ MoE experts

def _grouped_ref(x, w, off, quantize_input, sf=6.0):
    """The oracle's QAT forward applied to each group's rows and its expert's
    weight (rows of x are independent, so this is the layer's definition)."""
    T, N = x.shape[0], w.shape[1]
    ref = np.zeros((T, N))
    for e in range(len(off) - 1):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            ref[r0:r1] = oracle.qat_linear_ref(x[r0:r1], w[e], None, scale_factor=sf, quantize_input=quantize_input)
    return ref


def _grouped_run(mxq, x, w, off, quantize_input, sf=6.0):
    d_off = torch.from_numpy(np.asarray(off, dtype=np.int64)).to(DEV)
    y = mxq.qat_grouped_fwd(x.to(DEV), w.to(DEV), d_off, quantize_input=quantize_input, scale_factor=sf)
    torch.cuda.synchronize()
    assert mxq.mxq_poll_device_error() == 0
    return y


@pytest.mark.parametrize("quantize_input", [True, False])
@pytest.mark.parametrize("sizes,N,K", [([3, 0, 200, 0, 97], 256, 128), ([128, 128], 384, 96), ([0, 0, 1], 128, 512)])
def test_grouped_exact_sums_bit_exact(mxq, quantize_input, sizes, N, K):
    """Each expert's rows against its own weight, operands chosen so that
    every partial sum is exact in fp32 (W on the MXFP4 grid; x on the grid for
    W4A4, on a 2^-4 grid for W4A16): y = bf16(exact), empty groups included."""
    off = mxq_inputs.offsets_from_sizes(sizes)
    T, E = int(off[-1]), len(sizes)
    if quantize_input:
        x = _on_grid(T, K, 11)
    else:
        x = np.random.default_rng(T + K).integers(-128, 129, size=(T, K)) / 16.0
    w = np.stack([_on_grid(N, K, 20 + e) for e in range(E)])
    y = _grouped_run(mxq, _bf16(x), _bf16(w), off, quantize_input)
    ref = _grouped_ref(_bf16(x), _bf16(w), off, quantize_input)
    exact = np.zeros((T, N))
    for e in range(E):
        exact[off[e]:off[e + 1]] = x[off[e]:off[e + 1]] @ w[e].T
    assert np.array_equal(ref, exact)
    assert np.array_equal(y.cpu().view(torch.int16).numpy(), _rne_bits(ref))


@pytest.mark.parametrize("quantize_input", [True, False])
@pytest.mark.parametrize("sf", [6.0, 7.5])
def test_grouped_random_within_tolerance(mxq, quantize_input, sf):
    sizes = [37, 0, 300, 129, 0, 1, 211]
    off, x, w, _ = mxq_inputs.moe_inputs(len(sizes), sum(sizes), 256, 384, seed=17, sizes=sizes)
    y = _grouped_run(mxq, x, w, off, quantize_input, sf)
    check_close(y, _grouped_ref(x, w, off, quantize_input, sf))


def test_grouped_many_experts(mxq):
    """300 experts, more than the GEMM's shared-memory group tables hold."""
    E, T, K, N = 300, 1200, 64, 128
    sizes = mxq_inputs.dirichlet_group_sizes(E, T, alpha=0.5, seed=3)
    off, x, w, _ = mxq_inputs.moe_inputs(E, T, K, N, seed=5, sizes=sizes)
    for qi in (True, False):
        check_close(_grouped_run(mxq, x, w, off, qi), _grouped_ref(x, w, off, qi))


def test_grouped_full_size_sampled_rows(mxq):
    """The MoE layer's shape (32 experts, 32768 Dirichlet-routed rows,
    K = 7168, N = 4096), both modes, on sampled rows of six experts."""
    E, T, K, N = 32, 32768, 7168, 4096
    off, x, w, _ = mxq_inputs.moe_inputs(E, T, K, N, seed=0, need_dy=False)
    n = np.diff(off)
    rng = np.random.default_rng(4)
    experts = rng.choice(np.nonzero(n > 0)[0], 6, replace=False)
    for qi in (True, False):
        y = _grouped_run(mxq, x, w, off, qi)
        for e in experts:
            r0, r1 = int(off[e]), int(off[e + 1])
            rows = np.unique(np.concatenate([[r0, r1 - 1], rng.integers(r0, r1, size=6)]))
            ref = oracle.qat_linear_ref(x[torch.from_numpy(rows)], w[int(e)], None, quantize_input=qi)
            check_close(y[torch.from_numpy(rows).to(DEV)], ref)
        del y
