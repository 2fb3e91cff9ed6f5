"""Host threads calling the library at the same time, in a fresh process, so
that each kernel's per-device first-launch setup (shared-memory attribute,
residency) runs while other threads launch too.  Each thread quantizes (dual
and per-group dual), multiplies (dense and grouped GEMMs) and runs the MXFP4
quant-dequant on its own stream; every result must equal, bit for bit, the
same calls made afterwards by one thread."""
import os
import subprocess
import sys
import threading

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N_THREADS = 8


def _inputs(torch, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(512, 1024, generator=g).bfloat16().cuda()
    w = (0.02 * torch.randn(384, 1024, generator=g)).bfloat16().cuda()
    f = torch.randn(256, 512, generator=g).cuda()
    sizes = [100, 0, 300, 112]
    off = torch.tensor([0, 100, 100, 400, 512], dtype=torch.int64).cuda()
    return x, w, f, sizes, off


def _calls(m, torch, inp, stream):
    """Launches on `stream`; returns the output tensors."""
    x, w, f, sizes, off = inp
    R, C = x.shape
    N = w.shape[0]
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device="cuda")  # noqa: E731
    q, s, qT, sT = u8(R * C), u8(m.mxq_scale_bytes(R, C // 32)), u8(R * C), u8(m.mxq_scale_bytes(C, R // 32))
    m.mxq_quantize(x, m.BF16, R, C, C, -1, m.E4M3, 1, q, s, qT, sT, stream)
    wq, ws = u8(N * C), u8(m.mxq_scale_bytes(N, C // 32))
    m.mxq_quantize(w, m.BF16, N, C, C, -1, m.E4M3, 0, wq, ws, None, None, stream)
    y = torch.empty(R, N, dtype=torch.bfloat16, device="cuda")
    m.mxq_gemm(q, s, wq, ws, R, N, C, y, N, stream)
    E, T = len(sizes), R
    tp = m.mxq_grouped_padded_rows(T, E)
    gq, gs, gqT, gsT = u8(T * C), u8(m.mxq_scale_bytes(tp, C // 32)), u8(C * tp), u8(m.mxq_scale_bytes(C, tp // 32))
    m.mxq_quantize_grouped_dual_padded(x, T, C, off, E, tp, gq, gs, gqT, gsT, stream)
    dw = torch.empty(E, C, C, dtype=torch.bfloat16, device="cuda")
    m.mxq_grouped_gemm(m.GG_DW, gqT, gsT, gqT, gsT, off, E, T, C, C, tp, dw, stream)
    fy = torch.empty_like(f)
    m.mxq_qdq_mxfp4(f, fy, f.shape[0], f.shape[1], 32, 6.0, stream)
    return [q, s, qT, sT, y, gq, gs, gqT, gsT, dw, fy]


def main():
    import torch
    import mx_block_scaled_mxq_gb300 as m
    m.load()
    torch.cuda.set_device(0)
    inputs = [_inputs(torch, 100 + i) for i in range(N_THREADS)]
    torch.cuda.synchronize()
    results, errors = [None] * N_THREADS, []
    start = threading.Barrier(N_THREADS)

    def run(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            start.wait()
            outs = _calls(m, torch, inputs[i], st)
            st.synchronize()
            results[i] = [o.cpu() for o in outs]
        except Exception as e:  # reported by the parent
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=run, args=(i,)) for i in range(N_THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert m.mxq_poll_device_error() == 0
    for i in range(N_THREADS):
        ref = [o.cpu() for o in _calls(m, torch, inputs[i], None)]
        torch.cuda.synchronize()
        for a, b in zip(results[i], ref):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"thread {i} differs"
    print("ok")


def test_concurrent_first_calls(mxq):
    r = subprocess.run([sys.executable, os.path.abspath(__file__)], cwd=ROOT, capture_output=True, text=True,
                       timeout=600, env=dict(os.environ, PYTHONPATH=ROOT))
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-3000:]


if __name__ == "__main__":
    main()
