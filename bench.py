#!/usr/bin/env python
"""Benchmark of the MX block-scaled hot path on GB300 -- prints ONE JSON line.

One step = one pass of the whole path over one batch of synthetic inputs,
everything resident in HBM before the timed region starts:
  * dense MXFP8 linear layer, M=8192 tokens, N=14336, K=4096: forward
    (dual-axis quant of X and W + GEMM), input gradient (dual quant of dY +
    GEMM), weight gradient (GEMM), in saved-quant mode (--mode recompute for
    the recompute-in-backward variant);
  * MoE expert layer, 32 experts, 32768 routed rows (Dirichlet(0.5) group
    sizes), K=7168, N=4096: row quant of X and dY, dual quant of the stacked
    weights, per-group column quant of dY and X, grouped GEMM forward, input
    gradient and weight gradient;
  * MXFP4 quant-dequant and packed MXFP4 quant of a 4096 x 4096 fp32 tensor.
value = GEMM FLOPs of the step (3*2*M*N*K + 3*2*T*N*K) / step time, TFLOP/s.

--impl reference times the CPU oracle on a bounded sample of the same workload
(the slow reference this tier compares against).  Multi-GPU (torchrun): every
rank runs an independent replica (weak scaling); barrier + max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

LIN = dict(M=8192, N=14336, K=4096)
MOE = dict(E=32, T=32768, K=7168, N=4096)
FP4 = dict(R=4096, C=4096)
LIN_FLOP = 3 * 2 * LIN["M"] * LIN["N"] * LIN["K"]
MOE_FLOP = 3 * 2 * MOE["T"] * MOE["N"] * MOE["K"]
STEP_FLOP = LIN_FLOP + MOE_FLOP
METRIC = "MXFP8 linear fwd+bwd + MoE grouped-GEMM fwd/dX/dW TFLOP/s (step incl. MX quant, MXFP4 QDQ)"
WORKLOAD = ("linear M8192 N14336 K4096 fwd+bwd (saved-quant) + MoE E32 T32768 K7168 N4096 fwd+dX+dW "
            "+ MXFP4 QDQ/pack 4096x4096")
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
GEMM_SOURCES = [os.path.join(ROOT, "mx_block_scaled_mxq_gb300", "csrc", f) for f in ("mxq_gemm.cu", "mxq_device.cuh")]
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the GEMM
# kernel for each launch the timed region brackets, from one ncu capture of the
# full-size launches (profiles/k_gemm__bench_launches_dram.md), keyed by a
# hash of the kernel source; when the source has changed since, traffic is null.
GEMM_DRAM_TRAFFIC = {
    "320d26573fb1d5aa": {"linear_dw_gemm": 287821568, "moe_fwd_gemm": 1499957504,
                         "moe_dx_gemm": 1531104768, "moe_dw_gemm": 2236594688},
}
FP8_PER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)


# ----------------------------------------------------------------------------- distributed

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("MXQ_BENCH_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Max of a per-rank scalar over all ranks (identity for one rank)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU workload

class Workload:
    """Device buffers for one step, built once; inputs are generated on the host
    by the seeded recipe and copied to the GPU before any timing."""

    def __init__(self, dev, mode: int, host_inputs):
        import mx_block_scaled_mxq_gb300 as m
        self.m = m
        self.dev = dev
        self.mode = mode
        (x, w, dy), (off, xm, wm, dym), a4 = host_inputs
        M, N, K = LIN["M"], LIN["N"], LIN["K"]
        E, T, Km, Nm = MOE["E"], MOE["T"], MOE["K"], MOE["N"]
        u8 = lambda n: torch.empty(max(int(n), 1), dtype=torch.uint8, device=dev)  # noqa: E731
        bf = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=dev)  # noqa: E731
        # linear
        self.x, self.w, self.dy = x.to(dev), w.to(dev), dy.to(dev)
        self.lctx = u8(m.mxq_linear_ctx_bytes(M, N, K, mode))
        self.lwsb = m.mxq_linear_workspace_bytes(M, N, K, mode)
        self.lws = u8(self.lwsb)
        self.y, self.dx, self.dw = bf(M, N), bf(M, K), bf(N, K)
        # MoE
        self.off = torch.from_numpy(off).to(dev)
        self.xm, self.wm, self.dym = xm.to(dev), wm.reshape(E * Nm, Km).to(dev), dym.to(dev)
        self.t_pad = m.mxq_grouped_padded_rows(T, E)
        self.xmq, self.xms = u8(T * Km), u8(m.mxq_scale_bytes(T, Km // 32))
        self.wmq, self.wms = u8(E * Nm * Km), u8(m.mxq_scale_bytes(E * Nm, Km // 32))
        self.wmqT, self.wmsT = u8(Km * E * Nm), u8(m.mxq_scale_bytes(Km, E * Nm // 32))
        self.dymq, self.dyms = u8(T * Nm), u8(m.mxq_scale_bytes(T, Nm // 32))
        self.dymqT, self.dymsT = u8(Nm * self.t_pad), u8(m.mxq_scale_bytes(Nm, self.t_pad // 32))
        self.xmqT, self.xmsT = u8(Km * self.t_pad), u8(m.mxq_scale_bytes(Km, self.t_pad // 32))
        self.ym, self.dxm, self.dwm = bf(T, Nm), bf(T, Km), bf(E, Nm, Km)
        # MXFP4
        self.a4 = torch.from_numpy(a4).to(dev)
        self.y4 = torch.empty_like(self.a4)
        self.p4, self.s4 = u8(FP4["R"] * FP4["C"] // 2), u8(m.mxq_scale_bytes(FP4["R"], FP4["C"] // 32))

    # kernel launches per step (counted from the entry points called below)
    def launches(self) -> int:
        lin = 6 if self.mode == self.m.SAVE_QUANT else 8
        return lin + 6 + 2

    def step(self, ev=None):
        """One pass; `ev` (a list) receives (name, start, end, flop) event pairs
        bracketing every call that launches the GEMM kernel alone."""
        m = self.m
        M, N, K = LIN["M"], LIN["N"], LIN["K"]
        E, T, Km, Nm = MOE["E"], MOE["T"], MOE["K"], MOE["N"]

        def timed(name, flop, fn):
            if ev is None:
                fn()
                return
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            ev.append((name, a, b, flop))

        mode = self.mode
        m.mxq_linear_fwd(self.x, self.w, M, N, K, mode, self.lctx, self.y, self.lws, self.lwsb)
        m.mxq_linear_bwd_dx(self.dy, self.w, M, N, K, mode, self.lctx, self.dx, self.lws, self.lwsb)
        dw_call = lambda: m.mxq_linear_bwd_dw(self.dy, self.x, M, N, K, mode, self.lctx, self.dw, self.lws,  # noqa
                                              self.lwsb)
        if mode == m.SAVE_QUANT:
            timed("linear_dw_gemm", 2 * M * N * K, dw_call)   # saved-quant dW launches the GEMM only
        else:
            dw_call()
        # X and dY: row quant (fwd / dX operands) and per-group column quant (dW
        # operands) from one read each; W: row quant and column quant along N
        m.mxq_quantize_grouped_dual(self.xm, T, Km, self.off, E, self.t_pad, self.xmq, self.xms, self.xmqT, self.xmsT)
        m.mxq_quantize(self.wm, m.BF16, E * Nm, Km, Km, -1, m.E4M3, 1, self.wmq, self.wms, self.wmqT, self.wmsT)
        m.mxq_quantize_grouped_dual(self.dym, T, Nm, self.off, E, self.t_pad, self.dymq, self.dyms, self.dymqT,
                                    self.dymsT)
        gf = 2 * T * Nm * Km
        timed("moe_fwd_gemm", gf, lambda: m.mxq_grouped_gemm(m.GG_FWD, self.xmq, self.xms, self.wmq, self.wms,
                                                             self.off, E, T, Nm, Km, 0, self.ym))
        timed("moe_dx_gemm", gf, lambda: m.mxq_grouped_gemm(m.GG_DX, self.dymq, self.dyms, self.wmqT, self.wmsT,
                                                            self.off, E, T, Nm, Km, 0, self.dxm))
        timed("moe_dw_gemm", gf, lambda: m.mxq_grouped_gemm(m.GG_DW, self.dymqT, self.dymsT, self.xmqT, self.xmsT,
                                                            self.off, E, T, Nm, Km, self.t_pad, self.dwm))
        m.mxq_qdq_mxfp4(self.a4, self.y4, FP4["R"], FP4["C"], 32, 6.0)
        m.mxq_quantize(self.a4, m.F32, FP4["R"], FP4["C"], FP4["C"], -1, m.E2M1, 0, self.p4, self.s4, None, None)



# ----------------------------------------------------------------------------- end to end

class E2EPipeline:
    """End-to-end steps through the public API with host buffers.

    Per step, the step's inputs -- the layers' activations and upstream
    gradients (X, dY of the dense layer; X, dY of the MoE layer; the MXFP4
    tensor) -- are copied from pinned host memory to the GPU, the step runs,
    and its results -- outputs and input gradients (Y, dX; MoE Y, dX; the MXFP4
    quant-dequant and packed tensors) -- are copied back to pinned host memory.
    Parameters (W, the experts' weights) and their gradients stay in HBM, as
    in training.  Copies in, compute and copies out run on three streams over
    two device slots, so step i's copies overlap steps i-1 / i+1's compute;
    every step's copies are inside the timed region."""
    IN = ("x", "dy", "xm", "dym", "a4")
    OUT = ("y", "dx", "ym", "dxm", "y4", "p4", "s4")

    def __init__(self, wl):
        self.wl = wl
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)  # noqa: E731
        self.h_in = {k: pin(getattr(wl, k)) for k in self.IN}
        for k in self.IN:
            self.h_in[k].copy_(getattr(wl, k))
        self.h_out = [{k: pin(getattr(wl, k)) for k in self.OUT} for _ in range(2)]
        self.slots = [{k: getattr(wl, k) for k in self.IN + self.OUT},
                      {k: torch.empty_like(getattr(wl, k)) for k in self.IN + self.OUT}]
        self.s_in, self.s_comp, self.s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]  # noqa: E731
        self.in_done, self.comp_done, self.out_done = ev(), ev(), ev()
        self.n = 0  # steps issued

    def bytes(self):
        nb = lambda t: t.numel() * t.element_size()  # noqa: E731
        return (sum(nb(self.h_in[k]) for k in self.IN), sum(nb(self.h_out[0][k]) for k in self.OUT))

    def step(self):
        i, slot = self.n, self.n % 2
        S = self.slots[slot]
        with torch.cuda.stream(self.s_in):
            if i >= 2:
                self.s_in.wait_event(self.comp_done[slot])  # step i-2 has read this slot's inputs
            for k in self.IN:
                S[k].copy_(self.h_in[k], non_blocking=True)
            self.in_done[slot].record()
        with torch.cuda.stream(self.s_comp):
            self.s_comp.wait_event(self.in_done[slot])
            if i >= 2:
                self.s_comp.wait_event(self.out_done[slot])  # step i-2's results have left this slot
            for k in self.IN + self.OUT:
                setattr(self.wl, k, S[k])
            self.wl.step()
            self.comp_done[slot].record()
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.comp_done[slot])
            for k in self.OUT:
                self.h_out[slot][k].copy_(S[k], non_blocking=True)
            self.out_done[slot].record()
        self.n += 1

    def restore(self):
        for k in self.IN + self.OUT:
            setattr(self.wl, k, self.slots[0][k])

    def timed(self, steps, world):
        """Seconds for `steps` pipelined steps: CUDA events from before the
        first copy in to after the last copy out, synchronized on both sides."""
        barrier(world)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(self.s_in)
        for _ in range(steps):
            self.step()
        self.s_out.wait_stream(self.s_comp)
        end.record(self.s_out)
        torch.cuda.synchronize()
        barrier(world)
        return start.elapsed_time(end) / 1e3


def make_host_inputs():
    import mxq_inputs
    x, w, dy = mxq_inputs.linear_inputs(LIN["M"], LIN["N"], LIN["K"], seed=0)
    moe = mxq_inputs.moe_inputs(MOE["E"], MOE["T"], MOE["K"], MOE["N"], seed=0)
    a4 = mxq_inputs.mxfp4_large(FP4["R"], FP4["C"], seed=0)
    return (x, w, dy), moe, a4


def time_steps(fn, steps, world):
    """CUDA-event time of `steps` calls of fn, bracketed by barrier + synchronize."""
    barrier(world)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        fn()
    e.record()
    torch.cuda.synchronize()
    barrier(world)
    return s.elapsed_time(e) / 1e3


L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


def time_flushed(fn, n, flush):
    """Mean CUDA-event time (ms) of fn over n calls, each after writing a buffer
    twice the size of L2 so that no call finds its inputs cached."""
    total = 0.0
    for _ in range(n):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        total += a.elapsed_time(b)
    return total / n


def gemm_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemm_traffic(per_kind):
    """Average measured DRAM bytes per bracketed GEMM launch, or None."""
    rec = GEMM_DRAM_TRAFFIC.get(gemm_source_hash())
    if not rec or any(k not in rec for k in per_kind):
        return None
    n = sum(v[1] for v in per_kind.values())
    return sum(rec[k] * v[1] for k, v in per_kind.items()) / n


def read_peaks():
    try:
        with open(PEAKS) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------------------- CPU oracle sample

CPU_ROWS = 128


def cpu_sample_step(host_inputs):
    """The oracle on a bounded sample of the same workload: the first 128 token
    rows of the dense layer (Y, dX rows and their dW contribution, full W), the
    first 128 routed rows of the MoE layer (their experts' full weights), and
    128 rows of the MXFP4 tensor.  Returns the GEMM FLOPs it covered."""
    import oracle
    (x, w, dy), (off, xm, wm, dym), a4 = host_inputs
    r = CPU_ROWS
    N, K = LIN["N"], LIN["K"]
    flop = 0
    # dense layer sample
    xs, dys = x[:r], dy[:r]
    qx, sx = oracle.mxfp8_quant_rows(xs)
    qw, sw = oracle.mxfp8_quant_rows(w)
    oracle.gemm_ref(qx, sx, qw, sw)
    qdy, sdy = oracle.mxfp8_quant_rows(dys)
    qwT, swT = oracle.mxfp8_quant_cols(w)
    oracle.gemm_ref(qdy, sdy, qwT, swT)
    qdyT, sdyT = oracle.mxfp8_quant_cols(dys)
    qxT, sxT = oracle.mxfp8_quant_cols(xs)
    oracle.gemm_ref(qdyT, sdyT, qxT, sxT)
    flop += 3 * 2 * r * N * K
    # MoE sample: rows [0, r) and the experts that own them
    Nm, Km = MOE["N"], MOE["K"]
    qx, sx = oracle.mxfp8_quant_rows(xm[:r])
    qdy, sdy = oracle.mxfp8_quant_rows(dym[:r])
    for e in range(MOE["E"]):
        r0, r1 = int(off[e]), min(int(off[e + 1]), r)
        if r1 <= r0:
            if r0 >= r:
                break
            continue
        qw, sw = oracle.mxfp8_quant_rows(wm[e])
        oracle.gemm_ref(qx[r0:r1], sx[r0:r1], qw, sw)
        qwT, swT = oracle.mxfp8_quant_cols(wm[e])
        oracle.gemm_ref(qdy[r0:r1], sdy[r0:r1], qwT, swT)
        a, sa = oracle.mxfp8_quant_cols(dym[r0:r1])
        b, sb = oracle.mxfp8_quant_cols(xm[r0:r1])
        oracle.gemm_ref(a, sa, b, sb)
        flop += 3 * 2 * (r1 - r0) * Nm * Km
    # MXFP4 sample
    oracle.mxfp4_qdq(a4[:r])
    oracle.mxfp4_quant(a4[:r])
    return flop


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_baseline(host_inputs, steps: int):
    t0 = time.perf_counter()
    flop = 0
    for _ in range(steps):
        flop += cpu_sample_step(host_inputs)
    dt = time.perf_counter() - t0
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": (f"{steps} x [first {CPU_ROWS} rows of the dense layer (Y, dX rows + their dW part, full W), "
                       f"first {CPU_ROWS} MoE rows with their experts' full weights, {CPU_ROWS} rows of the MXFP4 "
                       "tensor]; C oracle single-threaded, binary64 numpy GEMMs on all cores"),
            "seconds": dt}


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--mode", choices=["save", "recompute"], default="save")
    ap.add_argument("--cpu-steps", type=int, default=5, help="oracle sample steps for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--quant-sweep", action="store_true",
                    help="instead of the step: dual-axis MXFP8 quant bandwidth over sizes (one JSON line each)")
    args = ap.parse_args()
    world, rank, local = dist_init()

    if args.quant_sweep:
        quant_sweep()
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import mx_block_scaled_mxq_gb300 as m
    m.load()
    mode = m.SAVE_QUANT if args.mode == "save" else m.RECOMPUTE
    host_inputs = make_host_inputs()
    wl = Workload(dev, mode, host_inputs)

    for _ in range(max(args.warmup, 3)):
        wl.step()
    torch.cuda.synchronize()
    assert m.mxq_poll_device_error() == 0, "a kernel reported a device error during warm-up"

    # ---- timed region: K steps, GEMM launches bracketed by events
    clocks = ClockSampler(dev.index)
    clocks.start()
    ev = []
    elapsed = time_steps(lambda: wl.step(ev), args.steps, world)
    clk = clocks.stop()
    elapsed = max_over_ranks(elapsed, world)
    gemm_ms = sum(a.elapsed_time(b) for _, a, b, _ in ev)
    gemm_flop = sum(f for *_, f in ev)
    per_kind = {}
    for name, a, b, f in ev:
        d = per_kind.setdefault(name, [0.0, 0])
        d[0] += a.elapsed_time(b)
        d[1] += 1

    # ---- component timings (outside the timed region, same buffers)
    comp = component_timings(wl, world)

    # ---- end to end through the public API with host buffers
    e2e = E2EPipeline(wl)
    hb_in, hb_out = e2e.bytes()
    for _ in range(2):
        e2e.step()
    e2e_t = e2e.timed(args.e2e_steps, world)
    e2e_t = max_over_ranks(e2e_t, world)
    e2e.restore()
    assert m.mxq_poll_device_error() == 0

    peaks, peak_kind = read_peaks()
    fp8_peak = FP8_PER_BF16 * float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    achieved = gemm_flop / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    value = world * STEP_FLOP * args.steps / elapsed / 1e12

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(elapsed / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded: N(0,1) X, N(0,0.02) W, N(0,1e-3) dY; Dirichlet(0.5) groups; t(3) MXFP4 input)",
        "config": {"workload": WORKLOAD, "mode": args.mode, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (step touches > 8 GB)", "step_gemm_flop": STEP_FLOP},
        "roofline": {"bound": "tensor",
                     "kernel": "k_gemm<1,MXF8,0,MC> (tcgen05 kind::mxf8f6f4; B-multicast CTA pairs for dense and dW)",
                     "achieved": round(achieved, 1) if achieved else None,
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp8_peak, 4) if achieved else None,
                     "peak_source": f"{peak_kind}: 2 x bf16_tflops_sustained (nominal fp8/bf16 ratio)",
                     "launches_timed": len(ev), "traffic": gemm_traffic(per_kind),
                     "traffic_unit": "bytes per launch", "kernel_source": gemm_source_hash()},
        "e2e": {"value": round(world * STEP_FLOP * args.e2e_steps / e2e_t / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": hb_in, "d2h_bytes_per_step": hb_out,
                "ms_per_step": round(e2e_t / args.e2e_steps * 1e3, 3)},
        "gpu_launches": wl.launches() * args.steps,
        "clocks": clk,
        "components": {**comp, "gemm_ms_per_launch": {k: round(v[0] / v[1], 4) for k, v in per_kind.items()}},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline(host_inputs, args.cpu_steps)
        line["cpu_baseline"]["value"] = float(f"{line['cpu_baseline']['value']:.4g}")
    if rank == 0:
        print(json.dumps(line), flush=True)


def quant_sweep():
    """Dual-axis MXFP8 quant of bf16 [R x C], C in {2048, 7168, 14336},
    R = ceil128(2^p / C) for p = 20, 22, ..., 30; algorithmic bytes 2 in +
    2 (1 + 1/32) out per element; L2 flushed before each timed launch."""
    import mxq_inputs
    import mx_block_scaled_mxq_gb300 as m
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    m.load()
    peaks, peak_kind = read_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for C in (2048, 7168, 14336):
        for p in range(20, 31, 2):
            R = ((1 << p) // C + 127) // 128 * 128
            x = mxq_inputs.sweep_bf16_device(R, C, seed=p * 100 + C, device=dev)
            q, s, qT, sT = (torch.empty(R * C, dtype=torch.uint8, device=dev),
                            torch.empty(m.mxq_scale_bytes(R, C // 32), dtype=torch.uint8, device=dev),
                            torch.empty(R * C, dtype=torch.uint8, device=dev),
                            torch.empty(m.mxq_scale_bytes(C, R // 32), dtype=torch.uint8, device=dev))
            fn = lambda: m.mxq_quantize(x, m.BF16, R, C, C, -1, m.E4M3, 1, q, s, qT, sT)  # noqa: E731
            fn()
            ms = time_flushed(fn, 5, flush)
            gbs = R * C * 4.0625 / (ms / 1e3) / 1e9
            print(json.dumps({"sweep": "mxfp8_dual_quant", "rows": R, "cols": C, "elements": R * C,
                              "ms": round(ms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / hbm, 3),
                              "peak": f"{hbm} GB/s ({peak_kind} HBM copy)"}), flush=True)
            del x, q, s, qT, sT
    assert m.mxq_poll_device_error() == 0


def component_timings(wl, world):
    """Per-part device times (ms) of one step's pieces, averaged over a few runs."""
    m = wl.m
    M, N, K = LIN["M"], LIN["N"], LIN["K"]
    E, T, Km, Nm = MOE["E"], MOE["T"], MOE["K"], MOE["N"]
    dq = torch.empty((M, N), dtype=torch.uint8, device=wl.dev)
    ds = torch.empty(m.mxq_scale_bytes(M, N // 32), dtype=torch.uint8, device=wl.dev)
    dqT = torch.empty((N, M), dtype=torch.uint8, device=wl.dev)
    dsT = torch.empty(m.mxq_scale_bytes(N, M // 32), dtype=torch.uint8, device=wl.dev)
    R4, C4 = FP4["R"], FP4["C"]
    m4 = torch.empty((R4, C4 // 32), dtype=torch.int32, device=wl.dev)
    g4 = torch.empty_like(wl.a4)
    qat_ws_bytes = max(m.mxq_qat_linear_workspace_bytes(M, N, K, 1), m.mxq_qat_linear_workspace_bytes(M, N, K, 0))
    qat_ws = torch.empty(qat_ws_bytes, dtype=torch.uint8, device=wl.dev)
    wc_bytes = m.mxq_linear_weight_cache_bytes(N, K)
    wcache = torch.empty(wc_bytes, dtype=torch.uint8, device=wl.dev)

    def layer_wq():  # one micro-batch with W's quantization taken from the cache (ctx layouts share a prefix)
        m.mxq_linear_fwd_wq(wl.x, wcache, M, N, K, wl.mode, wl.lctx, wl.y, wl.lws, wl.lwsb)
        m.mxq_linear_bwd_dx_wq(wl.dy, wcache, M, N, K, wl.mode, wl.lctx, wl.dx, wl.lws, wl.lwsb)
        m.mxq_linear_bwd_dw(wl.dy, wl.x, M, N, K, wl.mode, wl.lctx, wl.dw, wl.lws, wl.lwsb)

    def layer_plain():
        m.mxq_linear_fwd(wl.x, wl.w, M, N, K, wl.mode, wl.lctx, wl.y, wl.lws, wl.lwsb)
        m.mxq_linear_bwd_dx(wl.dy, wl.w, M, N, K, wl.mode, wl.lctx, wl.dx, wl.lws, wl.lwsb)
        m.mxq_linear_bwd_dw(wl.dy, wl.x, M, N, K, wl.mode, wl.lctx, wl.dw, wl.lws, wl.lwsb)
    parts = {
        "linear_fwd": lambda: m.mxq_linear_fwd(wl.x, wl.w, M, N, K, wl.mode, wl.lctx, wl.y, wl.lws, wl.lwsb),
        "linear_bwd_dx": lambda: m.mxq_linear_bwd_dx(wl.dy, wl.w, M, N, K, wl.mode, wl.lctx, wl.dx, wl.lws, wl.lwsb),
        "linear_bwd_dw": lambda: m.mxq_linear_bwd_dw(wl.dy, wl.x, M, N, K, wl.mode, wl.lctx, wl.dw, wl.lws, wl.lwsb),
        "dual_quant_dY": lambda: m.mxq_quantize(wl.dy, m.BF16, M, N, N, -1, m.E4M3, 1, dq, ds, dqT, dsT),
        "moe_grouped_col_quant_X": lambda: m.mxq_quantize_grouped_col(wl.xm, T, Km, wl.off, E, wl.t_pad, wl.xmqT,
                                                                      wl.xmsT),
        "moe_grouped_dual_quant_X": lambda: m.mxq_quantize_grouped_dual(wl.xm, T, Km, wl.off, E, wl.t_pad, wl.xmq,
                                                                        wl.xms, wl.xmqT, wl.xmsT),
        "moe_fwd": lambda: m.mxq_grouped_gemm(m.GG_FWD, wl.xmq, wl.xms, wl.wmq, wl.wms, wl.off, E, T, Nm, Km, 0, wl.ym),
        "mxfp4_qdq": lambda: m.mxq_qdq_mxfp4(wl.a4, wl.y4, R4, C4, 32, 6.0),
        "mxfp4_ste_fwd": lambda: m.mxq_mxfp4_ste_forward(wl.a4, wl.y4, m4, R4, C4, 32, 6.0),
        "mxfp4_ste_bwd": lambda: m.mxq_mxfp4_ste_backward(wl.y4, m4, R4, C4, g4),
        "linear_weight_quant": lambda: m.mxq_linear_quantize_weight(wl.w, N, K, wcache, wc_bytes),
        "linear_layer": layer_plain,
        "linear_wq": layer_wq,
        "qat_linear_fwd_w4a4": lambda: m.mxq_qat_linear_fwd(wl.x, wl.w, None, M, N, K, 1, 6.0, wl.y, qat_ws,
                                                            qat_ws_bytes),
        "qat_linear_fwd_w4a16": lambda: m.mxq_qat_linear_fwd(wl.x, wl.w, None, M, N, K, 0, 6.0, wl.y, qat_ws,
                                                             qat_ws_bytes),
    }
    out = {}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=wl.dev)
    for name, fn in parts.items():
        fn()
        out[name + "_ms"] = round(time_flushed(fn, 5, flush), 4)
    # derived throughputs
    out["linear_tflops"] = round(LIN_FLOP / ((out["linear_fwd_ms"] + out["linear_bwd_dx_ms"] + out["linear_bwd_dw_ms"])
                                             / 1e3) / 1e12, 1)
    dual_bytes = M * N * (2 + 2 * (1 + 1 / 32))
    out["dual_quant_dY_gbs"] = round(dual_bytes / (out["dual_quant_dY_ms"] / 1e3) / 1e9, 1)
    tp = wl.t_pad
    gcol_bytes = T * Km * 2 + Km * tp * (1 + 1 / 32)
    out["moe_grouped_col_quant_X_gbs"] = round(gcol_bytes / (out["moe_grouped_col_quant_X_ms"] / 1e3) / 1e9, 1)
    gdual_bytes = gcol_bytes + T * Km * (1 + 1 / 32)
    out["moe_grouped_dual_quant_X_gbs"] = round(gdual_bytes / (out["moe_grouped_dual_quant_X_ms"] / 1e3) / 1e9, 1)
    out["mxfp4_qdq_gbs"] = round(R4 * C4 * 8 / (out["mxfp4_qdq_ms"] / 1e3) / 1e9, 1)
    # clipped STE: 4 B in + 4 B out + 1/8 B of mask per element, both directions
    out["mxfp4_ste_fwd_gbs"] = round(R4 * C4 * 8.125 / (out["mxfp4_ste_fwd_ms"] / 1e3) / 1e9, 1)
    out["mxfp4_ste_bwd_gbs"] = round(R4 * C4 * 8.125 / (out["mxfp4_ste_bwd_ms"] / 1e3) / 1e9, 1)
    out["qat_linear_fwd_w4a4_tflops"] = round(2 * M * N * K / (out["qat_linear_fwd_w4a4_ms"] / 1e3) / 1e12, 1)
    out["qat_linear_fwd_w4a16_tflops"] = round(2 * M * N * K / (out["qat_linear_fwd_w4a16_ms"] / 1e3) / 1e12, 1)
    out["moe_fwd_tflops"] = round(2 * T * Nm * Km / (out["moe_fwd_ms"] / 1e3) / 1e12, 1)
    # the other linear mode on the same buffers
    other = m.RECOMPUTE if wl.mode == m.SAVE_QUANT else m.SAVE_QUANT
    need_ctx = m.mxq_linear_ctx_bytes(M, N, K, other)
    need_ws = m.mxq_linear_workspace_bytes(M, N, K, other)
    ctx = torch.empty(need_ctx, dtype=torch.uint8, device=wl.dev)
    ws = torch.empty(need_ws, dtype=torch.uint8, device=wl.dev)

    def layer():
        m.mxq_linear_fwd(wl.x, wl.w, M, N, K, other, ctx, wl.y, ws, need_ws)
        m.mxq_linear_bwd_dx(wl.dy, wl.w, M, N, K, other, ctx, wl.dx, ws, need_ws)
        m.mxq_linear_bwd_dw(wl.dy, wl.x, M, N, K, other, ctx, wl.dw, ws, need_ws)
    layer()
    t = time_steps(layer, 3, 1) / 3 * 1e3
    name = "recompute" if other == m.RECOMPUTE else "save"
    out[f"linear_{name}_ms"] = round(t, 4)
    out["linear_saved_bytes"] = {"save": m.mxq_linear_saved_bytes(M, N, K, m.SAVE_QUANT),
                                 "recompute": m.mxq_linear_saved_bytes(M, N, K, m.RECOMPUTE)}
    del ctx, ws, dq, ds, dqT, dsT, m4, g4, flush, qat_ws, wcache
    return out


def run_reference(args, world, rank):
    """The CPU oracle, as it stands, on a bounded sample per step (rank 0 only)."""
    if rank != 0:
        return
    host_inputs = make_host_inputs()
    for _ in range(args.warmup):
        cpu_sample_step(host_inputs)
    t0 = time.perf_counter()
    flop = 0
    for _ in range(args.steps):
        flop += cpu_sample_step(host_inputs)
    dt = time.perf_counter() - t0
    value = flop / dt / 1e12
    sample = (f"per step: first {CPU_ROWS} rows of the dense layer (Y, dX rows + their dW part, full W), first "
              f"{CPU_ROWS} MoE rows with their experts' full weights, {CPU_ROWS} rows of the MXFP4 tensor")
    line = {"impl": "reference", "metric": METRIC, "value": float(f"{value:.4g}"), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD + " (oracle on a bounded row sample)", "mode": args.mode},
            "cpu_baseline": {"value": float(f"{value:.4g}"), "unit": "TFLOP/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": float(f"{value:.4g}"), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
