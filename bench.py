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
# same full-size launches in the parity tests, keyed by a hash of the kernel
# source; when the source has changed since, traffic is null.
GEMM_DRAM_TRAFFIC = {
    "07342afad1665483": {"linear_dw_gemm": 259970560, "moe_fwd_gemm": 1491981056,
                         "moe_dx_gemm": 1538263296, "moe_dw_gemm": 2237048576},
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
        n_e = np.diff(np.asarray(off, dtype=np.int64))
        self.off_padded_total = int(((n_e + 127) // 128 * 128).sum())  # sum of the groups' padded lengths
        self.xm, self.wm, self.dym = xm.to(dev), wm.reshape(E * Nm, Km).to(dev), dym.to(dev)
        self.t_pad = m.mxq_grouped_padded_rows(T, E)
        # row quants of X and dY with per-group padded row scales (each expert's
        # rows start a scale tile, so the forward and dX tile each expert from its
        # first row)
        self.xmq, self.xms = u8(T * Km), u8(m.mxq_scale_bytes(self.t_pad, Km // 32))
        self.wmq, self.wms = u8(E * Nm * Km), u8(m.mxq_scale_bytes(E * Nm, Km // 32))
        self.wmqT, self.wmsT = u8(Km * E * Nm), u8(m.mxq_scale_bytes(Km, E * Nm // 32))
        self.dymq, self.dyms = u8(T * Nm), u8(m.mxq_scale_bytes(self.t_pad, Nm // 32))
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
        m.mxq_quantize_grouped_dual_padded(self.xm, T, Km, self.off, E, self.t_pad, self.xmq, self.xms, self.xmqT,
                                           self.xmsT)
        m.mxq_quantize(self.wm, m.BF16, E * Nm, Km, Km, -1, m.E4M3, 1, self.wmq, self.wms, self.wmqT, self.wmsT)
        m.mxq_quantize_grouped_dual_padded(self.dym, T, Nm, self.off, E, self.t_pad, self.dymq, self.dyms, self.dymqT,
                                           self.dymsT)
        gf = 2 * T * Nm * Km
        tp = self.t_pad
        timed("moe_fwd_gemm", gf, lambda: m.mxq_grouped_gemm(m.GG_FWD, self.xmq, self.xms, self.wmq, self.wms,
                                                             self.off, E, T, Nm, Km, tp, self.ym))
        timed("moe_dx_gemm", gf, lambda: m.mxq_grouped_gemm(m.GG_DX, self.dymq, self.dyms, self.wmqT, self.wmsT,
                                                            self.off, E, T, Nm, Km, tp, self.dxm))
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


L2_BYTES = 129 << 20


def time_rotating(fns, reps=8, warm=2):
    """Mean device time (ms) of one call, over back-to-back calls that cycle
    through `fns` -- each on its own buffers, together larger than L2, so no
    call finds its inputs cached and every call pays the write-back of its
    predecessor's output, as inside a running step.  The calls are captured
    once in a CUDA graph and replayed, so the host's launch overhead between
    short kernels does not count; if capture is refused, each call is
    bracketed by its own events instead."""
    n = len(fns)
    for i in range(warm * n):
        fns[i % n]()
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps * n):
                fns[i % n]()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / (reps * n)
        del g
        return ms
    except RuntimeError:
        torch.cuda.synchronize()
    pairs = []
    for i in range(reps * n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fns[i % n]()
        b.record()
        pairs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs) / len(pairs)


def copies_past_l2(nbytes_per_set: int, cap: int = 8) -> int:
    """Buffer sets to rotate through so that together they exceed twice L2."""
    return max(1, min(cap, -(-2 * L2_BYTES // max(nbytes_per_set, 1))))


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


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def quant_oracle_rates(host_inputs, threads: int):
    """The quant oracle on bounded samples of the step's tensors, at 1 thread
    and at `threads` threads, in GB/s of the same algorithmic bytes as the GPU
    kernel of that name.  The sample is cut into slices before the clock
    starts (rows, or columns for the per-group quant); one thread runs them
    in turn, the pool all at once (the oracle's C calls release the GIL)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    (x, w, dy), (off, xm, wm, dym), a4 = host_inputs
    tasks = {}
    # dual quant of the dense dY: 2048 of its 8192 rows
    dyb = oracle._bf16_bits(dy[:2048])
    sl = [np.ascontiguousarray(dyb[r:r + 256]) for r in range(0, dyb.shape[0], 256)]
    tasks["dual_quant_dY"] = ([lambda a=a: (oracle.mxfp8_quant_rows(a), oracle.mxfp8_quant_cols(a)) for a in sl],
                              dyb.size * DUAL_QUANT_B, "dY rows 0..2047 (2048 x 14336)")
    # grouped dual quant of the MoE X: its first 2048 routed rows, groups clipped there
    Ts = 2048
    offs = np.minimum(np.asarray(off, dtype=np.int64), Ts)
    xb = oracle._bf16_bits(xm[:Ts])
    C = xb.shape[1]
    cols = [np.ascontiguousarray(xb[:, c:c + 896]) for c in range(0, C, 896)]
    padded = int(((np.diff(offs) + 127) // 128 * 128).sum())
    tasks["grouped_dual_quant_moe_X"] = (
        [lambda a=a: (oracle.mxfp8_quant_rows(a), oracle.mxfp8_quant_cols_grouped(a, offs)) for a in cols],
        Ts * C * (2 + 1 + 1 / 32) + C * padded * (1 + 1 / 32), "MoE X rows 0..2047 (2048 x 7168), groups clipped")
    # MXFP4 kernels: 1024 of the 4096 rows
    a = np.ascontiguousarray(a4[:1024])
    rs = [np.ascontiguousarray(a[r:r + 128]) for r in range(0, a.shape[0], 128)]
    masks = [oracle.mxfp4_saturation_mask(b) for b in rs]
    tasks["mxfp4_qdq"] = ([lambda b=b: oracle.mxfp4_qdq(b) for b in rs], a.size * QDQ_F32_B,
                          "MXFP4 tensor rows 0..1023 (1024 x 4096)")
    tasks["mxfp4_ste_fwd"] = ([lambda b=b: (oracle.mxfp4_qdq(b), oracle.mxfp4_saturation_mask(b)) for b in rs],
                              a.size * STE_B, "MXFP4 tensor rows 0..1023")
    tasks["mxfp4_ste_bwd"] = ([lambda b=b, mk=mk: oracle.mxfp4_ste_backward(b, mk) for b, mk in zip(rs, masks)],
                              a.size * STE_B, "MXFP4 tensor rows 0..1023")
    tasks["mxfp4_pack"] = ([lambda b=b: oracle.mxfp4_quant(b) for b in rs], a.size * PACK_F32_B,
                           "MXFP4 tensor rows 0..1023")
    out = {}
    with ThreadPoolExecutor(threads) as pool:
        for name, (fns, nbytes, sample) in tasks.items():
            t0 = time.perf_counter()
            for fn in fns:
                fn()
            t1 = time.perf_counter() - t0
            t0 = time.perf_counter()
            list(pool.map(lambda fn: fn(), fns))
            tn = time.perf_counter() - t0
            out[name] = {"gbs_1_thread": round(nbytes / t1 / 1e9, 4), f"gbs_{threads}_threads": round(nbytes / tn / 1e9, 4),
                         "sample": sample}
    return out


def gemm_oracle_times():
    """The binary64 GEMM oracle (numpy BLAS on all cores) on the 256 x 512 x 512
    forward and on the 8192 x 14336 x 4096 dense forward, operands quantized by
    the quant oracle first (not timed)."""
    import mxq_inputs
    import oracle
    res = {}
    for tag, (Mg, Ng, Kg) in (("fwd_256x512x512", (256, 512, 512)), ("fwd_8192x14336x4096", (8192, 14336, 4096))):
        xg, wg, _ = mxq_inputs.linear_inputs(Mg, Ng, Kg, seed=0)
        qx, sx = oracle.mxfp8_quant_rows(xg)
        qw, sw = oracle.mxfp8_quant_rows(wg)
        t0 = time.perf_counter()
        oracle.gemm_ref(qx, sx, qw, sw)
        dt = time.perf_counter() - t0
        res[tag] = {"seconds": round(dt, 4), "gflops": round(2 * Mg * Ng * Kg / dt / 1e9, 2)}
        del qx, sx, qw, sw, xg, wg
    return res


def run_cpu_baseline(host_inputs, steps: int):
    t0 = time.perf_counter()
    flop = 0
    for _ in range(steps):
        flop += cpu_sample_step(host_inputs)
    dt = time.perf_counter() - t0
    cores = cpu_cores()
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": (f"{steps} x [first {CPU_ROWS} rows of the dense layer (Y, dX rows + their dW part, full W), "
                       f"first {CPU_ROWS} MoE rows with their experts' full weights, {CPU_ROWS} rows of the MXFP4 "
                       "tensor]; C oracle single-threaded, binary64 numpy GEMMs on all cores"),
            "seconds": round(dt, 3), "cpu_model": cpu_model(),
            "quant_oracle": quant_oracle_rates(host_inputs, cores),
            "gemm_oracle": gemm_oracle_times()}


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
    ap.add_argument("--ncu-case", choices=["mxfp4", "dense", "moe_small", "dualquant"],
                    help="instead of the step: run one small profiling case once (for ncu captures) and exit")
    args = ap.parse_args()
    world, rank, local = dist_init()

    if args.quant_sweep:
        quant_sweep()
        return
    if args.ncu_case:
        ncu_case(args.ncu_case)
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

    peaks, peak_kind = read_peaks()
    # The timed region's length picks the tensor peak: a region under a second
    # runs at full clock (the burst cuBLAS figure), a longer one settles under
    # the power cap (the sustained figure).
    burst = elapsed < 1.0
    bf16_peak = float(peaks["bf16_tflops"] if burst else peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    fp8_peak = FP8_PER_BF16 * bf16_peak
    achieved = gemm_flop / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    value = world * STEP_FLOP * args.steps / elapsed / 1e12
    per_launch = []
    for name, (ms_sum, n) in per_kind.items():
        f = next(fl for nm, _, _, fl in ev if nm == name)
        ms = ms_sum / n
        tf = f / (ms / 1e3) / 1e12
        per_launch.append({"name": name, "flop": int(f), "ms": round(ms, 4), "achieved": round(tf, 1),
                           "frac": round(tf / fp8_peak, 3)})

    # ---- every kernel on its own (outside the timed region, same inputs)
    comp, kernels = component_timings(wl, {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"]})
    cfg1 = cfg1_latency(dev)

    # ---- end to end through the public API with host buffers
    e2e = E2EPipeline(wl)
    hb_in, hb_out = e2e.bytes()
    for _ in range(2):
        e2e.step()
    e2e_t = e2e.timed(args.e2e_steps, world)
    e2e_t = max_over_ranks(e2e_t, world)
    e2e.restore()
    assert m.mxq_poll_device_error() == 0

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(elapsed / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded: N(0,1) X, N(0,0.02) W, N(0,1e-3) dY; Dirichlet(0.5) groups; t(3) MXFP4 input)",
        "config": {"workload": WORKLOAD, "mode": args.mode, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (step touches > 8 GB); kernels alone rotate buffer sets > 2x L2",
                   "step_gemm_flop": STEP_FLOP},
        "roofline": {"bound": "tensor",
                     "kernel": "k_gemm<1,MXF8,0> (tcgen05 kind::mxf8f6f4.block_scale, 128x256 tiles, 8 epilogue warps)",
                     "achieved": round(achieved, 1) if achieved else None,
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / fp8_peak, 4) if achieved else None,
                     "peak_source": (f"{peak_kind}: 2 x bf16_tflops{'' if burst else '_sustained'} "
                                     f"(nominal fp8/bf16 ratio; timed region {elapsed:.3f} s "
                                     f"{'< 1 s at full clock: burst' if burst else '>= 1 s: sustained'})"),
                     "launches_timed": len(ev), "per_launch": per_launch, "traffic": gemm_traffic(per_kind),
                     "traffic_unit": "bytes per launch", "kernel_source": gemm_source_hash()},
        "e2e": {"value": round(world * STEP_FLOP * args.e2e_steps / e2e_t / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": hb_in, "d2h_bytes_per_step": hb_out,
                "ms_per_step": round(e2e_t / args.e2e_steps * 1e3, 3)},
        "gpu_launches": wl.launches() * args.steps,
        "clocks": clk,
        "per_kernel": kernels,
        "cfg1_latency": cfg1,
        "components": {**comp, "gemm_ms_per_launch": {k: round(v[0] / v[1], 4) for k, v in per_kind.items()}},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = run_cpu_baseline(host_inputs, args.cpu_steps)
        cb["value"] = float(f"{cb['value']:.4g}")
        for k in kernels:  # the oracle's rate for the same kernel, where it was timed
            if k["name"] in cb["quant_oracle"]:
                k["oracle"] = cb["quant_oracle"][k["name"]]
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)


def ncu_case(case: str):
    """One launch of each kernel of a small case, for profiler captures that
    must end quickly (a few hundred MB on the device, no timing loop):
      mxfp4      QDQ, clipped-STE forward and backward, packed quant of the
                 4096 x 4096 fp32 tensor, then the W4A4 QAT forward
                 (8192 x 14336 x 4096: its two operand quants and the GEMM) and
                 the bf16 QDQ of its 14336 x 4096 weight;
      dense      row quants and one forward GEMM, 8192 x 14336 x 4096;
      moe_small  the MoE layer's GEMMs (fwd, dX, dW) at E=8, T=8192, K=7168,
                 N=4096 (the bench's 1024 routed rows per expert on average);
      dualquant  the dual quant of the dense layer's dY (8192 x 14336) and the
                 per-group dual quant, with per-group padded row scales, of the
                 MoE layer's dY (32768 x 4096, 32 Dirichlet(0.5) groups)."""
    import mxq_inputs
    import mx_block_scaled_mxq_gb300 as m
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    m.load()
    bf = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=dev)  # noqa: E731
    u8 = lambda n: torch.empty(max(int(n), 1), dtype=torch.uint8, device=dev)  # noqa: E731
    if case == "mxfp4":
        R, C = FP4["R"], FP4["C"]
        a4 = torch.from_numpy(mxq_inputs.mxfp4_large(R, C, seed=0)).to(dev)
        y4, g4 = torch.empty_like(a4), torch.empty_like(a4)
        mk = torch.empty((R, C // 32), dtype=torch.int32, device=dev)
        m.mxq_qdq_mxfp4(a4, y4, R, C, 32, 6.0)
        m.mxq_mxfp4_ste_forward(a4, y4, mk, R, C, 32, 6.0)
        m.mxq_mxfp4_ste_backward(y4, mk, R, C, g4)
        m.mxq_quantize(a4, m.F32, R, C, C, -1, m.E2M1, 0, u8(R * C // 2), u8(m.mxq_scale_bytes(R, C // 32)), None, None)
        M, N, K = LIN["M"], LIN["N"], LIN["K"]
        x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=0)
        x, w = x.to(dev), w.to(dev)
        wsb = m.mxq_qat_linear_workspace_bytes(M, N, K, 1)
        m.mxq_qat_linear_fwd(x, w, None, M, N, K, 1, 6.0, bf(M, N), u8(wsb), wsb)
        m.mxq_qdq_mxfp4_bf16(w, bf(N, K), N, K, 32, 6.0)
    elif case == "dualquant":
        M, N, K = LIN["M"], LIN["N"], LIN["K"]
        _, _, dy = mxq_inputs.linear_inputs(M, N, K, seed=0)
        m.quantize_mxfp8(dy.to(dev), dual=True)
        E, T, Nm = MOE["E"], MOE["T"], MOE["N"]
        off = mxq_inputs.offsets_from_sizes(mxq_inputs.dirichlet_group_sizes(E, T, seed=0))
        off_d = torch.from_numpy(np.asarray(off, dtype=np.int64)).to(dev)
        dym = mxq_inputs.normal_bf16((T, Nm), 1e-3, seed=5).to(dev)
        tp = m.mxq_grouped_padded_rows(T, E)
        m.mxq_quantize_grouped_dual_padded(dym, T, Nm, off_d, E, tp, u8(T * Nm), u8(m.mxq_scale_bytes(tp, Nm // 32)),
                                           u8(Nm * tp), u8(m.mxq_scale_bytes(Nm, tp // 32)))
    elif case == "dense":
        M, N, K = LIN["M"], LIN["N"], LIN["K"]
        x, w, _ = mxq_inputs.linear_inputs(M, N, K, seed=0)
        xq, xs = m.quantize_mxfp8(x.to(dev))[:2]
        wq, ws = m.quantize_mxfp8(w.to(dev))[:2]
        m.mxq_gemm(xq, xs, wq, ws, M, N, K, bf(M, N), N)
    else:
        E, T, K, N = 8, 8192, MOE["K"], MOE["N"]
        off, xm, wm, dym = mxq_inputs.moe_inputs(E, T, K, N, seed=0)
        d_off = torch.from_numpy(off).to(dev)
        tp = m.mxq_grouped_padded_rows(T, E)
        xmd, dymd = xm.to(dev), dym.to(dev)
        wq, ws, wqT, wsT = m.quantize_mxfp8(wm.reshape(E * N, K).to(dev), dual=True)
        xq, xs, xqT, xsT = u8(T * K), u8(m.mxq_scale_bytes(tp, K // 32)), u8(K * tp), u8(m.mxq_scale_bytes(K, tp // 32))
        dq, ds, dqT, dsT = u8(T * N), u8(m.mxq_scale_bytes(tp, N // 32)), u8(N * tp), u8(m.mxq_scale_bytes(N, tp // 32))
        m.mxq_quantize_grouped_dual_padded(xmd, T, K, d_off, E, tp, xq, xs, xqT, xsT)
        m.mxq_quantize_grouped_dual_padded(dymd, T, N, d_off, E, tp, dq, ds, dqT, dsT)
        m.mxq_grouped_gemm(m.GG_FWD, xq, xs, wq, ws, d_off, E, T, N, K, tp, bf(T, N))
        m.mxq_grouped_gemm(m.GG_DX, dq, ds, wqT, wsT, d_off, E, T, N, K, tp, bf(T, K))
        m.mxq_grouped_gemm(m.GG_DW, dqT, dsT, xqT, xsT, d_off, E, T, N, K, tp, bf(E, N, K))
    torch.cuda.synchronize()
    assert m.mxq_poll_device_error() == 0
    print(json.dumps({"ncu_case": case, "ok": True}), flush=True)


def quant_sweep():
    """Dual-axis MXFP8 quant of bf16 [R x C], C in {2048, 7168, 14336},
    R = ceil128(2^p / C) for p = 20, 22, ..., 30; algorithmic bytes 2 in +
    2 (1 + 1/32) out per element; back-to-back calls rotating over buffer sets
    that together exceed twice L2."""
    import mxq_inputs
    import mx_block_scaled_mxq_gb300 as m
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    m.load()
    peaks, peak_kind = read_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    for C in (2048, 7168, 14336):
        for p in range(20, 31, 2):
            R = ((1 << p) // C + 127) // 128 * 128
            sets = copies_past_l2(int(R * C * 4.0625))
            fns = []
            for j in range(sets):
                x = mxq_inputs.sweep_bf16_device(R, C, seed=p * 100 + C, device=dev)
                q, sc, qT, sT = (torch.empty(R * C, dtype=torch.uint8, device=dev),
                                 torch.empty(m.mxq_scale_bytes(R, C // 32), dtype=torch.uint8, device=dev),
                                 torch.empty(R * C, dtype=torch.uint8, device=dev),
                                 torch.empty(m.mxq_scale_bytes(C, R // 32), dtype=torch.uint8, device=dev))
                fns.append(lambda x=x, q=q, sc=sc, qT=qT, sT=sT:
                           m.mxq_quantize(x, m.BF16, R, C, C, -1, m.E4M3, 1, q, sc, qT, sT))
            ms = time_rotating(fns, reps=max(2, 16 // sets))
            gbs = R * C * 4.0625 / (ms / 1e3) / 1e9
            print(json.dumps({"sweep": "mxfp8_dual_quant", "rows": R, "cols": C, "elements": R * C,
                              "buffer_sets": sets, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                              "frac": round(gbs / hbm, 3),
                              "peak": f"{hbm} GB/s ({peak_kind} HBM copy)"}), flush=True)
            del fns
            torch.cuda.empty_cache()
    assert m.mxq_poll_device_error() == 0


# Algorithmic bytes per element of each quant kernel (reads of the input,
# writes of codes and E8M0 scales; swz padding not counted).
ROW_QUANT_B = 2 + (1 + 1 / 32)            # bf16 -> E4M3 codes + scales
DUAL_QUANT_B = 2 + 2 * (1 + 1 / 32)       # one read, row and column outputs
QDQ_F32_B = 8                             # fp32 in, fp32 out
STE_B = 8 + 1 / 8                         # fp32 in/out + one mask bit
PACK_F32_B = 4 + 1 / 2 + 1 / 32           # fp32 in, nibbles + scales out
QDQ_BF16_B = 4                            # bf16 in, bf16 out


def component_timings(wl, peaks):
    """Every kernel of the step timed on its own, back to back over buffer
    sets larger than L2 (time_rotating); returns (flat ms/throughput dict,
    per-kernel roofline entries)."""
    m = wl.m
    dev = wl.dev
    M, N, K = LIN["M"], LIN["N"], LIN["K"]
    E, T, Km, Nm = MOE["E"], MOE["T"], MOE["K"], MOE["N"]
    R4, C4 = FP4["R"], FP4["C"]
    hbm = float(peaks["hbm_gbs"])
    tensor_peak = FP8_PER_BF16 * float(peaks["bf16_tflops"])
    u8 = lambda n: torch.empty(max(int(n), 1), dtype=torch.uint8, device=dev)  # noqa: E731
    bf = lambda *sh: torch.empty(sh, dtype=torch.bfloat16, device=dev)  # noqa: E731
    out, entries = {}, []

    def hbm_entry(name, kernel, nbytes, ms, note=""):
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name + "_ms"] = round(ms, 4)
        out[name + "_gbs"] = round(gbs, 1)
        entries.append({"name": name, "kernel": kernel, "bound": "hbm", "bytes": int(nbytes), "ms": round(ms, 4),
                        "achieved": round(gbs, 1), "unit": "GB/s", "peak": hbm, "frac": round(gbs / hbm, 3),
                        **({"note": note} if note else {})})

    def tensor_entry(name, kernel, flop, ms, note=""):
        tf = flop / (ms / 1e3) / 1e12
        out[name + "_ms"] = round(ms, 4)
        out[name + "_tflops"] = round(tf, 1)
        entries.append({"name": name, "kernel": kernel, "bound": "tensor", "flop": int(flop), "ms": round(ms, 4),
                        "achieved": round(tf, 1), "unit": "TFLOP/s", "peak": round(tensor_peak, 1),
                        "frac": round(tf / tensor_peak, 3), **({"note": note} if note else {})})

    # ---- MXFP8 quant kernels
    def dual_set(x, R, C):
        q, sc, qT, sT = u8(R * C), u8(m.mxq_scale_bytes(R, C // 32)), u8(R * C), u8(m.mxq_scale_bytes(C, R // 32))
        return lambda: m.mxq_quantize(x, m.BF16, R, C, C, -1, m.E4M3, 1, q, sc, qT, sT)

    ms = time_rotating([dual_set(wl.dy, M, N) for _ in range(2)])
    hbm_entry("dual_quant_dY", "k_quant_cols_tma<1,0,1,0>", M * N * DUAL_QUANT_B, ms)
    ms = time_rotating([dual_set(wl.w, N, K) for _ in range(2)])
    hbm_entry("dual_quant_W", "k_quant_cols_tma<1,0,1,0>", N * K * DUAL_QUANT_B, ms)

    def row_set(x, R, C):
        q, sc = u8(R * C), u8(m.mxq_scale_bytes(R, C // 32))
        return lambda: m.mxq_quantize(x, m.BF16, R, C, C, -1, m.E4M3, 0, q, sc, None, None)

    ms = time_rotating([row_set(wl.xm, T, Km)])
    hbm_entry("row_quant_moe_X", "k_quant_cols_tma<1,0,0,0>", T * Km * ROW_QUANT_B, ms)
    tp = wl.t_pad

    def gdual_set(x, C):
        q, sc = u8(T * C), u8(m.mxq_scale_bytes(tp, C // 32))
        qT, sT = u8(C * tp), u8(m.mxq_scale_bytes(C, tp // 32))
        return lambda: m.mxq_quantize_grouped_dual_padded(x, T, C, wl.off, E, tp, q, sc, qT, sT)

    padded = int(wl.off_padded_total)
    for name, x, C in (("grouped_dual_quant_moe_X", wl.xm, Km), ("grouped_dual_quant_moe_dY", wl.dym, Nm)):
        ms = time_rotating([gdual_set(x, C)])
        nbytes = T * C * (2 + 1) + padded * C / 32 + C * padded * (1 + 1 / 32)
        hbm_entry(name, "k_quant_cols_tma<1,1,1,0>", nbytes, ms,
                  note="row scales and column output counted over the groups' padded length")

    # ---- MXFP4 kernels on the 4096 x 4096 fp32 tensor
    nset = copies_past_l2(R4 * C4 * 8)
    xs4 = [wl.a4.clone() for _ in range(nset)]
    ys4 = [torch.empty_like(wl.a4) for _ in range(nset)]
    ms4 = [torch.empty((R4, C4 // 32), dtype=torch.int32, device=dev) for _ in range(nset)]
    ms = time_rotating([lambda i=i: m.mxq_qdq_mxfp4(xs4[i], ys4[i], R4, C4, 32, 6.0) for i in range(nset)])
    hbm_entry("mxfp4_qdq", "k_qdq_mxfp4_vec<0>", R4 * C4 * QDQ_F32_B, ms)
    ms = time_rotating([lambda i=i: m.mxq_mxfp4_ste_forward(xs4[i], ys4[i], ms4[i], R4, C4, 32, 6.0)
                        for i in range(nset)])
    hbm_entry("mxfp4_ste_fwd", "k_qdq_mxfp4_vec<1>", R4 * C4 * STE_B, ms)
    ms = time_rotating([lambda i=i: m.mxq_mxfp4_ste_backward(ys4[i], ms4[i], R4, C4, xs4[(i + 1) % nset])
                        for i in range(nset)])
    hbm_entry("mxfp4_ste_bwd", "k_ste_backward_vec", R4 * C4 * STE_B, ms)
    for i in range(nset):
        xs4[i].copy_(wl.a4)
    p4 = [u8(R4 * C4 // 2) for _ in range(nset)]
    s4 = [u8(m.mxq_scale_bytes(R4, C4 // 32)) for _ in range(nset)]
    ms = time_rotating([lambda i=i: m.mxq_quantize(xs4[i], m.F32, R4, C4, C4, -1, m.E2M1, 0, p4[i], s4[i], None, None)
                        for i in range(nset)])
    hbm_entry("mxfp4_pack", "k_quant_rows<float,1>", R4 * C4 * PACK_F32_B, ms)
    del xs4, ys4, ms4, p4, s4
    wq4 = [bf(N, K) for _ in range(2)]
    ms = time_rotating([lambda i=i: m.mxq_qdq_mxfp4_bf16(wl.w, wq4[i], N, K, 32, 6.0) for i in range(2)])
    hbm_entry("mxfp4_qdq_bf16_W", "k_qdq_mxfp4_bf16", N * K * QDQ_BF16_B, ms)
    del wq4

    # ---- GEMMs alone (operands quantized once, two sets where they fit in L2)
    def lin_ops(j):
        xq, xsc, xqT, xsT = m.quantize_mxfp8(wl.x, dual=True)
        wq_, wsc, wqT, wsT = m.quantize_mxfp8(wl.w, dual=True)
        dq, dsc, dqT, dsT = m.quantize_mxfp8(wl.dy, dual=True)
        return dict(xq=xq, xs=xsc, xqT=xqT, xsT=xsT, wq=wq_, ws=wsc, wqT=wqT, wsT=wsT, dq=dq, ds=dsc, dqT=dqT,
                    dsT=dsT)
    ops = [lin_ops(j) for j in range(2)]
    y2 = [bf(M, N) for _ in range(2)]
    fl = 2 * M * N * K
    ms = time_rotating([lambda o=o, y=y: m.mxq_gemm(o["xq"], o["xs"], o["wq"], o["ws"], M, N, K, y, N)
                        for o, y in zip(ops, y2)])
    tensor_entry("dense_fwd_gemm", "k_gemm<1,MXF8,0>", fl, ms)
    dx2 = [bf(M, K) for _ in range(2)]
    ms = time_rotating([lambda o=o, d=d: m.mxq_gemm(o["dq"], o["ds"], o["wqT"], o["wsT"], M, K, N, d, K)
                        for o, d in zip(ops, dx2)])
    tensor_entry("dense_dx_gemm", "k_gemm<1,MXF8,0>", fl, ms)
    dw2 = [bf(N, K) for _ in range(2)]
    ms = time_rotating([lambda o=o, d=d: m.mxq_gemm(o["dqT"], o["dsT"], o["xqT"], o["xsT"], N, K, M, d, K)
                        for o, d in zip(ops, dw2)])
    tensor_entry("dense_dw_gemm", "k_gemm<1,MXF8,0>", fl, ms)
    del ops, y2, dx2, dw2
    gf = 2 * T * Nm * Km
    ms = time_rotating([lambda: m.mxq_grouped_gemm(m.GG_FWD, wl.xmq, wl.xms, wl.wmq, wl.wms, wl.off, E, T, Nm, Km,
                                                   wl.t_pad, wl.ym)])
    tensor_entry("moe_fwd_gemm", "k_gemm<1,MXF8,0> grouped rows", gf, ms)
    ms = time_rotating([lambda: m.mxq_grouped_gemm(m.GG_DX, wl.dymq, wl.dyms, wl.wmqT, wl.wmsT, wl.off, E, T, Nm, Km,
                                                   wl.t_pad, wl.dxm)])
    tensor_entry("moe_dx_gemm", "k_gemm<1,MXF8,0> grouped rows", gf, ms)
    ms = time_rotating([lambda: m.mxq_grouped_gemm(m.GG_DW, wl.dymqT, wl.dymsT, wl.xmqT, wl.xmsT, wl.off, E, T, Nm,
                                                   Km, wl.t_pad, wl.dwm)])
    tensor_entry("moe_dw_gemm", "k_gemm<1,MXF8,0> grouped K", gf, ms)

    # ---- layer-level pieces (single set; each call touches > 1 GB)
    qat_ws_bytes = max(m.mxq_qat_linear_workspace_bytes(M, N, K, 1), m.mxq_qat_linear_workspace_bytes(M, N, K, 0))
    qat_ws = u8(qat_ws_bytes)
    wc_bytes = m.mxq_linear_weight_cache_bytes(N, K)
    wcache = u8(wc_bytes)
    mode = wl.mode

    def layer_plain():
        m.mxq_linear_fwd(wl.x, wl.w, M, N, K, mode, wl.lctx, wl.y, wl.lws, wl.lwsb)
        m.mxq_linear_bwd_dx(wl.dy, wl.w, M, N, K, mode, wl.lctx, wl.dx, wl.lws, wl.lwsb)
        m.mxq_linear_bwd_dw(wl.dy, wl.x, M, N, K, mode, wl.lctx, wl.dw, wl.lws, wl.lwsb)

    def layer_wq():  # one micro-batch with W's quantization taken from the cache
        m.mxq_linear_fwd_wq(wl.x, wcache, M, N, K, mode, wl.lctx, wl.y, wl.lws, wl.lwsb)
        m.mxq_linear_bwd_dx_wq(wl.dy, wcache, M, N, K, mode, wl.lctx, wl.dx, wl.lws, wl.lwsb)
        m.mxq_linear_bwd_dw(wl.dy, wl.x, M, N, K, mode, wl.lctx, wl.dw, wl.lws, wl.lwsb)

    m.mxq_linear_quantize_weight(wl.w, N, K, wcache, wc_bytes)
    parts = {
        "linear_fwd": lambda: m.mxq_linear_fwd(wl.x, wl.w, M, N, K, mode, wl.lctx, wl.y, wl.lws, wl.lwsb),
        "linear_bwd_dx": lambda: m.mxq_linear_bwd_dx(wl.dy, wl.w, M, N, K, mode, wl.lctx, wl.dx, wl.lws, wl.lwsb),
        "linear_bwd_dw": lambda: m.mxq_linear_bwd_dw(wl.dy, wl.x, M, N, K, mode, wl.lctx, wl.dw, wl.lws, wl.lwsb),
        "linear_layer": layer_plain,
        "linear_wq": layer_wq,
        "linear_weight_quant": lambda: m.mxq_linear_quantize_weight(wl.w, N, K, wcache, wc_bytes),
        "qat_linear_fwd_w4a4": lambda: m.mxq_qat_linear_fwd(wl.x, wl.w, None, M, N, K, 1, 6.0, wl.y, qat_ws,
                                                            qat_ws_bytes),
        "qat_linear_fwd_w4a16": lambda: m.mxq_qat_linear_fwd(wl.x, wl.w, None, M, N, K, 0, 6.0, wl.y, qat_ws,
                                                             qat_ws_bytes),
    }
    for name, fn in parts.items():
        out[name + "_ms"] = round(time_rotating([fn], reps=5), 4)
    layer_parts = [name for name in ("linear_fwd", "linear_bwd_dx", "linear_bwd_dw")]
    out["linear_tflops"] = round(LIN_FLOP / (sum(out[n + "_ms"] for n in layer_parts) / 1e3) / 1e12, 1)
    out["qat_linear_fwd_w4a4_tflops"] = round(fl / (out["qat_linear_fwd_w4a4_ms"] / 1e3) / 1e12, 1)
    out["qat_linear_fwd_w4a16_tflops"] = round(fl / (out["qat_linear_fwd_w4a16_ms"] / 1e3) / 1e12, 1)
    # the W4A4 forward is two MXFP4-as-E4M3 quants (X, W) and the dense GEMM
    # above: its quant rate, derived from the two timings
    w4a4_quant_ms = out["qat_linear_fwd_w4a4_ms"] - out["dense_fwd_gemm_ms"]
    if w4a4_quant_ms > 0:
        hbm_entry("w4a4_operand_quant", "k_quant_cols_tma<1,0,0,2> (x2, derived)", (M + N) * K * ROW_QUANT_B,
                  w4a4_quant_ms, note="W4A4 forward time minus the dense forward GEMM time")
    # the other linear mode on the same buffers
    other = m.RECOMPUTE if mode == m.SAVE_QUANT else m.SAVE_QUANT
    need_ws = m.mxq_linear_workspace_bytes(M, N, K, other)
    ctx, ws = u8(m.mxq_linear_ctx_bytes(M, N, K, other)), u8(need_ws)

    def layer_other():
        m.mxq_linear_fwd(wl.x, wl.w, M, N, K, other, ctx, wl.y, ws, need_ws)
        m.mxq_linear_bwd_dx(wl.dy, wl.w, M, N, K, other, ctx, wl.dx, ws, need_ws)
        m.mxq_linear_bwd_dw(wl.dy, wl.x, M, N, K, other, ctx, wl.dw, ws, need_ws)
    name = "recompute" if other == m.RECOMPUTE else "save"
    out[f"linear_{name}_ms"] = round(time_rotating([layer_other], reps=5), 4)
    out["linear_saved_bytes"] = {"save": m.mxq_linear_saved_bytes(M, N, K, m.SAVE_QUANT),
                                 "recompute": m.mxq_linear_saved_bytes(M, N, K, m.RECOMPUTE)}
    del ctx, ws, qat_ws, wcache
    # the MoE layer through its orchestration entry points, both modes
    E, T, Km, Nm = MOE["E"], MOE["T"], MOE["K"], MOE["N"]
    for gmode, tag in ((m.SAVE_QUANT, "save"), (m.RECOMPUTE, "recompute")):
        gctx = u8(m.mxq_grouped_linear_ctx_bytes(T, E, Nm, Km, gmode))
        gwsb = m.mxq_grouped_linear_workspace_bytes(T, E, Nm, Km, gmode)
        gws = u8(gwsb)

        def moe_layer(gmode=gmode, gctx=gctx, gws=gws, gwsb=gwsb):
            m.mxq_grouped_linear_fwd(wl.xm, wl.wm, wl.off, E, T, Nm, Km, gmode, gctx, wl.ym, gws, gwsb)
            m.mxq_grouped_linear_bwd_dx(wl.dym, wl.wm, wl.off, E, T, Nm, Km, gmode, gctx, wl.dxm, gws, gwsb)
            m.mxq_grouped_linear_bwd_dw(wl.dym, wl.xm, wl.off, E, T, Nm, Km, gmode, gctx, wl.dwm, gws, gwsb)
        ms = time_rotating([moe_layer], reps=3)
        out[f"moe_layer_{tag}_ms"] = round(ms, 4)
        out[f"moe_layer_{tag}_tflops"] = round(3 * 2 * T * Nm * Km / (ms / 1e3) / 1e12, 1)
        del gctx, gws
    out["moe_layer_saved_bytes"] = {"save": m.mxq_grouped_linear_saved_bytes(T, E, Nm, Km, m.SAVE_QUANT),
                                    "recompute": m.mxq_grouped_linear_saved_bytes(T, E, Nm, Km, m.RECOMPUTE)}
    # the MXFP4 QAT forward of the MoE layer (32 experts, 32768 routed rows)
    for qi, tag in ((1, "w4a4"), (0, "w4a16")):
        gq_bytes = m.mxq_qat_grouped_fwd_workspace_bytes(T, E, Nm, Km, qi)
        gq_ws = u8(gq_bytes)
        ms = time_rotating([lambda: m.mxq_qat_grouped_fwd(wl.xm, wl.wm, wl.off, E, T, Nm, Km, qi, 6.0, wl.ym, gq_ws,
                                                          gq_bytes)], reps=5)
        out[f"qat_grouped_fwd_{tag}_ms"] = round(ms, 4)
        out[f"qat_grouped_fwd_{tag}_tflops"] = round(2 * T * Nm * Km / (ms / 1e3) / 1e12, 1)
        del gq_ws
    torch.cuda.empty_cache()
    return out, entries


def cfg1_latency(dev):
    """The 256 x 512 x 512 MXFP8 linear forward (row quant of X and W, then the
    GEMM; 3 launches): per-call device time back to back, host-to-completion
    time of one call, and the time per forward replayed from a CUDA graph."""
    import mx_block_scaled_mxq_gb300 as m
    import mxq_inputs
    M1, N1, K1 = 256, 512, 512
    x, w, _ = mxq_inputs.linear_inputs(M1, N1, K1, seed=0)
    x, w = x.to(dev), w.to(dev)
    mode = m.RECOMPUTE
    ctx = torch.empty(max(m.mxq_linear_ctx_bytes(M1, N1, K1, mode), 1), dtype=torch.uint8, device=dev)
    wsb = m.mxq_linear_workspace_bytes(M1, N1, K1, mode)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    y = torch.empty((M1, N1), dtype=torch.bfloat16, device=dev)
    fn = lambda: m.mxq_linear_fwd(x, w, M1, N1, K1, mode, ctx, y, ws, wsb)  # noqa: E731
    for _ in range(20):
        fn()
    torch.cuda.synchronize()
    n = 500
    back_to_back = time_steps(fn, n, 1) / n * 1e6
    single = []
    for _ in range(100):
        t0 = time.perf_counter()
        fn()
        torch.cuda.synchronize()
        single.append((time.perf_counter() - t0) * 1e6)
    single.sort()
    res = {"shape": "X 256x512, W 512x512 bf16 -> Y 256x512 (row quant x2 + GEMM)",
           "us_per_fwd_back_to_back": round(back_to_back, 2), "us_single_call_median": round(single[50], 2)}
    try:
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for _ in range(50):
                fn()
        g.replay()
        torch.cuda.synchronize()
        res["us_per_fwd_graph_replay"] = round(time_steps(g.replay, 20, 1) / (20 * 50) * 1e6, 2)
    except Exception as exc:  # capture refused: report without the graph figure
        res["graph_replay_error"] = str(exc)[:200]
    return res


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
