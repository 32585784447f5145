"""Benchmark: row-wise normalization forward + backward on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl mine|reference]

A step is one forward and one backward of the workload's op (every stage of the path:
row load, reduction, statistics, apply, backward row pass, dgamma/dbeta partials and
their fixed-order reduction) on device-resident inputs. The metric is achieved HBM
throughput: compulsory bytes (fp16 activations read and written once, fp32 stats and
parameter gradients) divided by the CUDA-event time of a step, plus rows/s.
Steps run back to back with no flush: the forward of step s uses buffer set s % n and
its backward set (s + 1) % n, with n = 2 when one set exceeds L2 and more for smaller
workloads (the n sets together hold at least three times L2), so no call finds in L2
the rows an earlier call touched, and each call pays for the write-backs the previous
one left behind. Events
mark only the start and the end of the K timed steps (an event between two calls would
stop the second from being scheduled while the first drains, which a training loop
does not do). Each call's own time (the roofline entries) comes from a separate loop of
that call alone, back to back, timed the same way.

One JSON line is printed by rank 0. Under torchrun (N > 1) every rank runs its own
replica of the workload (weak scaling; the path has no cross-rank exchange in this
build) and the time is the max over ranks.

``--impl reference`` times the fp64 CPU oracle instead, on host cores, over a bounded
row sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = ("achieved HBM GB/s (% of ~8 TB/s) and rows/s, norm fwd+bwd at N×D fp16")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
# The headline is the largest workload that fits one GPU: the fused residual-add + RMSNorm
# over 32768 x 4096 (about 1.07 GB read and written per direction).
DEFAULT_WORKLOAD = "add_rmsnorm_32768x4096"
# The three large workloads the >= 80 % bar applies to; each gets its own roofline block.
GATED_WORKLOADS = ["rmsnorm_16384x4096", "add_rmsnorm_32768x4096", "layernorm_2048x16384"]
LARGE_WORKLOADS = GATED_WORKLOADS + ["rmsnorm_4096x32768", "layernorm_1024x131072"]

# The kernels each call of a workload launches (fp16 storage), for the roofline blocks.
# The backward is one user-visible call: the row kernel then the fixed-order reduction.
KERNELS = {
    ("rmsnorm_16384x4096", "forward"): ["norm_fwd_packed_kernel"],
    ("rmsnorm_16384x4096", "backward"): ["norm_bwd_pipe_kernel", "param_reduce_kernel"],
    ("add_rmsnorm_32768x4096", "forward"): ["norm_fwd_vec8_kernel"],
    ("add_rmsnorm_32768x4096", "backward"): ["norm_bwd_pipe_kernel", "param_reduce_kernel"],
    ("layernorm_2048x16384", "forward"): ["norm_fwd_packed_kernel"],
    ("layernorm_2048x16384", "backward"): ["norm_bwd_pipe_kernel", "param_reduce_kernel"],
    ("rmsnorm_4096x32768", "forward"): ["norm_fwd_stream_kernel"],
    ("rmsnorm_4096x32768", "backward"): ["norm_bwd_pipe_kernel (2-CTA clusters)",
                                         "param_reduce_kernel"],
    ("layernorm_1024x131072", "forward"): ["norm_fwd_stream_kernel"],
    ("layernorm_1024x131072", "backward"): ["norm_bwd_pipe_kernel (8-CTA clusters)",
                                            "param_reduce_kernel"],
}
CSRC = os.path.join(ROOT, "row_wise_rmsnorm_gb300", "csrc")


# --------------------------------------------------------------- helpers ---

def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs, copy, burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def _code_only(text: str) -> str:
    """C++/CUDA source with comments and blank space removed (the sources hold no "//" or
    "/*" inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of the code the normalization kernels are built from, comments and blank space
    left out (the softmax, cross-entropy and norm + GEMV sources are left out too: they do
    not change these kernels)."""
    h = hashlib.sha256()
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh")) and not f.startswith(("softmax", "gemv")):
            with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
                h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    entry = rec.get("entries", {}).get(f"{workload}:{kernel}")
    return None if entry is None else entry.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clock, power and clock-event reasons while the timed region runs, read through
    NVML (the library nvidia-smi itself uses; read-only queries) every millisecond from a
    background thread, plus one synchronous sample as soon as the timed work is enqueued
    (`mark()`), so that even a region of a few milliseconds carries its own clock record.
    The main thread enqueues the timed calls in Python and holds the interpreter lock
    between them; at the default 5 ms switch interval the sampler would get one turn in
    five periods, so the interval is lowered to a quarter period while sampling and
    restored afterwards. Falls back to `nvidia-smi -lms 200` when NVML cannot be loaded."""
    REASONS = ((0x8, "hw_slowdown"), (0x40, "hw_thermal_slowdown"),
               (0x20, "sw_thermal_slowdown"), (0x4, "sw_power_cap"))
    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device, period_s: float = 0.001):
        self.device = device
        self.period = period_s
        self.rows = []
        self.nvml = None
        self.handle = None
        self.proc = None
        self.source = None

    # -- NVML through ctypes
    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.device).uuid)
            key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            ok = lib.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(h)) == 0
        except Exception:  # noqa: BLE001 - any failure falls back to the index
            ok = False
        if not ok:
            idx = self.device.index or 0
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            ids = [v for v in vis.split(",") if v.strip().isdigit()]
            if idx < len(ids):
                idx = int(ids[idx])
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) == 0
        if not ok:
            return False
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.nvml, self.handle = lib, h
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        self.max_mhz = mx.value
        return True

    def sample(self, tag="thread"):
        import ctypes
        if self.nvml is None:
            return
        sm, pw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(sm)) != 0:
            return
        self.nvml.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(pw))
        self.reasons_fn(self.handle, ctypes.byref(rs))
        self.rows.append(dict(t=time.perf_counter(), sm=float(sm.value), smax=float(self.max_mhz),
                              power=pw.value / 1000.0, mask=int(rs.value), tag=tag))

    def mark(self):
        """One synchronous sample (call right after enqueuing the timed work)."""
        self.sample("sync")

    def _loop(self):
        while not self._stop.is_set():
            self.sample()
            self._stop.wait(self.period)

    def __enter__(self):
        import threading
        if self._open_nvml():
            self.source = "nvml, 1 ms"
            self._switch = sys.getswitchinterval()
            sys.setswitchinterval(min(self._switch, self.period / 4))
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self.t0 = time.perf_counter()
            self._thread.start()
        else:
            self.source = "nvidia-smi, 200 ms"
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.device.index or 0}",
                     f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
            self.t0 = time.perf_counter()
        return self

    def __exit__(self, *exc):
        self.t1 = time.perf_counter()
        if self.nvml is not None:
            self._stop.set()
            self._thread.join(timeout=5)
            sys.setswitchinterval(self._switch)
            self.nvml.nvmlShutdown()
            return
        out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
        for r in csv.reader(io.StringIO(out or "")):
            if len(r) < 9:
                continue
            try:
                mask = sum(bit for (bit, _), col in zip(self.REASONS, (5, 6, 7, 8))
                           if r[col].strip().lower() == "active")
                self.rows.append(dict(t=0.0, sm=float(r[1]), smax=float(r[2]), power=float(r[3]),
                                      mask=mask, tag="smi"))
            except ValueError:
                continue

    def summary(self):
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "source": self.source}
        reasons = [name for bit, name in self.REASONS if any(x["mask"] & bit for x in rows)]
        return {"sm_mhz": statistics.median(x["sm"] for x in rows),
                "sm_mhz_min": min(x["sm"] for x in rows),
                "sm_max_mhz": max(x["smax"] for x in rows),
                "power_w_max": round(max(x["power"] for x in rows), 1),
                "reasons": reasons, "samples": len(rows),
                "sync_samples": sum(1 for x in rows if x["tag"] == "sync"),
                "source": self.source}


# ------------------------------------------------------------ GPU arm ---

class OpRunner:
    """Holds one workload's device buffers and issues its forward/backward C-ABI calls.

    ``dtype`` (a torch dtype) stores every activation, parameter and cotangent in that
    type and goes through the explicit-dtype entry points; None keeps the fp16 ones."""

    def __init__(self, name: str, device, seed: int, dtype=None):
        import torch
        import row_wise_rmsnorm_gb300 as mt
        self.mt = mt
        self.w = W.WORKLOADS[name]
        self.dev = device
        w = self.w
        self.dtype = dtype
        dt = torch.float16 if dtype is None else dtype
        self.t = W.generate(w.op, w.N, w.D, device=device, seed=seed, x_kind=w.x_kind,
                            dy_std=w.dy_std, beta_std=w.beta_std, x_dtype=dt, w_dtype=dt,
                            g_dtype=dt)
        N, D = w.N, w.D
        h = dict(dtype=dt, device=device)
        f = dict(dtype=torch.float32, device=device)
        self.Y = torch.empty((N, D), **h)
        self.rstd = torch.empty(N, **f)
        self.dX = torch.empty((N, D), **h)
        self.dg = torch.empty(D, **f)
        self.mean = torch.empty(N, **f) if w.op == W.LAYERNORM else None
        self.db = torch.empty(D, **f) if w.op == W.LAYERNORM else None
        self.S = torch.empty((N, D), **h) if w.op == W.ADD_RMSNORM else None
        opcode = {W.RMSNORM: mt.MT_OP_RMSNORM, W.LAYERNORM: mt.MT_OP_LAYERNORM,
                  W.ADD_RMSNORM: mt.MT_OP_ADD_RMSNORM}[w.op]
        self.ws_bytes = mt.mt_norm_backward_workspace_size(opcode, N, D, device.index or 0)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        eb = torch.empty(0, dtype=dt).element_size()
        self.fwd_bytes = W.compulsory_bytes(w.op, "forward", N, D, xb=eb, wb=eb, gb=eb)
        self.bwd_bytes = W.compulsory_bytes(w.op, "backward", N, D, xb=eb, wb=eb, gb=eb)
        self.opcode = opcode

    def forward(self, stream):
        w, t, mt = self.w, self.t, self.mt
        if self.dtype is not None:
            c = mt.dtype_code(self.dtype)
            mt.mt_norm_forward_ex(self.opcode, c, c, t["X"], t.get("R"), t["gamma"],
                                  t.get("beta"), self.S, self.Y, self.mean, self.rstd, w.N, w.D,
                                  w.eps, stream)
            return
        if w.op == W.RMSNORM:
            mt.mt_rmsnorm_forward(t["X"], t["gamma"], self.Y, self.rstd, w.N, w.D, w.eps, stream)
        elif w.op == W.LAYERNORM:
            mt.mt_layernorm_forward(t["X"], t["gamma"], t["beta"], self.Y, self.mean, self.rstd,
                                    w.N, w.D, w.eps, stream)
        else:
            mt.mt_add_rmsnorm_forward(t["X"], t["R"], t["gamma"], self.S, self.Y, self.rstd,
                                      w.N, w.D, w.eps, stream)

    def backward(self, stream):
        w, t, mt = self.w, self.t, self.mt
        if self.dtype is not None:
            c = mt.dtype_code(self.dtype)
            x = self.S if w.op == W.ADD_RMSNORM else t["X"]
            mt.mt_norm_backward_ex(self.opcode, c, c, c, x, t["gamma"], t["dY"], t.get("dS"),
                                   self.mean, self.rstd, self.dX, self.dg, self.db, w.N, w.D,
                                   self.ws, self.ws_bytes, stream)
            return
        if w.op == W.RMSNORM:
            mt.mt_rmsnorm_backward_ws(t["X"], t["gamma"], t["dY"], self.rstd, self.dX, self.dg,
                                      w.N, w.D, self.ws, self.ws_bytes, stream)
        elif w.op == W.LAYERNORM:
            mt.mt_layernorm_backward_ws(t["X"], t["gamma"], t["dY"], self.mean, self.rstd,
                                        self.dX, self.dg, self.db, w.N, w.D, self.ws,
                                        self.ws_bytes, stream)
        else:
            mt.mt_add_rmsnorm_backward_ws(self.S, t["gamma"], t["dY"], t["dS"], self.rstd,
                                          self.dX, self.dg, w.N, w.D, self.ws, self.ws_bytes,
                                          stream)


class SoftmaxRunner:
    """Row softmax forward + backward on synthetic N(0, 3^2) rows (same timing protocol)."""

    def __init__(self, N, D, device, seed, dtype):
        import torch
        import row_wise_rmsnorm_gb300 as mt
        self.mt, self.N, self.D = mt, N, D
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.x = (torch.randn((N, D), generator=g, device=device) * 3).to(dtype)
        self.dy = torch.randn((N, D), generator=g, device=device).to(dtype)
        self.y = torch.empty_like(self.x)
        self.dx = torch.empty_like(self.x)
        self.code = mt.dtype_code(dtype)
        eb = self.x.element_size()
        self.fwd_bytes = 2 * eb * N * D
        self.bwd_bytes = 3 * eb * N * D

    def forward(self, stream):
        self.mt.mt_softmax_forward(self.code, self.x, self.y, self.N, self.D, 0, stream)

    def backward(self, stream):
        self.mt.mt_softmax_backward(self.code, self.y, self.dy, self.dx, self.N, self.D, 0, stream)


class CrossEntropyRunner:
    """Per-row cross-entropy (mean reduction, label smoothing 0.1, z-loss 1e-4) forward +
    backward on synthetic N(0, 2^2) logits with uniform random targets."""

    def __init__(self, N, D, device, seed, dtype):
        import torch
        import row_wise_rmsnorm_gb300 as mt
        self.mt, self.N, self.D = mt, N, D
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.x = (torch.randn((N, D), generator=g, device=device) * 2).to(dtype)
        self.t = torch.randint(0, D, (N,), generator=g, device=device, dtype=torch.int64)
        f = dict(dtype=torch.float32, device=device)
        self.rows, self.lse = torch.empty(N, **f), torch.empty(N, **f)
        self.out, self.nv, self.dl = torch.empty(1, **f), torch.empty(1, **f), torch.ones(1, **f)
        self.dx = torch.empty_like(self.x)
        self.code = mt.dtype_code(dtype)
        eb = self.x.element_size()
        self.fwd_bytes = eb * N * D + 16 * N + 8     # logits, targets, loss and lse rows
        self.bwd_bytes = 2 * eb * N * D + 12 * N     # logits, dlogits, targets, lse

    def forward(self, stream):
        self.mt.mt_cross_entropy_forward(self.code, self.x, self.t, self.N, self.D, -100, 0.1,
                                         1e-4, self.mt.MT_REDUCTION_MEAN, self.rows, self.lse,
                                         self.out, self.nv, stream)

    def backward(self, stream):
        self.mt.mt_cross_entropy_backward(self.code, self.x, self.t, self.lse, self.N, self.D, -100,
                                          0.1, 1e-4, self.mt.MT_REDUCTION_MEAN, self.dl, self.nv,
                                          self.dx, stream)


def time_steps(sets, steps: int, warmup: int, stream, on_enqueued=None) -> float:
    """Mean CUDA-event time (ms) of one step over `steps` back-to-back steps. Step s runs
    the forward on buffer set s % n and the backward on set (s + 1) % n, so no call finds
    in L2 the rows the previous call touched and each call pays for the write-backs the
    previous one left dirty. Events mark only the start and the end of the steps: an
    event recorded between two kernels would keep the second from being scheduled while
    the first drains (programmatic dependent launch), a gap no training loop has.
    `on_enqueued` runs once every timed step is enqueued, while the GPU works on them."""
    import torch
    n = len(sets)
    for r in sets:
        r.forward(stream)  # every set holds valid saved statistics
    for s in range(warmup):
        sets[s % n].forward(stream)
        sets[(s + 1) % n].backward(stream)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for s in range(steps):
        sets[s % n].forward(stream)
        sets[(s + 1) % n].backward(stream)
    z.record(stream)
    if on_enqueued is not None:
        on_enqueued()
    torch.cuda.synchronize()
    return a.elapsed_time(z) / steps


def time_calls(sets, direction: str, calls: int, warmup: int, stream, chunks: int = 10) -> dict:
    """Per-call CUDA-event time (ms) of one direction ("forward" or "backward") over
    `calls` back-to-back calls alternating the buffer sets, in `chunks` runs with events
    at their ends: the mean over all calls and each chunk's mean (the spread)."""
    import torch
    n = len(sets)
    fn = [getattr(r, direction) for r in sets]
    for i in range(warmup):
        fn[i % n](stream)
    per = max(1, calls // chunks)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(chunks + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for c in range(chunks):
        for i in range(per):
            fn[(c * per + i) % n](stream)
        ev[c + 1].record(stream)
    torch.cuda.synchronize()
    ch = [ev[c].elapsed_time(ev[c + 1]) / per for c in range(chunks)]
    return {"mean": ev[0].elapsed_time(ev[chunks]) / (per * chunks), "chunks": ch,
            "calls": per * chunks}


def time_ops(sets, steps: int, warmup: int, stream):
    """Forward and backward per-call times (ms), each from its own back-to-back loop."""
    calls = max(steps, 100)
    return (time_calls(sets, "forward", calls, warmup, stream),
            time_calls(sets, "backward", calls, warmup, stream))


E2E_COPY_STREAMS = 1  # measured on GB300: 1, 2, 4, 8 streams per direction: 404, 391, 378, 283 GB/s


def e2e_run(name: str, device, steps: int, warmup: int, seed: int,
            copy_streams: int = E2E_COPY_STREAMS):
    """Same metric through the public API with pinned-host inputs/outputs: every step
    copies X, gamma, dY (and R, dS / beta) host->device, runs forward + backward, and
    copies Y, stats, dX, dgamma (and S / dbeta) back to pinned host memory.

    Steps are pipelined the way a serving or training loop would run them: copy-in
    streams, a compute stream and copy-out streams, with two device buffer sets, so the
    copy-in of step s runs beside the compute of step s-1 and the copy-out of step s-2.
    Each tensor's copy is split by rows over `copy_streams` streams per direction (one
    cudaMemcpyAsync each), so several copy engines share it. Events order every step's
    three stages and keep a buffer set from being refilled before its previous step's
    outputs are out. The timed region runs from before the first copy-in to after the
    last copy-out."""
    import torch
    sets = [OpRunner(name, device, seed + i) for i in range(2)]
    ins = {k: v.cpu().pin_memory() for k, v in sets[0].t.items()}

    def outs(r):
        return [r.Y, r.rstd, r.dX, r.dg] + [x for x in (r.mean, r.db, r.S) if x is not None]

    outs_host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs(sets[0])]
    h2d = sum(v.numel() * v.element_size() for v in ins.values())
    d2h = sum(x.numel() * x.element_size() for x in outs(sets[0]))
    P = max(1, copy_streams)
    s_in = [torch.cuda.Stream(device=device) for _ in range(P)]
    s_out = [torch.cuda.Stream(device=device) for _ in range(P)]
    s_comp = torch.cuda.Stream(device=device)
    total = warmup + steps
    in_done = [[torch.cuda.Event() for _ in range(P)] for _ in range(total)]
    comp_done = [torch.cuda.Event() for _ in range(total)]
    out_done = [[torch.cuda.Event() for _ in range(P)] for _ in range(total)]

    def pieces(t):
        return t.chunk(P, dim=0) if t.dim() > 0 and t.shape[0] >= P else [t] + [None] * (P - 1)

    def copy_all(dsts, srcs, streams, done):
        for i, st in enumerate(streams):
            with torch.cuda.stream(st):
                for d, s_ in zip(dsts, srcs):
                    dp, sp = pieces(d)[i], pieces(s_)[i]
                    if dp is not None:
                        dp.copy_(sp, non_blocking=True)
            done[i].record(st)

    def step(j):
        r = sets[j % 2]
        if j >= 2:
            for st in s_in:
                st.wait_event(comp_done[j - 2])  # this set's inputs are consumed
        copy_all([r.t[k] for k in ins], list(ins.values()), s_in, in_done[j])
        for ev in in_done[j]:
            s_comp.wait_event(ev)
        if j >= 2:
            for ev in out_done[j - 2]:
                s_comp.wait_event(ev)            # this set's outputs are copied out
        with torch.cuda.stream(s_comp):
            r.forward(s_comp)
            r.backward(s_comp)
        comp_done[j].record(s_comp)
        for st in s_out:
            st.wait_event(comp_done[j])
        copy_all(outs_host, outs(r), s_out, out_done[j])

    for j in range(warmup):
        step(j)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in[0])
    for st in s_in[1:] + s_out + [s_comp]:
        st.wait_event(a)
    for j in range(warmup, total):
        step(j)
    for st in s_out[1:]:
        s_out[0].wait_stream(st)
    b.record(s_out[0])
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    r = sets[0]
    gbs = (r.fwd_bytes + r.bwd_bytes) / (ms * 1e-3) / 1e9
    del sets, r
    return {"value": round(gbs, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "pipeline": (f"{P} copy-in streams, a compute stream, {P} copy-out streams, two "
                         "device buffer sets")}


# ------------------------------------------------------------ CPU oracle ---

_SHARD = {}


def _shard_init(name: str, rows: int, lo: int, hi: int):
    """Worker start-up for the all-cores baseline: draw the workload's first `rows` rows
    (the same draw as the single-core run) and keep this worker's rows lo..hi-1."""
    sys.path.insert(0, ROOT)
    import numpy as np  # noqa: F401
    t = W.generate_workload(name, rows=rows)
    _SHARD.update(name=name, a={k: (v.double().numpy()[lo:hi] if v.dim() == 2 else v.double().numpy())
                               for k, v in t.items()})


def _shard_run(_):
    """One forward + backward of this worker's rows with the oracle; returns its dgamma
    (and dbeta) partial sums for the fixed-order combine."""
    import numpy as np
    import oracle
    w = W.WORKLOADS[_SHARD["name"]]
    a = _SHARD["a"]
    eps = float(np.float32(w.eps))
    if w.op == W.RMSNORM:
        _, rstd = oracle.rmsnorm_forward(a["X"], a["gamma"], eps)
        return oracle.rmsnorm_backward(a["X"], a["gamma"], a["dY"], rstd)[1]
    if w.op == W.LAYERNORM:
        _, mean, rstd = oracle.layernorm_forward(a["X"], a["gamma"], a["beta"], eps)
        r = oracle.layernorm_backward(a["X"], a["gamma"], a["dY"], mean, rstd)
        return r[1], r[3]
    _, s_, rstd = oracle.add_rmsnorm_forward(a["X"], a["R"], a["gamma"], eps)
    s16 = oracle.round_fp16(s_).astype(np.float64)
    return oracle.add_rmsnorm_backward(s16, a["gamma"], a["dY"], a["dS"], rstd)[1]


def oracle_baseline_all_cores(name: str, rows: int, passes: int = 20):
    """The same per-row oracle code on every host core: one spawned process per core, each
    with a contiguous shard of the first `rows` rows; the shards' dgamma (dbeta) partials
    are added in shard order. Reported beside the single-core baseline, not instead of it."""
    import multiprocessing as mp
    import numpy as np
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")  # never fork a process that holds a CUDA context
    bounds = [(rows * i // cores, rows * (i + 1) // cores) for i in range(cores)]
    pools = [ctx.Pool(1, initializer=_shard_init, initargs=(name, rows, lo, hi)) for lo, hi in bounds]
    try:
        for pl in pools:  # warm: library compiled and loaded, inputs drawn
            pl.apply(_shard_run, (0,))
        t0 = time.perf_counter()
        for _ in range(passes):
            parts = [pl.apply_async(_shard_run, (0,)) for pl in pools]
            res = [r.get() for r in parts]
            total = res[0]
            for r_ in res[1:]:  # fixed shard order
                total = tuple(x + y for x, y in zip(total, r_)) if isinstance(total, tuple) else total + r_
        secs = time.perf_counter() - t0
    finally:
        for pl in pools:
            pl.close()
            pl.join()
    w = W.WORKLOADS[name]
    nbytes = passes * (W.compulsory_bytes(w.op, "forward", rows, w.D)
                       + W.compulsory_bytes(w.op, "backward", rows, w.D))
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle, row shards on every core",
            "sample": f"first {rows} of {w.N} rows of {name}, forward + backward, {passes} "
                      f"pass(es), {cores} processes, {secs:.2f} s",
            "rows_per_s": round(passes * rows / secs, 1)}


_ORACLE_INPUTS = {}


def _oracle_inputs(name: str, rows: int, seed: int):
    """The first `rows` rows of the workload as fp64 arrays, drawn once per (name, rows,
    seed) and kept: repeated timing steps reuse them instead of drawing them again."""
    key = (name, rows, seed)
    if key not in _ORACLE_INPUTS:
        _ORACLE_INPUTS.clear()
        t = W.generate_workload(name, rows=rows, seed=seed)
        _ORACLE_INPUTS[key] = {k: v.double().numpy() for k, v in t.items()}
    return _ORACLE_INPUTS[key]


def oracle_step_seconds(name: str, rows: int, seed: int = 0):
    """Wall time of one oracle forward + backward over `rows` rows of the workload."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle
    w = W.WORKLOADS[name]
    a = _oracle_inputs(name, rows, seed)
    eps = float(np.float32(w.eps))
    t0 = time.perf_counter()
    if w.op == W.RMSNORM:
        _, rstd = oracle.rmsnorm_forward(a["X"], a["gamma"], eps)
        oracle.rmsnorm_backward(a["X"], a["gamma"], a["dY"], rstd)
    elif w.op == W.LAYERNORM:
        _, mean, rstd = oracle.layernorm_forward(a["X"], a["gamma"], a["beta"], eps)
        oracle.layernorm_backward(a["X"], a["gamma"], a["dY"], mean, rstd)
    else:
        _, s, rstd = oracle.add_rmsnorm_forward(a["X"], a["R"], a["gamma"], eps)
        s16 = oracle.round_fp16(s).astype(np.float64)
        oracle.add_rmsnorm_backward(s16, a["gamma"], a["dY"], a["dS"], rstd)
    return time.perf_counter() - t0


def oracle_baseline(name: str, budget_s: float = 10.0):
    """The oracle, as it stands, on a bounded sample sized to about `budget_s` of CPU
    work: the first rows of the workload (all of them if they fit), repeated."""
    w = W.WORKLOADS[name]
    probe = min(w.N, 64)
    t_probe = oracle_step_seconds(name, probe)
    rows = int(min(w.N, max(probe, probe * budget_s / max(t_probe, 1e-6))))
    secs, reps = 0.0, 0
    while reps == 0 or (secs < 0.8 * budget_s and reps < 10):
        secs += oracle_step_seconds(name, rows)
        reps += 1
    nbytes = reps * (W.compulsory_bytes(w.op, "forward", rows, w.D)
                     + W.compulsory_bytes(w.op, "backward", rows, w.D))
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {rows} of {w.N} rows of {name}, forward + backward, {reps} "
                      f"pass(es), fp64 single-threaded C, {secs:.2f} s",
            "rows_per_s": round(reps * rows / secs, 1),
            "host_cores": os.cpu_count(), "host_cpu": host_cpu()}


def host_cpu() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, or the Arm implementer and
    part numbers), else the machine type."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model name"):
        for line in info.splitlines():
            if line.startswith(key):
                return line.split(":", 1)[1].strip()
    parts = sorted({line.split(":", 1)[1].strip() for line in info.splitlines()
                    if line.startswith(("CPU implementer", "CPU part"))})
    return f"{platform.machine()} ({', '.join(parts)})" if parts else platform.machine()


def n_buffer_sets(name: str, l2: int) -> int:
    """Buffer sets the timed loops rotate through: 2 when one step's arrays exceed L2, more
    for smaller workloads, so that together they hold at least three times L2 and no call
    finds its inputs in L2 (the same rule as the norm + GEMV's weight sets)."""
    w = W.WORKLOADS[name]
    per_set = (W.compulsory_bytes(w.op, "forward", w.N, w.D)
               + W.compulsory_bytes(w.op, "backward", w.N, w.D))
    return int(max(2, min(4096, -(-3 * l2 // per_set))))


def bench_config(name: str, world: int = 1) -> dict:
    """The workload description both arms print (the same keys and values)."""
    w = W.WORKLOADS[name]
    return {"workload": name, "op": w.op, "N": w.N, "D": w.D, "eps": w.eps,
            "step": "forward + backward",
            "l2": ("not flushed: steps run back to back, rotating the forward and the backward "
                   "over buffer sets that together hold more than L2 (2 sets when one set alone "
                   "exceeds L2), so no call re-reads what an earlier one left in L2, and "
                   "write-backs are paid inside the timed region"),
            "parallelism": f"{world} independent replica(s)"}


def run_reference(args):
    """--impl reference: the oracle on host cores, K steps of a bounded row sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    name = args.workload
    w = W.WORKLOADS[name]
    probe = min(w.N, 512)
    per_row = oracle_step_seconds(name, probe) / probe
    per_step_budget = max(0.02, 60.0 / max(1, args.steps + args.warmup))
    rows = int(max(1, min(w.N, per_step_budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle_step_seconds(name, rows)
    times = [oracle_step_seconds(name, rows) for _ in range(args.steps)]
    secs = sum(times)
    nbytes = args.steps * (W.compulsory_bytes(w.op, "forward", rows, w.D)
                           + W.compulsory_bytes(w.op, "backward", rows, w.D))
    gbs = nbytes / secs / 1e9
    sample = (f"first {rows} of {w.N} rows of {name} per step, forward + backward, fp64 "
              f"single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "rows_per_s": round(args.steps * rows / secs, 2), "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(name, args.gpus),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "rows_per_step": rows},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------- multi-rank ---

def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the step time of the slowest replica)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# Softmax / cross-entropy workloads: name -> (runner, N, D, storage type name).
ROW_OPS = {
    "softmax_16384x4096_f16": ("softmax", 16384, 4096, "float16"),
    "softmax_256x262144_f16": ("softmax", 256, 262144, "float16"),
    "cross_entropy_4096x32768_bf16": ("cross_entropy", 4096, 32768, "bfloat16"),
}


def row_op_line(name, device, steps, warmup, stream, peak):
    """Forward and backward of one ROW_OPS workload, back to back over two buffer sets."""
    import torch
    kind, N, D, tname = ROW_OPS[name]
    cls = SoftmaxRunner if kind == "softmax" else CrossEntropyRunner
    r2 = [cls(N, D, device, i, getattr(torch, tname)) for i in range(2)]
    f2, b2 = time_ops(r2, steps, warmup, stream)
    fg = r2[0].fwd_bytes / (f2["mean"] * 1e-3) / 1e9
    bg = r2[0].bwd_bytes / (b2["mean"] * 1e-3) / 1e9
    return {"row_op": name, "forward_gbs": round(fg, 2), "backward_gbs": round(bg, 2),
            "forward_frac_of_measured": round(fg / peak, 4),
            "backward_frac_of_measured": round(bg / peak, 4),
            "forward_us": round(1e3 * f2["mean"], 3),
            "backward_us": round(1e3 * b2["mean"], 3),
            "compulsory_bytes": {"forward": r2[0].fwd_bytes, "backward": r2[0].bwd_bytes}}


# Fused normalization + GEMV for decode: name -> (op, M, K, N). K x N = 4096 x 12288 is a
# Llama-7B fused QKV projection (three 4096 x 4096 weights side by side).
GEMV_OPS = {
    "rmsnorm_gemv_m1_4096x12288": ("rmsnorm", 1, 4096, 12288),
    "rmsnorm_gemv_m4_4096x12288": ("rmsnorm", 4, 4096, 12288),
    "layernorm_gemv_m4_4096x12288": ("layernorm", 4, 4096, 12288),
    "rmsnorm_gemv_m4_4096x4096": ("rmsnorm", 4, 4096, 4096),
}


def gemv_line(name, device, steps, warmup, stream, peak):
    """CUDA-event time of the fused norm + GEMV, back to back over enough weight sets that
    together they hold three times the L2 (so every call streams its W from HBM).
    Compulsory bytes: W (2KN), X (2MK), gamma (2K), beta (2K, LayerNorm) and Y (2MN)."""
    import torch
    import row_wise_rmsnorm_gb300 as mt
    op, M, K, N = GEMV_OPS[name]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nsets = max(2, -(-3 * l2 // (2 * K * N)))
    sets = []
    for i in range(nsets):
        g = torch.Generator(device=device)
        g.manual_seed(i)
        x = torch.randn((M, K), generator=g, device=device).half()
        gamma = (1 + 0.1 * torch.randn(K, generator=g, device=device)).half()
        beta = (0.1 * torch.randn(K, generator=g, device=device)).half()
        w = (torch.randn((K, N), generator=g, device=device) / K ** 0.5).half()
        sets.append((x, gamma, beta, w, torch.empty((M, N), dtype=torch.float16, device=device)))

    def call(j):
        x, gamma, beta, w, y = sets[j % nsets]
        if op == "rmsnorm":
            mt.mt_fused_rmsnorm_gemv(x, gamma, w, y, M, N, K, 1e-5, stream)
        else:
            mt.mt_fused_layernorm_gemv(x, gamma, beta, w, y, M, N, K, 1e-5, stream)

    for j in range(warmup):
        call(j)
    # back-to-back calls in chunks, events only at the chunks' ends (see time_steps)
    chunks, per = 10, max(1, max(steps, 100) // 10)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(chunks + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for c in range(chunks):
        for j in range(per):
            call(c * per + j)
        ev[c + 1].record(stream)
    torch.cuda.synchronize()
    ts = [ev[c].elapsed_time(ev[c + 1]) / per for c in range(chunks)]
    nbytes = 2 * K * N + 2 * M * K + 2 * K * (2 if op == "layernorm" else 1) + 2 * M * N
    ms = ev[0].elapsed_time(ev[chunks]) / (per * chunks)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"gemv": name, "us": round(1e3 * ms, 3), "us_chunk_min": round(1e3 * min(ts), 3),
            "us_chunk_max": round(1e3 * max(ts), 3),
            "gbs": round(gbs, 2), "frac_of_measured": round(gbs / peak, 4),
            "compulsory_bytes": nbytes, "M": M, "K": K, "N": N,
            "gflops": round(2 * M * K * N / (ms * 1e-3) / 1e9, 1)}


# --------------------------------------------------------------- main ---

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--workload", choices=W.WORKLOAD_ORDER, default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the per-op numbers of the other large workloads")
    ap.add_argument("--gemv", choices=list(GEMV_OPS),
                    help="time only this fused norm + GEMV workload (a side measurement) and "
                         "print its own line")
    ap.add_argument("--row-op", choices=list(ROW_OPS),
                    help="time only this softmax / cross-entropy workload (a side measurement, "
                         "e.g. for a profiler) and print its own line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    import row_wise_rmsnorm_gb300 as mt
    mt.load()  # fails loudly if the CUDA library is not built

    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    peak, peak_src = measured_peak_gbs()
    if args.row_op or args.gemv:
        line = (row_op_line(args.row_op, device, args.steps, args.warmup, stream, peak)
                if args.row_op else gemv_line(args.gemv, device, args.steps, args.warmup, stream,
                                              peak))
        if rank == 0:
            print(json.dumps(line))
        return 0
    nsets = n_buffer_sets(args.workload, l2)
    sets = [OpRunner(args.workload, device, seed=nsets * rank + i) for i in range(nsets)]
    runner = sets[0]
    w = runner.w

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    with ClockSampler(device) as clocks:
        t0 = time.perf_counter()
        step_ms = time_steps(sets, args.steps, args.warmup, stream, on_enqueued=clocks.mark)
        barrier()
        wall = time.perf_counter() - t0
    step_ms = max_over_ranks(step_ms, device)
    # each call's own time, from back-to-back loops of that call alone
    fwd, bwd = time_ops(sets, args.steps, args.warmup, stream)
    fwd_ms, bwd_ms = fwd["mean"], bwd["mean"]

    step_bytes = runner.fwd_bytes + runner.bwd_bytes
    value = world * step_bytes / (step_ms * 1e-3) / 1e9
    rows_s = world * w.N / (step_ms * 1e-3)

    def op_line(nbytes, t, rows):
        ms = t["mean"]
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"us": round(1e3 * ms, 3),
                "us_chunk_min": round(1e3 * min(t["chunks"]), 3),
                "us_chunk_max": round(1e3 * max(t["chunks"]), 3), "calls": t["calls"],
                "gbs": round(gbs, 2), "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                "frac_of_measured": round(gbs / peak, 4), "rows_per_s": round(rows / (ms * 1e-3), 1),
                "compulsory_bytes": nbytes}

    ops = {"forward": op_line(runner.fwd_bytes, fwd, w.N),
           "backward": op_line(runner.bwd_bytes, bwd, w.N)}
    dom = "backward" if bwd_ms >= fwd_ms else "forward"
    del runner, sets
    torch.cuda.empty_cache()

    def roofline_block(name, direction, line):
        """One kernel call's roofline entry: algorithmic (compulsory) bytes per call over
        its mean CUDA-event time, against the measured copy peak and 8 TB/s."""
        return {"bound": "hbm", "kernels": KERNELS.get((name, direction)),
                "achieved": line["gbs"], "peak": peak, "unit": "GB/s",
                "frac": line["frac_of_measured"], "frac_of_8tbs": line["frac_of_8tbs"],
                "us": line["us"], "rows_per_s": line["rows_per_s"],
                "algorithmic_bytes_per_launch": line["compulsory_bytes"],
                "traffic": recorded_traffic(name, direction)}

    rooflines = {args.workload: {d: roofline_block(args.workload, d, ops[d]) for d in ops}}
    others = {}
    if not args.no_others and rank == 0:
        for name in LARGE_WORKLOADS:
            if name == args.workload:
                continue
            r2 = [OpRunner(name, device, seed=i) for i in range(2)]
            f2, b2 = time_ops(r2, args.steps, args.warmup, stream)
            r2 = r2[0]
            w2 = r2.w
            lines = {"forward": op_line(r2.fwd_bytes, f2, w2.N),
                     "backward": op_line(r2.bwd_bytes, b2, w2.N)}
            others[name] = {"forward_gbs": lines["forward"]["gbs"],
                            "backward_gbs": lines["backward"]["gbs"],
                            "forward_us": lines["forward"]["us"],
                            "backward_us": lines["backward"]["us"]}
            if name in GATED_WORKLOADS:
                rooflines[name] = {d: roofline_block(name, d, lines[d]) for d in lines}
            del r2
            torch.cuda.empty_cache()

    # Storage types other than fp16 on the headline workload (bf16, fp32), per op time.
    dtypes = {}
    if not args.no_others and rank == 0:
        for dname, tdt in (("bf16", torch.bfloat16), ("f32", torch.float32)):
            r2 = [OpRunner(args.workload, device, seed=i, dtype=tdt) for i in range(nsets)]
            f2, b2 = time_ops(r2, args.steps, args.warmup, stream)
            r2 = r2[0]
            fg = r2.fwd_bytes / (f2["mean"] * 1e-3) / 1e9
            bg = r2.bwd_bytes / (b2["mean"] * 1e-3) / 1e9
            dtypes[dname] = {
                "forward_gbs": round(fg, 2), "backward_gbs": round(bg, 2),
                "forward_frac_of_measured": round(fg / peak, 4),
                "backward_frac_of_measured": round(bg / peak, 4),
                "forward_us": round(1e3 * f2["mean"], 3),
                "backward_us": round(1e3 * b2["mean"], 3),
                "compulsory_bytes": {"forward": r2.fwd_bytes, "backward": r2.bwd_bytes}}
            del r2
            torch.cuda.empty_cache()

    # The row softmax and the per-row cross-entropy (the next row-reduction family).
    row_ops = {}
    if not args.no_others and rank == 0:
        for name in ROW_OPS:
            row_ops[name] = row_op_line(name, device, args.steps, args.warmup, stream, peak)
            del row_ops[name]["row_op"]
            torch.cuda.empty_cache()

    # Fused normalization + GEMV (decode).
    gemv = {}
    if not args.no_others and rank == 0:
        for name in GEMV_OPS:
            gemv[name] = gemv_line(name, device, args.steps, args.warmup, stream, peak)
            del gemv[name]["gemv"]
            torch.cuda.empty_cache()

    e2e = None
    if not args.no_e2e:
        e2e = e2e_run(args.workload, device, max(20, min(50, args.steps // 40)), 3, seed=rank)
        if world > 1:
            e2e["ms_per_step"] = round(max_over_ranks(e2e["ms_per_step"], device), 4)
            e2e["value"] = round(world * step_bytes / (e2e["ms_per_step"] * 1e-3) / 1e9, 2)

    cpu = cpu_all = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline and args.gpus == 1:
        cpu = oracle_baseline(args.workload)
        cpu_all = oracle_baseline_all_cores(args.workload,
                                            min(W.WORKLOADS[args.workload].N, 8192))

    dom_block = rooflines[args.workload][dom]
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "rows_per_s": round(rows_s, 1),
        "frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "frac_of_measured": round(value / world / peak, 4),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "storage": "f16",
        "data": "synthetic",
        "config": bench_config(args.workload, world),
        "l2_note": (f"{nsets} buffer sets of {step_bytes >> 20} MiB "
                    f"of compulsory traffic each against {l2 >> 20} MiB of L2"),
        "ops": ops,
        "roofline": {"bound": "hbm", "kernel": f"{w.op} {dom}: " + " + ".join(
            KERNELS.get((args.workload, dom), ["the row kernel"] + (["param_reduce_kernel"]
                                                                    if dom == "backward" else []))),
                     "achieved": dom_block["achieved"], "peak": peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": dom_block["frac"], "traffic": dom_block["traffic"],
                     "algorithmic_bytes_per_launch": dom_block["algorithmic_bytes_per_launch"]},
        "rooflines": rooflines,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": e2e,
        "gpu_launches": args.steps * 3,  # per step: the forward, the backward row kernel, the reduction
        "clocks": clocks.summary(),
        "timed_region_wall_s": round(wall, 3),
        "other_workloads": others,
        "storage_types": {"workload": args.workload, **dtypes},
        "row_ops": row_ops,
        "norm_gemv": gemv,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
