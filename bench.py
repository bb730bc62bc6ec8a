"""Benchmark: fused causal SDPA forward on one GB300, plus the fp64 oracle's
CPU baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 3] [--impl reference]

One step = one fused forward (one kernel launch) over the workload's whole
batch.  Default workload: causal [B=4, H=32, L=4096, D=128] bf16, q/k/v drawn
N(0,1)*0.5 from fixed seeds.  Prints ONE JSON line (rank 0).

value        algorithmic TFLOP/s (causal: 2*B*H*L^2*D per forward) with inputs
             resident in HBM, K steps timed with CUDA events on the launch
             stream; q, k, v, out total 537 MB > the 129 MB L2, so no flush.
e2e          the same metric through the same C-ABI call, with pinned host
             buffers: every step copies its q, k, v (and mask) in and its out
             back inside the timed region; steps are pipelined over two device
             buffer sets and three streams (copy-in, compute, copy-out).
roofline     achieved = algorithmic FLOPs per launch / mean per-launch kernel
             time (CUDA events around each launch in the timed region); peak =
             the measured dense bf16 GEMM rate (burst) of this GPU model.  A
             workload whose algorithmic FLOP per byte is below the ridge of
             the measured peaks (the rank-3 and [8,16,1024,64] cases) is
             reported against HBM instead: GB/s of algorithmic bytes against
             the measured copy bandwidth.
cpu_baseline the fp64 oracle on the host cores, on a bounded sample of query
             rows of the same workload, in the same unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal SDPA fwd TFLOP/s at B4·H32·L4096·D128 bf16; % of GB300 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
# The code each kernel is built from (a traffic figure is valid only for the
# code it was captured on): head size 128, head size 64, sparse top-k.
KERNEL_SOURCES = ["scaled_dot_product_forward_gb300/csrc/sdpa_fwd_sm103a.cu",
                  "scaled_dot_product_forward_gb300/csrc/sdpa_sched.cuh",
                  "scaled_dot_product_forward_gb300/csrc/ptx.cuh"]
KERNEL64_SOURCES = ["scaled_dot_product_forward_gb300/csrc/sdpa_fwd64_sm103a.cu",
                    "scaled_dot_product_forward_gb300/csrc/sdpa_sched.cuh",
                    "scaled_dot_product_forward_gb300/csrc/ptx.cuh"]
SPARSE_SOURCES = ["scaled_dot_product_forward_gb300/csrc/sdpa_sparse_sm103a.cu",
                  "scaled_dot_product_forward_gb300/csrc/ptx.cuh"]


def code_of(text: str) -> str:
    """A source file without its // comments and blank lines (the kernel
    sources hold no '//' inside string literals and no block comments), so
    that a comment edit keeps the identity of code that was profiled."""
    lines = []
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            lines.append(code)
    return "\n".join(lines)


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("hbm_gbs", 0.0)), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 6800.0, "fallback"


def roofline_of(w, flops, mean_launch_ms, peak, hbm_peak, peak_kind, traffic):
    """The bound a workload's arithmetic intensity puts it under at the
    measured peaks: the tensor core (TFLOP/s against the bf16 GEMM rate) when
    its algorithmic FLOP per algorithmic byte is at or above the ridge, else
    HBM (GB/s of algorithmic bytes against the measured copy bandwidth)."""
    # (a rank with a range of the heads moves that share of the bytes)
    alg_bytes = w.alg_bytes() * flops / w.flops()
    tflops = flops / (mean_launch_ms * 1e-3) / 1e12
    gbs = alg_bytes / (mean_launch_ms * 1e-3) / 1e9
    ridge = peak * 1e12 / (hbm_peak * 1e9) if hbm_peak > 0 else 0.0
    common = {"traffic": traffic, "alg_flops_per_launch": flops,
              "alg_bytes_per_launch": alg_bytes, "flop_per_byte": flops / alg_bytes,
              "ridge_flop_per_byte": ridge, "mean_launch_ms": mean_launch_ms}
    if hbm_peak > 0 and flops / alg_bytes < ridge:
        return {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": gbs / hbm_peak, "peak_source": f"{peak_kind} HBM copy",
                "tflops": tflops, **common}
    return {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": UNIT,
            "frac": tflops / peak, "peak_source": f"{peak_kind} dense bf16 (burst)",
            "gbs": gbs, **common}


def load_traffic(workload_id, sources=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None).  ``workload_id`` is a dense
    workload number, "varlen" or "sparse"."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    entry = t.get(str(workload_id))
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    return entry.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) over the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

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
        if self.thread:
            self.thread.join(timeout=5)
        sms, maxes, reasons, powers = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
                powers.append(float(parts[3]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms),
                "power_w_max": max(powers) if powers else None}


# --------------------------------------------------------- CPU (oracle) leg
class OracleSampler:
    """Times the fp64 oracle on random query rows (b, h, i) of workload
    ``w`` (the operands are generated and widened once).  The rows it
    evaluates, and their oracle outputs, double as the parity sample of the
    GPU output."""

    def __init__(self, w, operands=None):
        import numpy as np
        import torch

        import oracle
        import sdpa_inputs

        self.w = w
        q, k, v, mask = operands if operands is not None else sdpa_inputs.make(w)
        if w.rank == 3:
            q, k, v = q[None], k[None], v[None]
        self.q, self.k, self.v = (x.to(torch.float64).numpy() for x in (q, k, v))
        self.mask = None if mask is None else (mask.numpy() != 0).astype(np.uint8)
        self.oracle = oracle
        self.rate = None  # rows per second
        self.last_rows = None
        self.last_out = None

    def _flops(self, rows):
        w = self.w
        if w.is_causal:
            return float(sum(4.0 * w.D * (i + 1) for i in rows[:, 2]))
        return float(len(rows) * 4.0 * w.D * w.L)

    def _rows(self, g, n):
        import numpy as np
        B, H = self.q.shape[0], self.q.shape[1]
        rows = np.zeros((n, 3), dtype=np.int64)
        rows[:, 0] = g.integers(0, B, size=n)
        rows[:, 1] = g.integers(0, H, size=n)
        rows[:, 2] = g.integers(0, self.w.L, size=n)
        return rows

    def run(self, budget_s: float, seed: int = 0):
        """(algorithmic FLOPs, seconds, rows) for about ``budget_s`` of work."""
        import numpy as np
        g = np.random.default_rng(seed)
        if self.rate is None:
            n0 = max(8, self.oracle.num_threads())
            rows = self._rows(g, n0)
            t0 = time.perf_counter()
            self.oracle.sdpa_rows(self.q, self.k, self.v, rows, mask=self.mask,
                                  is_causal=self.w.is_causal, scale=self.w.scale)
            self.rate = n0 / max(time.perf_counter() - t0, 1e-6)
        n = max(1, int(self.rate * budget_s))
        rows = self._rows(g, n)
        t0 = time.perf_counter()
        out = self.oracle.sdpa_rows(self.q, self.k, self.v, rows, mask=self.mask,
                                    is_causal=self.w.is_causal, scale=self.w.scale)
        dt = time.perf_counter() - t0
        self.last_rows, self.last_out = rows, out
        return self._flops(rows), dt, n

    @property
    def cores(self):
        return self.oracle.num_threads()


PARITY_L2, PARITY_MAX = 1e-2, 2e-2


def parity_of(got, ref, rows: int, against: str, extra_ok: bool = True, extra: str = ""):
    """L2-relative and max-abs error of GPU values ``got`` against oracle
    values ``ref`` (same shape), and whether both are inside the tolerance
    (and ``extra_ok``, a further exact check named by ``extra``)."""
    import numpy as np
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = got - ref
    nref = float(np.linalg.norm(ref))
    l2 = float(np.linalg.norm(err)) / (nref if nref > 0 else 1.0)
    mx = float(np.abs(err).max()) if err.size else 0.0
    finite = bool(np.all(np.isfinite(got)))
    ok = finite and l2 <= PARITY_L2 and mx <= PARITY_MAX and extra_ok
    d = {"l2_rel": l2 if finite else None, "max_abs": mx if finite else None, "pass": ok,
         "rows": rows, "tolerance": {"l2_rel": PARITY_L2, "max_abs": PARITY_MAX},
         "against": against}
    if extra:
        d["exact_check"] = {"what": extra, "pass": bool(extra_ok)}
    return d


# ---------------------------------------------------------------- GPU leg
def pipelined_e2e(torch, dev, comp, fwd, dsets, hins, n):
    """Milliseconds per step of the end-to-end job: each step copies its
    inputs in from pinned host buffers, runs the forward through the public
    call and copies its output back to a pinned host buffer.  Steps are
    pipelined over two device buffer sets and three streams (copy-in,
    compute, copy-out), so step i+1's inputs travel while step i computes and
    step i-1's output returns; every step's copies are inside the timed
    region, which runs from before the first copy-in to after the last
    copy-out."""
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    houts = [torch.empty(dsets[0][-1].shape, dtype=dsets[0][-1].dtype).pin_memory()
             for _ in range(2)]

    def run(count):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_done, comp_done, out_done = ([ev() for _ in range(count)] for _ in range(3))
        for i in range(count):
            b = i % 2
            d = dsets[b]
            if i >= 2:
                s_in.wait_event(comp_done[i - 2])   # set b no longer read
            with torch.cuda.stream(s_in):
                for dst, src in zip(d[:-1], hins):
                    dst.copy_(src, non_blocking=True)
            in_done[i].record(s_in)
            comp.wait_event(in_done[i])
            if i >= 2:
                comp.wait_event(out_done[i - 2])    # set b's output copied out
            fwd(d, comp)
            comp_done[i].record(comp)
            s_out.wait_event(comp_done[i])
            with torch.cuda.stream(s_out):
                houts[b].copy_(d[-1], non_blocking=True)
            out_done[i].record(s_out)

    run(2)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    run(n)
    comp.synchronize()
    s_in.synchronize()
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    return t0.elapsed_time(t1) / n


def gpu_leg(args, w, rank, world):
    import torch

    import scaled_dot_product_forward_gb300 as sdpa
    import sdpa_inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    sdpa.load_library()
    q, k, v, mask = sdpa_inputs.make(w)
    flops = w.flops()
    if getattr(args, "shard", "replicas") == "heads" and world > 1:
        # This rank's contiguous range of the heads of the one problem (the
        # heads are independent: no exchange), held as its own tensors.
        if world > w.H:
            raise SystemExit(f"--shard heads: {world} ranks for {w.H} heads")
        h0, h1 = sdpa.head_range(w.H, rank, world)
        hd = 1 if q.dim() == 4 else 0
        q, k, v = (x.narrow(hd, h0, h1 - h0).contiguous() for x in (q, k, v))
        flops = w.flops() * (h1 - h0) / w.H
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    md = mask.to(dev) if mask is not None else None
    out = torch.empty_like(qd)
    stream = torch.cuda.Stream(dev)

    def step():
        sdpa.sdpa_forward(qd, kd, vd, out, is_causal=w.is_causal, mask=md, stream=stream)

    plan = sdpa.SdpaPlan(qd, kd, vd, out, is_causal=w.is_causal, mask=md)

    def plan_step():
        plan.launch(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
            plan_step()
    stream.synchronize()
    rc, detail = sdpa.sdpa_last_device_status(stream)
    if rc != 0:
        raise RuntimeError(f"warm-up reported {sdpa.sdpa_status_string(rc)} ({detail:#x})")

    # Host cost of one call (no synchronisation inside; the GPU queue absorbs
    # the launches), through the one-shot entry point and through a plan.
    host_us = {}
    for name, fn in (("sdpa_forward", step), ("plan_launch", plan_step)):
        n = 64
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        host_us[name] = (time.perf_counter() - t0) / n * 1e6
        stream.synchronize()

    # Inputs that fit in L2 are flushed from it before every timed launch
    # (a 256 MB write, outside the launch's event pair); larger ones cannot
    # stay in L2 between steps anyway.
    flush = None
    if flush_l2(args, w):
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    graph = None
    if args.graph:
        # K plan launches captured once; the timed region replays them with
        # no host work between kernels.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(args.steps):
                plan.launch(stream)
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()

    # --- timed region: K launches, an event pair around each one
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the work
    t_begin.record(stream)
    if graph is not None:
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            graph.replay()
    else:
        timed = plan_step if args.plan else step
        for i in range(args.steps):
            if flush is not None:
                with torch.cuda.stream(stream):
                    flush.zero_()   # outside the event pair: L2 holds none of the inputs
            starts[i].record(stream)
            timed()
            ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_begin.elapsed_time(t_end)
    if graph is not None:
        per_launch_ms = [total_ms / args.steps]  # back to back, no host gaps
    else:
        per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        if flush is not None:
            total_ms = sum(per_launch_ms)  # the K launches, without the flushes between them
    rc, detail = sdpa.sdpa_last_device_status(stream)
    if rc != 0:
        raise RuntimeError(f"timed region reported {sdpa.sdpa_status_string(rc)} ({detail:#x})")

    # --- end to end through host buffers
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    hins = [x.pin_memory() for x in (q, k, v)] + ([mask.pin_memory()] if mask is not None else [])
    dsets = [[qd, kd, vd] + ([md] if md is not None else []) + [out]]
    dsets.append([torch.empty_like(x) for x in dsets[0]])

    def fwd(dset, s):
        m = dset[3] if md is not None else None
        sdpa.sdpa_forward(dset[0], dset[1], dset[2], dset[-1], is_causal=w.is_causal, mask=m,
                          stream=s)

    e2e_ms = pipelined_e2e(torch, dev, stream, fwd, dsets, hins, e2e_steps)
    h2d = sum(x.numel() * x.element_size() for x in hins)
    d2h = out.numel() * out.element_size()
    plan.close()
    return dict(total_ms=total_ms, per_launch_ms=per_launch_ms, clocks=clk, e2e_ms=e2e_ms,
                h2d=h2d, d2h=d2h, flops=flops, host_us=host_us, out=out,
                operands=(q, k, v, mask))


def extra_leg(args, path):
    """Packed documents (``--path varlen``) or sparse top-k (``--path
    sparse``): W warm-up launches, then K launches each timed alone with CUDA
    events on the launch stream, the 256 MB L2-flush write between them
    outside the timed pair; e2e through pinned host buffers."""
    import torch

    import scaled_dot_product_forward_gb300 as sdpa
    import sdpa_inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    sdpa.load_library()
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    if path == "varlen":
        cfgd = sdpa_inputs.VARLEN_DOCS
        q, k, v, cu, lengths = sdpa_inputs.make_varlen(**cfgd)
        H, D = cfgd["H"], cfgd["D"]
        flops = float(sum(2.0 * H * n * n * D for n in lengths))   # causal convention
        metric = (f"packed-document causal SDPA fwd TFLOP/s ({cfgd['n_docs']} documents of "
                  f"{cfgd['lo']}-{cfgd['hi']} tokens, H{H} D{D} bf16)")
        config = {"workload": "packed causal documents", "n_docs": cfgd["n_docs"],
                  "lengths": lengths, "total": int(cu[-1]), "H": H, "D": D,
                  "launch": "sdpa_forward_varlen per step", "l2": "flushed between launches"}
        ins = [q, k, v, cu]
        maxlen = max(lengths)

        def launch(t, out):
            sdpa.sdpa_forward_varlen(t[0], t[1], t[2], t[3], maxlen, out, is_causal=True,
                                     stream=stream)
    else:
        cfgd = sdpa_inputs.SPARSE_DSA
        q, kv, idx, length = sdpa_inputs.make_sparse(**cfgd)
        H, D = cfgd["H"], cfgd["D"]
        flops = 4.0 * H * D * float(length.sum())
        metric = (f"sparse top-k SDPA fwd TFLOP/s ({cfgd['total']} tokens, H{H} D{D}, "
                  f"top-{cfgd['topk']} causal index rows, one shared KV head, bf16)")
        config = {"workload": "sparse top-k (DSA-style)", "total": cfgd["total"], "H": H,
                  "D": D, "topk": cfgd["topk"], "index_rows": "causal, hole-free",
                  "kv": "one tensor as key and value (fwd(q, kv, idx))",
                  "launch": "sdpa_sparse_forward per step", "l2": "flushed between launches"}
        ins = [q, kv, idx, length]

        def launch(t, out):
            sdpa.sdpa_sparse_forward(t[0], t[1], t[1], t[2], t[3], out, stream=stream)
    dins = [x.to(dev) for x in ins]
    out = torch.empty_like(dins[0])
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            launch(dins, out)
    stream.synchronize()
    rc, detail = sdpa.sdpa_last_device_status(stream)
    if rc != 0:
        raise RuntimeError(f"warm-up reported {sdpa.sdpa_status_string(rc)} ({detail:#x})")
    clocks = ClockSampler(dev.index)
    clocks.start()
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch(dins, out)
            e1.record(stream)
            evs.append((e0, e1))
    stream.synchronize()
    clk = clocks.stop()
    per = [a.elapsed_time(b) for a, b in evs]
    ms = statistics.fmean(per)
    # e2e: pinned host inputs in, output back, every step (pipelined)
    hins = [x.pin_memory() for x in ins]
    dsets = [dins + [out], [torch.empty_like(x) for x in dins + [out]]]

    def fwd(dset, s):
        with torch.cuda.stream(s):
            launch(dset[:-1], dset[-1])

    e2e_ms = pipelined_e2e(torch, dev, stream, fwd, dsets, hins, max(3, args.e2e_steps))
    peak, _, peak_kind = load_peaks()
    achieved = flops / (ms * 1e-3) / 1e12
    line = {"metric": metric, "value": achieved, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "peak_source": f"{peak_kind} dense bf16 (burst)",
                         "traffic": (load_traffic("sparse", SPARSE_SOURCES) if path == "sparse"
                                     else load_traffic("varlen")),
                         "alg_flops_per_launch": flops, "mean_launch_ms": ms},
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in ins),
                    "d2h_bytes_per_step": out.numel() * out.element_size(),
                    "ms_per_step": e2e_ms},
            "gpu_launches": args.steps, "clocks": clk, "parity": None}
    if not args.no_cpu_baseline:
        # the oracle on a bounded sample, whose outputs also check the same
        # rows of the timed launches' output
        import numpy as np
        import oracle
        # random (document, head) pairs / random query rows until the oracle
        # has run for the budget (only the oracle calls are timed)
        gen = torch.Generator().manual_seed(4242)
        refs, gots = [], []
        f, t, rows, units = 0.0, 0.0, 0, 0
        out_h = out.cpu()
        if path == "varlen":
            for pid in torch.randperm(len(lengths) * H, generator=gen).tolist():
                d, hh = divmod(pid, H)
                a, n = int(cu[d]), lengths[d]
                t0 = time.perf_counter()
                ref = oracle.sdpa_varlen(q[a:a + n, hh:hh + 1], k[a:a + n, hh:hh + 1],
                                         v[a:a + n, hh:hh + 1], [0, n], is_causal=True)
                t += time.perf_counter() - t0
                refs.append(np.asarray(ref).reshape(-1, D))
                gots.append(out_h[a:a + n, hh:hh + 1].double().numpy().reshape(-1, D))
                f += 2.0 * n * n * D
                rows += n
                units += 1
                if t >= args.cpu_budget_s:
                    break
            sample = f"{units} random (document, head) pairs, {rows} rows"
        else:
            perm = torch.randperm(q.shape[0], generator=gen)
            for c0 in range(0, q.shape[0], 128):
                sel = perm[c0:c0 + 128]
                t0 = time.perf_counter()
                ref = oracle.sdpa_sparse(q[sel], kv, kv, idx[sel].numpy(),
                                         topk_length=length[sel].numpy())
                t += time.perf_counter() - t0
                refs.append(np.asarray(ref).reshape(-1, D))
                gots.append(out_h[sel].double().numpy().reshape(-1, D))
                f += 4.0 * H * D * float(length[sel].sum())
                rows += len(sel)
                if t >= args.cpu_budget_s:
                    break
            sample = f"{rows} random query rows (all heads)"
        ref, got = np.concatenate(refs), np.concatenate(gots)
        line["cpu_baseline"] = {"value": f / t / 1e12, "unit": UNIT,
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"{sample}, {t:.1f} s"}
        line["parity"] = parity_of(got, ref, rows,
                                   "fp64 oracle on the cpu_baseline sample of the timed "
                                   "launches' output")
    return line


def job_flops(workload_flops: float, rank_flops: float, world: int, sharded: bool) -> float:
    """The work one timed step of the whole job did: with replicas every rank
    ran the workload (rank_flops each); with the heads split the ranks
    together ran it once."""
    return workload_flops if (sharded and world > 1) else world * rank_flops


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--shard", choices=["replicas", "heads"], default="replicas",
                    help="with N > 1: every rank runs the whole workload (weak scaling), or "
                         "each computes its range of the heads of one problem (strong)")
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--plan", action="store_true",
                    help="time sdpa_plan_launch per step (with a mask: the mask summary kernel "
                         "and the forward, both inside each timed launch)")
    ap.add_argument("--graph", action="store_true",
                    help="time a CUDA graph of K plan launches (no host gaps between kernels)")
    ap.add_argument("--path", choices=["dense", "varlen", "sparse"], default="dense",
                    help="dense (the default contract line), packed documents or sparse top-k")
    ap.add_argument("--all-workloads", action="store_true",
                    help="one line per specified dense workload (1-5), each with its roofline "
                         "and parity")
    ap.add_argument("--flush-l2", choices=["auto", "yes", "no"], default="auto",
                    help="auto: flush L2 before each timed launch when the operands fit in it")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.path != "dense":
        if args.impl == "reference" or int(os.environ.get("WORLD_SIZE", "1")) > 1:
            ap.error("--path varlen/sparse measures one GPU with the fused kernels only")
        print(json.dumps(extra_leg(args, args.path)))
        return 0

    import sdpa_inputs
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    wids = sorted(sdpa_inputs.WORKLOADS) if args.all_workloads else [args.workload]
    if args.impl == "reference":
        # The reference arm is the fp64 oracle on the host cores.
        if rank != 0:
            return 0
        for wid in wids:
            print(json.dumps(reference_line(args, sdpa_inputs.WORKLOADS[wid])), flush=True)
        return 0

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    for wid in wids:
        line = dense_line(args, wid, rank, world)
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def flush_l2(args, w) -> bool:
    """Flush L2 between timed launches: when the operands fit in twice the
    129 MB L2 (else they cannot stay resident between steps), except under
    --graph (back-to-back replay) or --flush-l2 no."""
    if args.graph or args.flush_l2 == "no":
        return False
    return args.flush_l2 == "yes" or 4 * w.heads * w.L * w.D * 2 < 2 * 129e6


def metric_of(w):
    return METRIC if w.wid == 3 else f"SDPA fwd TFLOP/s, {w.name}"


def config_of(args, w):
    return {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "D": w.D,
            "launch": ("cuda graph of plan launches" if args.graph else
                       "sdpa_plan_launch per step" if args.plan else "sdpa_forward per step") +
                      (" (mask summary kernel + forward)" if (args.graph or args.plan) and
                       w.p_masked is not None else ""),
            "is_causal": w.is_causal, "mask": w.p_masked is not None,
            "rank": w.rank, "scale": "1/sqrt(D)",
            "l2": ("flushed before every timed launch (256 MB write outside the launch's "
                   "events): q, k, v, out total %.1f MB" if flush_l2(args, w) else
                   "no flush: q, k, v, out total %.1f MB (> 2 x the 129 MB L2, or a graph "
                   "replayed back to back)") % (4 * w.heads * w.L * w.D * 2 / 1e6)}


def reference_line(args, w):
    per_step = max(0.02, 120.0 / (args.steps + args.warmup))
    sampler = OracleSampler(w)
    for i in range(args.warmup):
        sampler.run(per_step / 4, seed=1000 + i)
    tf, tt, rows = 0.0, 0.0, 0
    for i in range(args.steps):
        f, t, n = sampler.run(per_step, seed=i + 1)
        tf, tt, rows = tf + f, tt + t, rows + n
    cores = sampler.cores
    val = tf / tt / 1e12
    return {"impl": "reference", "metric": metric_of(w), "value": val, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args, w),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{rows} random query rows (b, h, i) of the workload, "
                                       f"{args.steps} steps"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def dense_line(args, wid, rank, world):
    import sdpa_inputs
    w = sdpa_inputs.WORKLOADS[wid]
    dtype = "bf16" if "bf16" in w.name else "fp16"
    r = gpu_leg(args, w, rank, world)
    total_ms = max_over_ranks(r["total_ms"], world)
    ms_per_step = total_ms / args.steps
    # replicas: every rank did the whole workload; heads: the ranks together
    # did one (work of all ranks / the slowest rank's time either way)
    sharded = args.shard == "heads" and world > 1
    done = job_flops(w.flops(), r["flops"], world, sharded)
    value = done / (ms_per_step * 1e-3) / 1e12
    mean_launch_ms = statistics.fmean(r["per_launch_ms"])
    peak, hbm_peak, peak_kind = load_peaks()
    # A masked plan runs the mask-summary path (its own ncu capture).
    summary = (args.plan or args.graph) and w.p_masked is not None
    traffic = load_traffic(f"{wid}plan" if summary else wid,
                           KERNEL64_SOURCES if w.D == 64 else KERNEL_SOURCES)
    e2e_ms = max_over_ranks(r["e2e_ms"], world)
    line = {"metric": metric_of(w), "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "strong" if sharded else "weak",
            "vs_baseline": None, "dtype": dtype,
            "data": "synthetic", "config": dict(config_of(args, w), parallelism=(
                f"heads split over {world} ranks" if sharded else f"{world} replicas")),
            "roofline": roofline_of(w, r["flops"], mean_launch_ms, peak, hbm_peak, peak_kind,
                                    traffic * r["flops"] / w.flops() if traffic else traffic),
            "e2e": {"value": done / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                    "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * (2 if (args.graph or args.plan) and
                                          w.p_masked is not None else 1),
            "host_us_per_call": r["host_us"],
            "clocks": r["clocks"], "parity": None}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # The oracle leg: timed on random rows of the workload, whose outputs
        # then check the same rows of the timed launches' output.
        sampler = OracleSampler(w, r["operands"])
        f, t, rows = sampler.run(args.cpu_budget_s)
        cores = sampler.cores
        line["cpu_baseline"] = {"value": f / t / 1e12, "unit": UNIT, "cores": cores,
                                "kind": "oracle",
                                "sample": f"{rows} random query rows (b, h, i) of the workload, "
                                          f"algorithmic FLOPs of those rows, {t:.1f} s"}
        out = r["out"]
        got_all = out if w.rank == 4 else out[None]
        idx = sampler.last_rows
        import torch
        ti = torch.as_tensor(idx, device=out.device)
        got = got_all[ti[:, 0], ti[:, 1], ti[:, 2]].double().cpu().numpy()
        extra_ok, extra = True, ""
        if w.p_masked is not None:
            dead = sdpa_inputs.full_rows(w).to(out.device)
            extra_ok = bool(torch.all(got_all[:, :, dead, :] == 0).item())
            extra = f"all {len(dead)} fully masked rows of every head exactly zero"
        line["parity"] = parity_of(got, sampler.last_out, rows,
                                   "fp64 oracle on the cpu_baseline sample's rows of the "
                                   "timed launches' output", extra_ok, extra)
    del r
    return line


if __name__ == "__main__":
    sys.exit(main())
