"""Benchmark of the MoE dispatch/combine hot path on GB300.

One step = layout + dispatch (ep_layout_dispatch) + combine (ep_combine)
over one batch of the DeepSeek-V3-shaped prefill workload (T=4096 tokens,
H=7168 bf16, E=256 experts, top-8), inputs resident in HBM. The headline
runs on all SMs; the same step is also timed as three calls
(ep_get_dispatch_layout, ep_dispatch, ep_combine) with a per-kernel
breakdown, with a 24-SM budget and in a 24-SM partition. Prints ONE JSON
line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (torchrun): every rank runs an independent replica on its own GPU
(the path has no exchange step on one GPU: replicas only); value = tokens
of all ranks / max-over-ranks time.
--impl reference: the CPU oracle (single thread) on a bounded sample of the
same workload, timed as the reference arm.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from combine_movement_gb300 import workloads as W  # noqa: E402

METRIC = "dispatch+combine tokens/s and HBM GB/s (% of GB300 peak) at 24 SMs / all SMs"
FALLBACK_HBM_GBS = 6800.0
# GB300's nominal HBM3e bandwidth (~8 TB/s); fractions of it are reported
# beside those of the measured copy peak, which is the practical ceiling.
NOMINAL_HBM_GBS = 7900.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# bytes the method must move (per launch)

def algorithmic_bytes(T: int, H: int, K: int, E: int, R: int) -> dict:
    row = 2 * H
    return {
        "layout": 8 * T * K + 4 * T * K + 4 * E + 4 * (E + 1),
        "dispatch": T * row + R * row + 4 * T * K,
        "combine": R * row + 4 * T * K + 4 * T * K + T * row,
    }


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: torch copy_, read+write bytes)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def sources_sha256(names) -> str:
    """sha256 over the named kernel sources (csrc/), concatenated in order."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "combine_movement_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, or None if absent
    or taken on a different version of the kernel's sources (the .cu and
    the headers it includes)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
        if sources_sha256(rec["sources"]) != rec["sources_sha256"]:
            return None
        return int(rec["bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the step

class Buffers:
    """Device buffers of one step (inputs, layout, receive buffer, output)."""

    def __init__(self, ep, wl: W.Workload, dev: torch.device):
        T, H, E, K = wl.T, wl.H, wl.E, wl.K
        self.x = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.idx = torch.empty((T, K), dtype=torch.int64, device=dev)
        self.w = torch.empty((T, K), dtype=torch.float32, device=dev)
        self.counts = torch.empty(E, dtype=torch.int32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        self.slot = torch.empty((T, K), dtype=torch.int32, device=dev)
        nws = ep.ep_layout_workspace_bytes(T, K, E)
        self.ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None
        self.recv_x = torch.empty((T * K, H), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)


class Step:
    """The three calls of one step on a set of device buffers."""

    def __init__(self, ep, inp: W.Inputs, dev: torch.device):
        wl = inp.wl
        self.ep, self.wl, self.dev = ep, wl, dev
        self.T, self.H, self.E, self.K = wl.T, wl.H, wl.E, wl.K
        self.R = wl.T * wl.K
        self.b = Buffers(ep, wl, dev)
        self.b.x.copy_(inp.x)
        self.b.idx.copy_(inp.topk_idx)
        self.b.w.copy_(inp.topk_w)
        self.layout_launches = ep.ep_layout_launches(self.T, self.K, self.E)
        # 2 where dispatch or combine adds a tail launch (the whole GPU,
        # prefill sizes)
        self.dispatch_launches = ep.ep_dispatch_launches(self.T, self.H, self.K)
        self.combine_launches = ep.ep_combine_launches(self.T, self.H, self.K)
        # x larger than 8 MB is rotated over four device copies, so that no
        # dispatch finds the previous call's x in L2 (the rotated copies
        # together exceed it); decode-size x stays warm, as in a decode loop
        self.x_ring = [self.b.x]
        if self.b.x.numel() * 2 > (8 << 20):
            self.x_ring += [self.b.x.clone() for _ in range(3)]
        self._xi = 0
        # the experts between dispatch and combine are a fixed stand-in
        self.layout(self.b)
        self.dispatch(self.b)
        self.expert_out = W.expert_standin(self.b.recv_x, wl.expert_scale)
        torch.cuda.synchronize(dev)

    def layout(self, b: Buffers, stream=None):
        self.ep.ep_get_dispatch_layout(b.idx, self.E, b.counts, b.offsets, b.slot, b.ws,
                                       b.status, stream)

    def next_x(self, b: Buffers) -> torch.Tensor:
        if b is not self.b:
            return b.x
        x = self.x_ring[self._xi]
        self._xi = (self._xi + 1) % len(self.x_ring)
        return x

    def dispatch(self, b: Buffers, stream=None):
        self.ep.ep_dispatch(self.next_x(b), b.slot, b.recv_x, None, None, None, b.status, stream)

    def combine(self, b: Buffers, stream=None):
        self.ep.ep_combine(self.expert_out, b.slot, b.w, b.y, b.status, stream)

    def layout_dispatch(self, b: Buffers, stream=None):
        self.ep.ep_layout_dispatch(b.idx, self.E, self.next_x(b), b.counts, b.offsets, b.slot,
                                   b.recv_x, None, None, None, b.status, stream)

    def run(self, b: Buffers, stream=None):
        self.layout(b, stream)
        self.dispatch(b, stream)
        self.combine(b, stream)

    def run_fused(self, b: Buffers, stream=None):
        self.layout_dispatch(b, stream)
        self.combine(b, stream)

    @property
    def launches_per_step(self) -> int:
        return self.layout_launches + self.dispatch_launches + self.combine_launches


def barrier(dist_on: bool):
    if dist_on:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, dist_on: bool) -> float:
    if not dist_on:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_steps(step: Step, steps: int, warmup: int, dist_on: bool, stream: torch.cuda.Stream,
               sampler_index: int = -1) -> dict:
    """W untimed steps, then exactly K steps between barrier+synchronize,
    timed by CUDA events on the launching stream around the whole loop (the
    headline: nothing between the kernels, so each may start while the
    previous one finishes). Then K more steps with an event between every
    two kernels for the per-kernel breakdown; those events stop the kernels
    from overlapping, so that pass can be a little slower at small budgets
    (its total is reported as total_ms_kernel_events)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step.run(step.b, stream)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(dist_on)
        sampler = ClockSampler(sampler_index) if sampler_index >= 0 else None
        if sampler:
            sampler.__enter__()
        start.record(stream)
        for _ in range(steps):
            step.run(step.b, stream)
        end.record(stream)
        torch.cuda.synchronize()
        if sampler:
            sampler.__exit__(None, None, None)
        barrier(dist_on)
        total_ms = start.elapsed_time(end)

        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        start2 = torch.cuda.Event(enable_timing=True)
        end2 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        start2.record(stream)
        for i in range(steps):
            e = ev[i]
            e[0].record(stream)
            step.layout(step.b, stream)
            e[1].record(stream)
            step.dispatch(step.b, stream)
            e[2].record(stream)
            step.combine(step.b, stream)
            e[3].record(stream)
        end2.record(stream)
        torch.cuda.synchronize()
        # K steps of dispatch + combine alone (the layout of the last pass
        # still in place): the step's cost without the layout
        start3 = torch.cuda.Event(enable_timing=True)
        end3 = torch.cuda.Event(enable_timing=True)
        start3.record(stream)
        for _ in range(steps):
            step.dispatch(step.b, stream)
            step.combine(step.b, stream)
        end3.record(stream)
        # K launches of each copy kernel back to back, events only around the
        # loop: its average launch duration (the next launch's start hides
        # behind the previous one's end, as it does between the kernels of
        # the step; an event between two kernels does not let it)
        b2b = {}
        for name, fn in (("dispatch", step.dispatch), ("combine", step.combine)):
            fn(step.b, stream)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                fn(step.b, stream)
            e1.record(stream)
            b2b[name] = (e0, e1)
        torch.cuda.synchronize()
    lay = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
    dis = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]
    com = [ev[i][2].elapsed_time(ev[i][3]) for i in range(steps)]
    return {"total_ms": total_ms, "total_ms_kernel_events": start2.elapsed_time(end2),
            "dispatch_combine_total_ms": start3.elapsed_time(end3),
            "b2b_ms": {k: e0.elapsed_time(e1) / steps for k, (e0, e1) in b2b.items()},
            "layout_ms": lay, "dispatch_ms": dis, "combine_ms": com,
            "clocks": sampler.summary() if sampler else None}


def calls_b2b_us(fn, stream, n: int) -> float:
    """Average duration of n calls of fn(stream) back to back on `stream`
    (CUDA events around the loop only)."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn(stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn(stream)
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n * 1e3


def time_fused_steps(step: Step, steps: int, warmup: int, dist_on: bool,
                     stream: torch.cuda.Stream, sampler_index: int = -1) -> dict:
    """The step with layout and dispatch in one call (ep_layout_dispatch), the
    headline: W untimed steps, then exactly K steps between barrier +
    synchronize, CUDA events on the launching stream around the loop only
    (the SM clock sampled meanwhile); then a pass with events between the
    calls for the per-call breakdown (as in time_steps)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step.run_fused(step.b, stream)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(dist_on)
        sampler = ClockSampler(sampler_index) if sampler_index >= 0 else None
        if sampler:
            sampler.__enter__()
        start.record(stream)
        for _ in range(steps):
            step.run_fused(step.b, stream)
        end.record(stream)
        torch.cuda.synchronize()
        if sampler:
            sampler.__exit__(None, None, None)
        barrier(dist_on)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            e = ev[i]
            e[0].record(stream)
            step.layout_dispatch(step.b, stream)
            e[1].record(stream)
            step.combine(step.b, stream)
            e[2].record(stream)
        torch.cuda.synchronize()
    return {"total_ms": start.elapsed_time(end),
            "layout_dispatch_ms": [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)],
            "combine_ms": [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)],
            "clocks": sampler.summary() if sampler else None}


def time_e2e(step: Step, inp: W.Inputs, steps: int, warmup: int) -> dict:
    """The headline step (ep_layout_dispatch + ep_combine) through the public
    API with host-resident inputs: every
    step copies x, topk_idx and topk_w from pinned host memory to the device
    and reads y back, inside the timed region. Two device buffer sets and
    separate copy streams let step i's copies overlap step i-1's kernels,
    as a caller pipelining batches would."""
    dev = step.dev
    hx = inp.x.pin_memory()
    hidx = inp.topk_idx.pin_memory()
    hw = inp.topk_w.pin_memory()
    hy = [torch.empty(step.b.y.shape, dtype=step.b.y.dtype).pin_memory() for _ in range(2)]
    # two buffer sets of their own (step.b's x is rotated over copies the
    # host copy would not reach)
    bufs = [Buffers(step.ep, step.wl, dev) for _ in range(2)]
    h2d = hx.numel() * hx.element_size() + hidx.numel() * 8 + hw.numel() * 4
    d2h = hy[0].numel() * hy[0].element_size()
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    done = [torch.cuda.Event() for _ in range(2)]   # kernels of the buffer set finished
    out = [torch.cuda.Event() for _ in range(2)]    # its y was read back
    for e in done + out:
        e.record(s_run)

    def one(i: int):
        j = i % 2
        b = bufs[j]
        ready = torch.cuda.Event()
        with torch.cuda.stream(s_in):
            s_in.wait_event(done[j])
            b.x.copy_(hx, non_blocking=True)
            b.idx.copy_(hidx, non_blocking=True)
            b.w.copy_(hw, non_blocking=True)
            ready.record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ready)
            s_run.wait_event(out[j])
            step.run_fused(b, s_run)
            done[j].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[j])
            hy[j].copy_(b.y, non_blocking=True)
            out[j].record(s_out)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        one(warmup + i)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_run)
    end.record(s_in)
    torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end) / steps
    return {"ms_per_step": ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and reference arm)

def oracle_sample(inp: W.Inputs, tokens: int):
    """Run the oracle's layout -> dispatch -> combine on the first `tokens`
    tokens of the workload; returns seconds."""
    import oracle
    o = oracle.Oracle()
    idx = np.ascontiguousarray(inp.topk_idx.numpy()[:tokens])
    xb = np.ascontiguousarray(inp.x_bits()[:tokens])
    w = np.ascontiguousarray(inp.topk_w.numpy()[:tokens])
    t0 = time.perf_counter()
    _, offsets, slot, _ = o.layout(idx, inp.wl.E)
    recv, _, _ = o.dispatch(xb, slot, int(offsets[-1]))
    o.combine(recv, slot, w)
    return time.perf_counter() - t0


def cpu_baseline(inp: W.Inputs, budget_s: float = 10.0) -> dict:
    tokens = min(inp.wl.T, 1024)
    done, spent = 0, 0.0
    while spent < budget_s and done < 64:
        spent += oracle_sample(inp, tokens)
        done += 1
    return {"value": tokens * done / spent, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "host_cores": os.cpu_count(),
            "sample": f"first {tokens} tokens of {inp.wl.name} (layout+dispatch+combine, "
                      f"identity experts), {done} repetitions, {spent:.1f} s single-threaded"}


def run_reference(args, wl: W.Workload, rank: int) -> None:
    if rank != 0:
        return
    inp = W.make_inputs(wl)
    tokens = min(wl.T, 256)
    for _ in range(args.warmup):
        oracle_sample(inp, tokens)
    secs = [oracle_sample(inp, tokens) for _ in range(args.steps)]
    total = sum(secs)
    value = tokens * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl_desc(wl), "sample_tokens": tokens},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {tokens} of {wl.T} tokens per step, single-threaded C oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def wl_desc(wl: W.Workload) -> str:
    return (f"{wl.name}: T={wl.T} H={wl.H} bf16 E={wl.E} top-{wl.K} {wl.routing} routing, "
            f"expert stand-in x{wl.expert_scale}")


# ---------------------------------------------------------------------------
# per-kernel timing with a cold L2 (decode latency, SM-budget sweep)

class _Flusher:
    """Writes a buffer larger than L2 between timed calls."""

    def __init__(self, dev):
        self.buf = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB

    def __call__(self):
        self.buf.zero_()


def spread(ms: list) -> list:
    """Median, 10th and 90th percentile of per-call event times, in µs."""
    q = statistics.quantiles([1e3 * v for v in ms], n=10)
    return [round(1e3 * statistics.median(ms), 2), round(q[0], 2), round(q[-1], 2)]


def time_call(fn, reps: int, flush=None) -> float:
    """Microseconds of fn() on the current stream (CUDA events): the mean of
    the middle 80 % of `reps` calls. Event timestamps on this GPU are
    quantised near 1 us, so a median would be too; the trimmed mean of calls
    that jitter across the quanta is not. The GPU is kept busy (L2 flush,
    or a ~100 us spin, longer than the host takes to enqueue a step through
    the Python binding) while the host enqueues the call, so host launch
    overhead is not counted."""
    ts = []
    for i in range(reps + 3):
        if flush is not None:
            flush()
        else:
            torch.cuda._sleep(200000)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        if i >= 3:
            ts.append(a.elapsed_time(b) * 1e3)
    ts.sort()
    cut = len(ts) // 10
    return statistics.mean(ts[cut:len(ts) - cut])


def empty_launch_us(reps: int = 200) -> float:
    """Event-to-event time of one empty kernel launched the same way as a
    timed call (after a spin): the launch and event overhead every single-
    kernel figure below carries."""
    return time_call(lambda: torch.cuda._sleep(0), reps)


def per_sm_ceilings(dev, budgets) -> dict:
    """Write-only and read-only rates of plain 16-byte streaming kernels (the
    probes of --ceilings) on n SMs, one 1024-thread CTA per SM: over 1 GiB
    (DRAM) and over 64 MB, 20 launches back to back (L2-resident, like a
    warm decode step). GB/s for the n SMs together; empty where nvcc or the
    probe library is unavailable."""
    import ctypes
    try:
        L = _probe_lib()
    except Exception as e:  # noqa: BLE001 - reported, not fatal
        log(f"per-SM ceilings unavailable: {e}")
        return {}
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    sms_all = torch.cuda.get_device_properties(dev).multi_processor_count
    big = 1 << 30
    a = torch.ones(big, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)

    def best(fn, nbytes, reps=8, per_event=1):
        """Best of `reps` timings; each times `per_event` launches back to
        back between two events (amortising the event and launch overhead
        over short launches)."""
        ts = []
        for i in range(reps + 2):
            s_ = torch.cuda.Event(enable_timing=True)
            e_ = torch.cuda.Event(enable_timing=True)
            s_.record()
            for _ in range(per_event):
                if fn() != 0:
                    raise RuntimeError("probe launch failed")
            e_.record()
            torch.cuda.synchronize()
            if i >= 2:
                ts.append(s_.elapsed_time(e_) / per_event)
        return nbytes / (min(ts) * 1e-3) / 1e9

    out = {}
    small = 64 << 20
    for b in budgets:
        n = min(b or sms_all, sms_all)
        g, blk = (n, 1024) if n < sms_all else (8 * n, 512)
        r = {
            "write_dram_gbs": best(lambda: L.bw_write(vp(a.data_ptr()), sz(big), g, blk), big),
            "read_dram_gbs": best(lambda: L.bw_read(vp(a.data_ptr()), sz(big), vp(sink.data_ptr()),
                                                    g, blk), big),
            "write_l2_gbs": best(lambda: L.bw_write(vp(a.data_ptr()), sz(small), g, blk), small,
                                 5, 20),
            "read_l2_gbs": best(lambda: L.bw_read(vp(a.data_ptr()), sz(small), vp(sink.data_ptr()),
                                                  g, blk), small, 5, 20),
        }
        out[n] = {k: round(v, 1) for k, v in r.items()}
    del a
    torch.cuda.empty_cache()
    return out


def decode_latency(ep, dev, budgets=(16, 24, 0), ceilings: dict | None = None) -> dict:
    """Per-call latency of layout + dispatch + combine on the decode
    workload (T=128, H=7168, E=256, top-8; 16.5 MB, L2-resident when warm),
    at each SM budget: the whole step (warm and cold, both step forms, as a
    CUDA graph, back to back), each kernel timed alone, and the step with
    launch overlap forced on. Each kernel's figure is also given net of the
    event-to-event time of an empty launch, and against what its n SMs can
    move (write ceiling for dispatch, read ceiling for combine; L2-resident
    probes, since the warm step's data sits in L2). Short launches are also
    timed back to back, beside plain 16-byte write-only and read-only
    kernels over the same receive-row bytes on the same n SMs: per launch,
    at this size, ramp and launch spacing weigh as much as bandwidth, and
    those probes are the floor a kernel moving these bytes meets."""
    import ctypes
    wl = W.DECODE
    step = Step(ep, W.make_inputs(wl), dev)
    flush = _Flusher(dev)
    ab = algorithmic_bytes(wl.T, wl.H, wl.K, wl.E, wl.T * wl.K)
    rows = wl.T * wl.K * 2 * wl.H  # receive-row bytes each copy kernel writes or reads
    sms_all = torch.cuda.get_device_properties(dev).multi_processor_count
    overhead = empty_launch_us()
    out = {"workload": wl_desc(wl), "empty_launch_us": round(overhead, 2)}
    mode0 = ep.ep_get_launch_overlap()
    try:
        L = _probe_lib()
    except Exception as e:  # noqa: BLE001 - reported, not fatal
        log(f"same-size probes unavailable: {e}")
        L = None
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    probe_buf = torch.empty(rows, dtype=torch.uint8, device=dev)
    for b in budgets:
        n = min(b or sms_all, sms_all)
        ep.ep_set_num_sms(b)
        warm = time_call(lambda: step.run(step.b), 200)
        cold = time_call(lambda: step.run(step.b), 30, flush)
        fwarm = time_call(lambda: step.run_fused(step.b), 200)
        fcold = time_call(lambda: step.run_fused(step.b), 30, flush)
        k_lay = time_call(lambda: step.layout(step.b), 200)
        k_dis = time_call(lambda: step.dispatch(step.b), 200)
        k_com = time_call(lambda: step.combine(step.b), 200)
        # the same three calls captured once into a CUDA graph and replayed
        # (one host launch per step)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step.run(step.b, torch.cuda.current_stream())
        gwarm = time_call(g.replay, 200)
        ep.ep_set_launch_overlap(1)
        owarm = time_call(lambda: step.run(step.b), 200)
        ep.ep_set_launch_overlap(mode0)

        def back_to_back(fn, n_=500):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n_):
                fn()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n_ * 1e3
        out_b2b = back_to_back(lambda: step.run(step.b))
        graph_b2b = back_to_back(g.replay)
        k_b2b = {"layout": back_to_back(lambda: step.layout(step.b)),
                 "dispatch": back_to_back(lambda: step.dispatch(step.b)),
                 "combine": back_to_back(lambda: step.combine(step.b))}
        probes = None
        if L is not None:
            # one 1024-thread CTA per SM over the receive-row bytes; the read
            # goes over rows the write just left in L2, as combine's do
            def p_write():
                if L.bw_write(vp(probe_buf.data_ptr()), sz(rows), n, 1024) != 0:
                    raise RuntimeError("probe launch failed")

            def p_read():
                if L.bw_read(vp(probe_buf.data_ptr()), sz(rows), vp(sink.data_ptr()), n, 1024) != 0:
                    raise RuntimeError("probe launch failed")
            probes = {"write": back_to_back(p_write), "read": back_to_back(p_read),
                      "empty": back_to_back(lambda: torch.cuda._sleep(0))}
        net = {k: max(v - overhead, 1e-3) for k, v in
               (("layout", k_lay), ("dispatch", k_dis), ("combine", k_com))}
        entry = {
            "num_sms": n,
            "warm_us": round(warm, 2), "cold_us": round(cold, 2),
            "cold_gbs": round((ab["dispatch"] + ab["combine"]) / (cold * 1e-6) / 1e9, 1),
            "fused_warm_us": round(fwarm, 2), "fused_cold_us": round(fcold, 2),
            # the same two warm steps net of what an empty launch measures
            # between the same events (event records and one launch)
            "warm_net_us": round(warm - overhead, 2), "fused_warm_net_us": round(fwarm - overhead, 2),
            "graph_warm_us": round(gwarm, 2),
            "launch_overlap_forced_warm_us": round(owarm, 2),
            # steps issued back to back from the host (no spin in between):
            # the eager calls are bound by the host's launch rate, the graph
            # is not
            "back_to_back_us": round(out_b2b, 2), "graph_back_to_back_us": round(graph_b2b, 2),
            # each kernel alone, warm, event to event (includes one launch)
            "kernel_us": {"layout": round(k_lay, 2), "dispatch": round(k_dis, 2),
                          "combine": round(k_com, 2)},
            "kernel_net_us": {k: round(v, 2) for k, v in net.items()},
            # each kernel launched 500 times back to back, per launch
            "kernel_back_to_back_us": {k: round(v, 2) for k, v in k_b2b.items()},
        }
        if probes:
            entry["same_size_probes_back_to_back_us"] = {
                k: round(v, 2) for k, v in probes.items()}
            entry["same_size_probes_source"] = (
                f"16-byte streaming write-only / read-only kernels over the {rows} receive-row "
                f"bytes on {n} SMs (one 1024-thread CTA per SM), read after write (L2-resident)")
            # probe time / kernel time, both back to back: 1.0 = as fast as a
            # plain stream of the same bytes on the same SMs
            entry["dispatch_frac_of_same_size_write"] = round(probes["write"] / k_b2b["dispatch"], 3)
            entry["combine_frac_of_same_size_read"] = round(probes["read"] / k_b2b["combine"], 3)
        if 0 < b < sms_all:
            # the same step in an SM partition of b SMs (ep_sm_partition): the
            # hardware keeps its kernels on those SMs, and the default policy
            # lets their launches overlap
            try:
                h, _, n_part, _ = ep.ep_sm_partition(b)
                ps = torch.cuda.ExternalStream(h, device=dev)
                with torch.cuda.stream(ps):
                    pw = time_call(lambda: step.run(step.b), 200)
                    pf = time_call(lambda: step.run_fused(step.b), 200)
                    pb = back_to_back(lambda: step.run(step.b))
                entry["partition"] = {"sms": n_part, "warm_us": round(pw, 2),
                                      "fused_warm_us": round(pf, 2),
                                      "warm_net_us": round(pw - overhead, 2),
                                      "fused_warm_net_us": round(pf - overhead, 2),
                                      "back_to_back_us": round(pb, 2)}
            except Exception as e:  # noqa: BLE001 - reported in the line
                entry["partition"] = {"unavailable": str(e)[:200]}
        c = (ceilings or {}).get(n)
        if c:
            w_cap, r_cap = c["write_l2_gbs"], c["read_l2_gbs"]
            entry["budget_ceilings_gbs"] = {"write": w_cap, "read": r_cap,
                                            "source": f"16-byte streaming probes on {n} SMs, "
                                                      "64 MB L2-resident"}
            # receive rows written by dispatch / read by combine, per net second
            entry["dispatch_write_frac_of_budget_ceiling"] = round(
                rows / (net["dispatch"] * 1e-6) / 1e9 / w_cap, 3)
            entry["combine_read_frac_of_budget_ceiling"] = round(
                rows / (net["combine"] * 1e-6) / 1e9 / r_cap, 3)
        out[f"sms_{b or 'all'}"] = entry
        del g
    ep.ep_set_num_sms(0)
    del probe_buf
    return out


def budget_ceiling_frac(c: dict | None, s: dict, step) -> dict | None:
    """Dispatch's receive-row writes and combine's receive-row reads on a
    budget of n SMs, as fractions of the n SMs' own DRAM write-only and
    read-only ceilings (c: per_sm_ceilings entry for n)."""
    if not c:
        return None
    rows = step.R * 2 * step.H
    w = rows / (s["dispatch_us"] * 1e-6) / 1e9
    r = rows / (s["combine_us"] * 1e-6) / 1e9
    return {"num_sms": s["num_sms"],
            "dispatch_write_gbs": round(w, 1), "write_ceiling_gbs": c["write_dram_gbs"],
            "dispatch_frac": round(w / c["write_dram_gbs"], 3),
            "combine_read_gbs": round(r, 1), "read_ceiling_gbs": c["read_dram_gbs"],
            "combine_frac": round(r / c["read_dram_gbs"], 3),
            "ceiling_source": "16-byte streaming write-only / read-only kernels over 1 GiB "
                              f"on {s['num_sms']} SMs (one 1024-thread CTA per SM)"}


def time_workload(ep, dev, wl: W.Workload, budget: int, steps: int, warmup: int,
                  peak: float) -> dict:
    """One workload at one SM budget: K steps back to back (events only
    around the loop) as three calls and with ep_layout_dispatch, the
    three-call step captured once in a CUDA graph and replayed K times, and
    a pass with events between the kernels for the per-kernel medians.
    Inputs resident in HBM."""
    step = Step(ep, W.make_inputs(wl), dev)
    sms_all = torch.cuda.get_device_properties(dev).multi_processor_count
    ep.ep_set_num_sms(budget)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        frun = time_fused_steps(step, steps, warmup, False, stream)
        run = time_steps(step, steps, warmup, False, stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step.run(step.b, stream)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    st = ep.ep_get_status(step.b.status)
    ep.ep_set_num_sms(0)
    if st != 0:
        raise SystemExit(f"{wl.name}: device status {st}: {ep.ep_status_string(st)}")
    ab = algorithmic_bytes(wl.T, wl.H, wl.K, wl.E, step.R)
    ms = run["total_ms"] / steps
    gms = e0.elapsed_time(e1) / steps
    med = {k: statistics.median(run[f"{k}_ms"]) * 1e3 for k in ("layout", "dispatch", "combine")}
    moved = ab["dispatch"] + ab["combine"]
    d_c = med["dispatch"] + med["combine"]
    return {
        "workload": wl_desc(wl), "num_sms": min(budget or sms_all, sms_all),
        "steps": steps,
        "ms_per_step": round(ms, 5), "tokens_per_s": round(wl.T / (ms * 1e-3)),
        # layout + dispatch through ep_layout_dispatch, then ep_combine
        "fused_ms_per_step": round(frun["total_ms"] / steps, 5),
        "fused_tokens_per_s": round(wl.T / (frun["total_ms"] / steps * 1e-3)),
        "graph_ms_per_step": round(gms, 5), "graph_tokens_per_s": round(wl.T / (gms * 1e-3)),
        "step_gbs": round((moved + ab["layout"]) / (min(ms, gms) * 1e-3) / 1e9, 1),
        "kernel_us_median": {k: round(v, 2) for k, v in med.items()},
        "dispatch_gbs": round(ab["dispatch"] / (med["dispatch"] * 1e-6) / 1e9, 1),
        "combine_gbs": round(ab["combine"] / (med["combine"] * 1e-6) / 1e9, 1),
        "dispatch_combine_gbs": round(moved / (d_c * 1e-6) / 1e9, 1),
        "dispatch_combine_frac_of_peak": round(moved / (d_c * 1e-6) / 1e9 / peak, 3),
        "algorithmic_bytes": ab,
    }


def run_workloads(ep, dev, budget: int, steps: int, warmup: int) -> None:
    """Every workload of the measurement plan at all SMs and at `budget`
    SMs: one JSON line each (time_workload), with the SM clock sampled over
    the workload's runs. Small workloads are L2-resident between steps (no
    flush); the large ones are many times the L2."""
    peak, peak_src = peak_hbm()
    wls = [W.TINY, W.DEEPSEEK_PREFILL, W.SKEWED, W.DECODE,
           W.sweep(max(W.SWEEP_T), max(W.SWEEP_H))]
    for wl in wls:
        for b in (0, budget):
            with ClockSampler(dev.index or 0) as cs:
                r = time_workload(ep, dev, wl, b, steps, warmup, peak)
            r["peak_gbs"] = peak
            r["peak_source"] = peak_src
            r["clocks"] = cs.summary()
            print(json.dumps(r), flush=True)
            torch.cuda.empty_cache()


def run_sweep(ep, dev, budgets) -> None:
    """SM-budget and size sweep: one JSON line per (T, H, budget) with each
    kernel's time (time_call's trimmed mean, cold L2) and GB/s against the
    HBM peak."""
    peak, _ = peak_hbm()
    flush = _Flusher(dev)
    sms_all = torch.cuda.get_device_properties(dev).multi_processor_count
    for T in W.SWEEP_T:
        for H in W.SWEEP_H:
            wl = W.sweep(T, H)
            step = Step(ep, W.make_inputs(wl), dev)
            ab = algorithmic_bytes(T, H, wl.K, wl.E, T * wl.K)
            for b in budgets:
                ep.ep_set_num_sms(b)
                lay = time_call(lambda: step.layout(step.b), 20, flush)
                dis = time_call(lambda: step.dispatch(step.b), 20, flush)
                com = time_call(lambda: step.combine(step.b), 20, flush)
                gbs = (ab["dispatch"] + ab["combine"]) / ((dis + com) * 1e-6) / 1e9
                print(json.dumps({
                    "T": T, "H": H, "E": wl.E, "K": wl.K, "num_sms": b or sms_all,
                    "layout_us": round(lay, 1), "dispatch_us": round(dis, 1),
                    "combine_us": round(com, 1),
                    "dispatch_gbs": round(ab["dispatch"] / (dis * 1e-6) / 1e9),
                    "combine_gbs": round(ab["combine"] / (com * 1e-6) / 1e9),
                    "dispatch_combine_gbs": round(gbs), "frac_of_peak": round(gbs / peak, 3),
                    "tokens_per_s": round(T / ((lay + dis + com) * 1e-6)),
                }), flush=True)
            del step
            torch.cuda.empty_cache()
    ep.ep_set_num_sms(0)


# ---------------------------------------------------------------------------
# bandwidth ceilings of this GPU (for reading the roofline fractions)

_CEILING_SRC = r"""
#include <cuda_runtime.h>
#include <cstdint>
__global__ void k_write(uint4* p, size_t n16) {
    const uint4 v = make_uint4(1, 2, 3, 4);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
         i += (size_t)gridDim.x * blockDim.x) p[i] = v;
}
__global__ void k_read(const uint4* p, size_t n16, uint32_t* sink) {
    uint32_t acc = 0;
    size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x, s = (size_t)gridDim.x * blockDim.x;
    for (; i + 3 * s < n16; i += 4 * s) {
        uint4 a = __ldcs(p + i), b = __ldcs(p + i + s), c = __ldcs(p + i + 2 * s), d = __ldcs(p + i + 3 * s);
        acc ^= a.x ^ b.y ^ c.z ^ d.w;
    }
    for (; i < n16; i += s) acc ^= __ldcs(p + i).x;
    if (acc == 0x12345678u) *sink = acc;
}
__global__ void k_copy(const uint4* a, uint4* b, size_t n16) {
    size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x, s = (size_t)gridDim.x * blockDim.x;
    for (; i + s < n16; i += 2 * s) { uint4 x = __ldcs(a + i), y = __ldcs(a + i + s); b[i] = x; b[i + s] = y; }
    for (; i < n16; i += s) b[i] = __ldcs(a + i);
}
__global__ void k_bulk_write(uint8_t* dst, size_t nbytes) {
    extern __shared__ __align__(128) uint8_t sm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
    uint8_t* my = sm + warp * 8192;
    for (int i = lane; i < 8192 / 4; i += 32) reinterpret_cast<uint32_t*>(my)[i] = i;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        size_t chunks = nbytes / 8192, gw = blockIdx.x * (size_t)nw + warp, W = (size_t)gridDim.x * nw;
        uint32_t src = (uint32_t)__cvta_generic_to_shared(my);
        int n = 0;
        for (size_t c = gw; c < chunks; c += W) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                         :: "l"(dst + c * 8192), "r"(src), "r"(8192) : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            if (++n >= 8) { asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); n = 4; }
        }
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
}
// Stage probes for the two-stage pipeline model of the dispatch ring: the
// same per-warp ring shape (3 or 4 stages, 2 loads ahead, one elected lane, the
// same chunk and units per warp) doing only its load stage or only its store
// stage, over buffers of their own. Every mbarrier wait gives up after 2 s
// and records it in *err; after a give-up the lane still waits (bounded) for
// the loads it issued, so no copy lands in shared memory after the CTA ends.
constexpr int kP = 2;
__device__ __forceinline__ bool probe_wait(uint32_t bar, uint32_t parity) {
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (true) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > 2000000000ull) return false;
    }
}
template <int kNS>
__host__ __device__ constexpr uint32_t ring_region(int warps) { return (8u * kNS * warps + 127u) & ~127u; }
template <int kNS>
__global__ void k_ring_load(const uint8_t* src, long long units, uint32_t chunk, int* err) {
    extern __shared__ __align__(128) uint8_t sm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
    if (lane != 0) return;
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(sm);
    const uint32_t bar0 = base + 8u * kNS * warp;
    const uint32_t buf0 = base + ring_region<kNS>(nw) + kNS * chunk * warp;
    for (int s = 0; s < kNS; ++s) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar0 + 8u * s) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const long long W = (long long)gridDim.x * nw, gw = (long long)blockIdx.x * nw + warp;
    const long long u0 = units * gw / W, n = units * (gw + 1) / W - u0;
    long long issued = 0;
    auto issue = [&]() {
        const int s = (int)(issued % kNS);
        const uint32_t bar = bar0 + 8u * s;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(chunk) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     :: "r"(buf0 + s * chunk), "l"(src + (u0 + issued) * (long long)chunk), "r"(chunk), "r"(bar) : "memory");
        ++issued;
    };
    while (issued < kP && issued < n) issue();
    for (long long j = 0; j < n; ++j) {
        if (issued < n) issue();  // its stage was last used by unit issued-kNS < j, already waited
        if (!probe_wait(bar0 + 8u * (j % kNS), (uint32_t)((j / kNS) & 1))) {
            atomicExch(err, 1);
            for (long long q = j + 1; q < issued; ++q) probe_wait(bar0 + 8u * (q % kNS), (uint32_t)((q / kNS) & 1));
            return;
        }
    }
}
template <int kNS>
__global__ void k_ring_store(uint8_t* dst, long long units, uint32_t chunk, int K) {
    extern __shared__ __align__(128) uint8_t sm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
    uint8_t* mine = sm + ring_region<kNS>(nw) + (size_t)kNS * chunk * warp;
    for (uint32_t i = lane; i < kNS * chunk / 4; i += 32) reinterpret_cast<uint32_t*>(mine)[i] = i;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane != 0) return;
    const uint32_t buf0 = (uint32_t)__cvta_generic_to_shared(mine);
    const long long W = (long long)gridDim.x * nw, gw = (long long)blockIdx.x * nw + warp;
    const long long u0 = units * gw / W, n = units * (gw + 1) / W - u0;
    for (long long j = 0; j < n; ++j) {
        asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(kNS - kP - 1) : "memory");
        const uint32_t src = buf0 + (uint32_t)(j % kNS) * chunk;
        for (int k = 0; k < K; ++k)
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                         :: "l"(dst + ((u0 + j) * K + k) * (long long)chunk), "r"(src), "r"(chunk) : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
template <int kNS>
int ring_load_ns(const void* src, long long units, unsigned chunk, int grid, int warps, int* err) {
    const int smem = (int)(ring_region<kNS>(warps) + (size_t)kNS * chunk * warps);
    cudaError_t e = cudaFuncSetAttribute(k_ring_load<kNS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k_ring_load<kNS><<<grid, warps * 32, smem>>>((const uint8_t*)src, units, chunk, err); return cudaGetLastError(); }
template <int kNS>
int ring_store_ns(void* dst, long long units, unsigned chunk, int K, int grid, int warps) {
    const int smem = (int)(ring_region<kNS>(warps) + (size_t)kNS * chunk * warps);
    cudaError_t e = cudaFuncSetAttribute(k_ring_store<kNS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k_ring_store<kNS><<<grid, warps * 32, smem>>>((uint8_t*)dst, units, chunk, K); return cudaGetLastError(); }
extern "C" {
int bw_write(void* p, size_t n, int grid, int block) { k_write<<<grid, block>>>((uint4*)p, n / 16); return cudaGetLastError(); }
int bw_read(void* p, size_t n, void* sink, int grid, int block) { k_read<<<grid, block>>>((const uint4*)p, n / 16, (uint32_t*)sink); return cudaGetLastError(); }
int bw_copy(void* a, void* b, size_t n, int grid, int block) { k_copy<<<grid, block>>>((const uint4*)a, (uint4*)b, n / 16); return cudaGetLastError(); }
int bw_copy_on(void* a, void* b, size_t n, int grid, int block, void* stream) {
    k_copy<<<grid, block, 0, (cudaStream_t)stream>>>((const uint4*)a, (uint4*)b, n / 16); return cudaGetLastError(); }
int host_dev_ptr(void* host, void** dev) { return cudaHostGetDevicePointer(dev, host, 0); }
int bw_bulk_write(void* p, size_t n, int grid, int warps) {
    cudaFuncSetAttribute(k_bulk_write, cudaFuncAttributeMaxDynamicSharedMemorySize, warps * 8192);
    k_bulk_write<<<grid, warps * 32, warps * 8192>>>((uint8_t*)p, n); return cudaGetLastError(); }
int ring_load(const void* src, long long units, unsigned chunk, int grid, int warps, int stages, int* err) {
    return stages == 3 ? ring_load_ns<3>(src, units, chunk, grid, warps, err)
                       : ring_load_ns<4>(src, units, chunk, grid, warps, err); }
int ring_store(void* dst, long long units, unsigned chunk, int K, int grid, int warps, int stages) {
    return stages == 3 ? ring_store_ns<3>(dst, units, chunk, K, grid, warps)
                       : ring_store_ns<4>(dst, units, chunk, K, grid, warps); }
}
"""


@functools.lru_cache(maxsize=1)
def _probe_lib():
    """The probes above, built with nvcc into a temporary directory (once per
    process)."""
    import ctypes
    import tempfile
    tmp = tempfile.mkdtemp(prefix="ep_probes_")
    src, so = os.path.join(tmp, "bw.cu"), os.path.join(tmp, "libbw.so")
    with open(src, "w") as f:
        f.write(_CEILING_SRC)
    subprocess.run(["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC",
                    "-gencode=arch=compute_103a,code=sm_103a", "-o", so, src], check=True)
    return ctypes.CDLL(so)


def pipeline_time(n: int, t_load: float, t_store: float) -> float:
    """Two-stage pipeline closed form ("tensor-memory-accelerator" atlas page,
    Science and assumptions): the first unit pays both stages, each of the
    other n-1 units one interval of the slower stage."""
    return 0.0 if n <= 0 else t_load + t_store + (n - 1) * max(t_load, t_store)


def run_pipeline_model(ep, dev, wl: W.Workload, budgets=(0, 24, 16)) -> None:
    """Model dispatch as the two-stage pipeline its ring implements and
    compare with the measured kernel. Per SM budget: time the ring's load
    stage alone and its store stage alone (same ring shape, chunk, units per
    warp; probes above), take per-unit stage times t = stage time / N with
    N = units per warp, and print the closed form, the serial sum and the
    measured dispatch time (all cold L2, time_call's trimmed means). One
    JSON line per budget."""
    import ctypes
    L = _probe_lib()
    step = Step(ep, W.make_inputs(wl), dev)
    flush = _Flusher(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sms_all = torch.cuda.get_device_properties(dev).multi_processor_count
    warps = 8  # warps per dispatch CTA in the library's build
    row = 2 * wl.H
    for b in budgets:
        ep.ep_set_num_sms(b)
        grid = min(b or sms_all, sms_all)
        chunk = ep.ep_dispatch_chunk_bytes(wl.T, wl.H, wl.K)
        if chunk <= 0:
            raise SystemExit("ep_dispatch_chunk_bytes failed")
        n_chunks = -(-row // chunk)
        units = wl.T * n_chunks
        src = torch.empty(units * chunk, dtype=torch.uint8, device=dev)
        dst = torch.empty(units * wl.K * chunk, dtype=torch.uint8, device=dev)
        vp, ll, u32 = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_uint
        errp = ctypes.cast(err.data_ptr(), ctypes.POINTER(ctypes.c_int))

        stages = ep.ep_dispatch_ring_stages()

        def load():
            if L.ring_load(vp(src.data_ptr()), ll(units), u32(chunk), grid, warps, stages, errp) != 0:
                raise SystemExit("ring load probe: launch failed")

        def store():
            if L.ring_store(vp(dst.data_ptr()), ll(units), u32(chunk), wl.K, grid, warps,
                            stages) != 0:
                raise SystemExit("ring store probe: launch failed")

        t_load = time_call(load, 20, flush)
        t_store = time_call(store, 20, flush)
        t_disp = time_call(lambda: step.dispatch(step.b), 20, flush)
        if int(err.item()) != 0:
            raise SystemExit("ring load probe: a wait gave up")
        n = -(-units // (grid * warps))
        model = pipeline_time(n, t_load / n, t_store / n)
        print(json.dumps({
            "workload": wl.name, "num_sms": grid, "chunk_bytes": chunk, "ring_stages": stages,
            "units_per_warp": n,
            "load_stage_us": round(t_load, 1), "store_stage_us": round(t_store, 1),
            "model_pipelined_us": round(model, 1), "model_serial_us": round(t_load + t_store, 1),
            "dispatch_us": round(t_disp, 1), "dispatch_over_model": round(t_disp / model, 3),
        }), flush=True)
        del src, dst
        torch.cuda.empty_cache()
    ep.ep_set_num_sms(0)


def measure_ceilings(dev) -> dict:
    """Write-only, read-only and copy bandwidth of plain streaming kernels
    (16-byte vectors; 8 KB bulk stores), all SMs and 24 SMs, plus pinned
    host<->device rates: copy engines one way and both ways at once, and the
    copy kernel reading or writing the pinned buffers directly (zero-copy).
    Built from the source above with nvcc."""
    import ctypes
    L = _probe_lib()
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n = 1 << 30
    a = torch.ones(n, dtype=torch.uint8, device=dev)
    b = torch.empty(n, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)

    def best(fn, nbytes):
        ts = []
        for i in range(12):
            s_ = torch.cuda.Event(enable_timing=True)
            e_ = torch.cuda.Event(enable_timing=True)
            s_.record()
            assert fn() == 0
            e_.record()
            torch.cuda.synchronize()
            if i >= 2:
                ts.append(s_.elapsed_time(e_))
        return round(nbytes / (min(ts) * 1e-3) / 1e9)

    r = {}
    for tag, g, blk in (("all_sms", sms * 8, 512), ("sms_24", 24, 1024)):
        r[f"write_{tag}"] = best(lambda: L.bw_write(vp(a.data_ptr()), sz(n), g, blk), n)
        r[f"read_{tag}"] = best(lambda: L.bw_read(vp(a.data_ptr()), sz(n), vp(sink.data_ptr()), g, blk), n)
        r[f"copy_{tag}"] = best(lambda: L.bw_copy(vp(a.data_ptr()), vp(b.data_ptr()), sz(n), g, blk), 2 * n)
    r["bulk_write_all_sms"] = best(lambda: L.bw_bulk_write(vp(a.data_ptr()), sz(n), sms, 8), n)
    r["bulk_write_sms_24"] = best(lambda: L.bw_bulk_write(vp(a.data_ptr()), sz(n), 24, 24), n)
    m = 59 * 1024 * 1024
    h = torch.ones(m, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(m, dtype=torch.uint8).pin_memory()
    d = torch.empty(m, dtype=torch.uint8, device=dev)
    d2 = torch.ones(m, dtype=torch.uint8, device=dev)
    r["h2d_gbs"] = best(lambda: (d.copy_(h, non_blocking=True), 0)[1], m)
    r["d2h_gbs"] = best(lambda: (h.copy_(d, non_blocking=True), 0)[1], m)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def both(f1, f2):
        ev = torch.cuda.Event()
        ev.record()
        s1.wait_event(ev)
        s2.wait_event(ev)
        f1(s1)
        f2(s2)
        for s_ in (s1, s2):
            e_ = torch.cuda.Event()
            e_.record(s_)
            torch.cuda.current_stream().wait_event(e_)
        return 0

    def ce(dst, src):
        def f(s_):
            with torch.cuda.stream(s_):
                dst.copy_(src, non_blocking=True)
        return f
    r["h2d_d2h_concurrent_gbs"] = best(lambda: both(ce(d, h), ce(h2, d2)), 2 * m)
    # SM-driven zero-copy: the copy kernel loads from / stores to the pinned
    # buffers through their device pointers (16-byte vectors)
    hp, hp2 = ctypes.c_void_p(), ctypes.c_void_p()
    if L.host_dev_ptr(vp(h.data_ptr()), ctypes.byref(hp)) == 0 and \
            L.host_dev_ptr(vp(h2.data_ptr()), ctypes.byref(hp2)) == 0:
        def sm(src, dst, g):
            return lambda s_: L.bw_copy_on(src, dst, sz(m), g, 1024, vp(s_.cuda_stream))
        for g in (16, 152):
            r[f"sm_h2d_gbs_{g}"] = best(lambda: L.bw_copy(hp, vp(d.data_ptr()), sz(m), g, 1024), m)
            r[f"sm_d2h_gbs_{g}"] = best(lambda: L.bw_copy(vp(d2.data_ptr()), hp2, sz(m), g, 1024), m)
        r["sm_h2d_d2h_concurrent_gbs"] = best(
            lambda: both(sm(hp, vp(d.data_ptr()), 32), sm(vp(d2.data_ptr()), hp2, 32)), 2 * m)
    return r


# ---------------------------------------------------------------------------
# overlap: data movement on n SMs next to arithmetic on the other SMs

_SPIN_SRC = r"""
#include <cuda_runtime.h>
// ALU-bound stand-in for the experts' arithmetic: every thread runs a chain
// of fp32 fmas; one CTA per SM (its shared-memory request forbids a second).
__global__ void k_fma(float* out, int iters) {
    float a = threadIdx.x * 1e-3f, b = 1.0f + blockIdx.x * 1e-6f, c = 0.5f, d = 0.25f;
    for (int i = 0; i < iters; ++i) {
        a = fmaf(a, b, c); c = fmaf(c, b, d); d = fmaf(d, b, a); b = fmaf(b, 0.999999f, 1e-7f);
    }
    if (a + c + d == 12345.0f) out[0] = a;
}
extern "C" int run_fma(void* out, int grid, int iters, void* stream) {
    cudaFuncSetAttribute(k_fma, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024);
    k_fma<<<grid, 1024, 120 * 1024, (cudaStream_t)stream>>>((float*)out, iters);
    return cudaGetLastError();
}
"""


def run_overlap(ep, dev, wl: W.Workload, budgets=(16, 24, 48), steps: int = 60) -> None:
    """For each budget n: time (a) an ALU-bound kernel on 152-n SMs alone,
    (b) `steps` dispatch+combine steps of `wl` (layout done beforehand) at
    budget n alone, (c) both at once on two streams. Decode-size workloads
    run the whole step (layout included) and 20x the steps. One JSON line
    per budget and launch-overlap mode, with the SM clock sampled during (c)."""
    import ctypes
    import tempfile
    tmp = tempfile.mkdtemp(prefix="ep_overlap_")
    src, so = os.path.join(tmp, "spin.cu"), os.path.join(tmp, "libspin.so")
    with open(src, "w") as f:
        f.write(_SPIN_SRC)
    subprocess.run(["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC",
                    "-gencode=arch=compute_103a,code=sm_103a", "-o", so, src], check=True)
    L = ctypes.CDLL(so)
    L.run_fma.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.zeros(1, device=dev)
    step = Step(ep, W.make_inputs(wl), dev)
    small = wl.T * wl.K * wl.H * 2 < (64 << 20)  # receive rows under 64 MB
    if small:
        steps *= 20
    s_move = torch.cuda.Stream(dev, priority=-1)
    s_comp = torch.cuda.Stream(dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def movement(n_steps):
        for _ in range(n_steps):
            if small:
                step.layout(step.b, s_move)
            step.dispatch(step.b, s_move)
            step.combine(step.b, s_move)

    plain = (s_move, s_comp)
    cases = [(n, m, False) for n in budgets for m in (0, 1)] + [(n, 0, True) for n in budgets]
    for n, mode, part in cases:
        ep.ep_set_num_sms(n)
        ep.ep_set_launch_overlap(mode)  # 0: library default (no overlap below the full budget)
        grid = sms - n
        s_move, s_comp = plain
        if part:
            # movement in an SM partition of n SMs, the ALU kernel in the
            # partition of the other SMs (the default policy overlaps
            # launches in a partition)
            h, hr, n_part, n_rest = ep.ep_sm_partition(n)
            s_move = torch.cuda.ExternalStream(h, device=dev)
            s_comp = torch.cuda.ExternalStream(hr, device=dev)
            grid = n_rest
        with torch.cuda.stream(s_move):
            movement(3)
        torch.cuda.synchronize(dev)
        # (b) movement alone
        a0, a1 = ev(), ev()
        a0.record(s_move)
        movement(steps)
        a1.record(s_move)
        torch.cuda.synchronize(dev)
        move_ms = a0.elapsed_time(a1)
        # size the ALU kernel to last about as long as the movement
        c0, c1 = ev(), ev()
        c0.record(s_comp)
        assert L.run_fma(out.data_ptr(), grid, 20000, s_comp.cuda_stream) == 0
        c1.record(s_comp)
        torch.cuda.synchronize(dev)
        iters = max(20000, int(20000 * move_ms / max(c0.elapsed_time(c1), 1e-3)))
        # (a) ALU alone
        c0.record(s_comp)
        L.run_fma(out.data_ptr(), grid, iters, s_comp.cuda_stream)
        c1.record(s_comp)
        torch.cuda.synchronize(dev)
        comp_ms = c0.elapsed_time(c1)
        # (c) both
        sampler = ClockSampler(dev.index or 0)
        sampler.__enter__()
        c0.record(s_comp)
        L.run_fma(out.data_ptr(), grid, iters, s_comp.cuda_stream)
        c1.record(s_comp)
        a0.record(s_move)
        movement(steps)
        a1.record(s_move)
        torch.cuda.synchronize(dev)
        sampler.__exit__(None, None, None)
        flops = 4 * 2 * iters * 1024 * grid
        print(json.dumps({
            "workload": wl.name, "step": "layout+dispatch+combine" if small else "dispatch+combine",
            "num_sms_movement": n, "num_sms_alu": grid, "steps": steps,
            "launch_overlap": ("auto (on in a partition)" if part else
                               "auto (off below the full budget)") if mode == 0 else "forced on",
            "sm_partition": part,
            "movement_ms_per_step_alone": round(move_ms / steps, 4),
            "movement_ms_per_step_overlapped": round(a0.elapsed_time(a1) / steps, 4),
            "alu_ms_alone": round(comp_ms, 3), "alu_ms_overlapped": round(c0.elapsed_time(c1), 3),
            "alu_tflops_alone": round(flops / (comp_ms * 1e-3) / 1e12, 2),
            "alu_tflops_overlapped": round(flops / (c0.elapsed_time(c1) * 1e-3) / 1e12, 2),
            "clocks_overlapped": sampler.summary(),
        }), flush=True)
    ep.ep_set_num_sms(0)
    ep.ep_set_launch_overlap(0)


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="deepseek-v3-prefill", choices=sorted(W.BY_NAME))
    ap.add_argument("--budget-sms", type=int, default=24, help="second SM budget to report")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (same shapes and seed; for "
                         "profiling captures on a smaller case of the same kernels)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: the T x H x SM-budget sweep, one JSON line each")
    ap.add_argument("--overlap", action="store_true",
                    help="instead of the bench line: dispatch+combine of --workload on n SMs "
                         "next to an ALU-bound kernel on the other SMs (n = 16, 24, 48)")
    ap.add_argument("--pipeline-model", action="store_true",
                    help="two-stage pipeline model of the dispatch ring vs the measured kernel")
    ap.add_argument("--ceilings", action="store_true",
                    help="instead of the bench line: bandwidth ceilings of plain streaming kernels")
    ap.add_argument("--only-main", action="store_true",
                    help="for profiling: only the all-SM timed loop (no 24-SM, fused, e2e or "
                         "decode passes)")
    ap.add_argument("--decode", action="store_true",
                    help="instead of the bench line: only the decode-latency breakdown "
                         "(16, 24, all SMs) as one JSON line")
    ap.add_argument("--workloads", action="store_true",
                    help="instead of the bench line: one JSON line per workload (tiny, "
                         "DeepSeek-V3 prefill, skewed Zipf, decode, largest sweep point) at "
                         "all SMs and at --budget-sms")
    ap.add_argument("--dispatch-tail", type=int, default=-1,
                    help="percentage of a full-GPU dispatch's units its tail launch takes "
                         "(ep_set_dispatch_tail; 0: one persistent launch; default: the "
                         "library's)")
    ap.add_argument("--combine-tail", type=int, default=-1,
                    help="the same for combine (ep_set_combine_tail)")
    ap.add_argument("--ncu-budgets", action="store_true",
                    help="for profiling: one layout+dispatch+combine step at each SM budget "
                         "(16, 24, 48, all), after one warm-up step")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    if dist_on:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    wl = W.BY_NAME[args.workload]
    if args.tokens > 0:
        import dataclasses
        wl = dataclasses.replace(wl, T=args.tokens)

    if args.impl == "reference":
        run_reference(args, wl, rank)
        if dist_on:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from combine_movement_gb300 import ep
    if args.dispatch_tail >= 0 and ep.ep_set_dispatch_tail(args.dispatch_tail) < 0:
        raise SystemExit("--dispatch-tail must be in [0, 90]")
    if args.combine_tail >= 0 and ep.ep_set_combine_tail(args.combine_tail) < 0:
        raise SystemExit("--combine-tail must be in [0, 90]")

    if args.overlap:
        if rank == 0:
            run_overlap(ep, dev, wl)
        return

    if args.pipeline_model:
        if rank == 0:
            run_pipeline_model(ep, dev, wl)
        return

    if args.ceilings:
        if rank == 0:
            print(json.dumps(measure_ceilings(dev)), flush=True)
        return

    if args.ncu_budgets:
        step = Step(ep, W.make_inputs(wl), dev)
        for b in (0, 16, 24, 48, 0):
            ep.ep_set_num_sms(b)
            step.run(step.b)
            torch.cuda.synchronize(dev)
        ep.ep_set_num_sms(0)
        print(json.dumps({"ncu_budgets": [16, 24, 48, "all"], "status": ep.ep_get_status(step.b.status)}))
        return

    if args.decode:
        if rank == 0:
            budgets = (16, args.budget_sms, 0) if args.budget_sms != 16 else (16, 0)
            ceil = per_sm_ceilings(dev, budgets)
            print(json.dumps(decode_latency(ep, dev, budgets, ceil)), flush=True)
        return

    if args.workloads:
        if rank == 0:
            run_workloads(ep, dev, args.budget_sms, args.steps, args.warmup)
        return

    if args.sweep:
        if rank == 0:
            run_sweep(ep, dev, budgets=(8, 16, 24, 48, 0))
        if dist_on:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    inp = W.make_inputs(wl)
    step = Step(ep, inp, dev)
    stream = torch.cuda.Stream(dev)
    sms_all = torch.cuda.get_device_properties(dev).multi_processor_count

    ep.ep_set_num_sms(0)
    if args.only_main:
        main_run = time_steps(step, args.steps, args.warmup, dist_on, stream)
        ms = max_over_ranks(main_run["total_ms"] / args.steps, dist_on)
        if rank == 0:
            print(json.dumps({"only_main": True, "ms_per_step": ms,
                              "tokens_per_s": world * step.T / (ms * 1e-3)}), flush=True)
        return
    # the headline: layout + dispatch through ep_layout_dispatch, then combine
    fused_run = time_fused_steps(step, args.steps, args.warmup, dist_on, stream,
                                 sampler_index=local)
    # the same step as three calls, with its per-kernel breakdown
    main_run = time_steps(step, args.steps, args.warmup, dist_on, stream)
    ep.ep_set_num_sms(args.budget_sms)
    budget_run = time_steps(step, args.steps, args.warmup, dist_on, stream)
    # the same budget as an SM partition (ep_sm_partition): its kernels stay
    # on those SMs and their launches may overlap
    part_run, part_sms = None, 0
    if 0 < args.budget_sms < sms_all:
        try:
            h, _, part_sms, _ = ep.ep_sm_partition(args.budget_sms)
            part_run = time_steps(step, args.steps, args.warmup, dist_on,
                                  torch.cuda.ExternalStream(h, device=dev))
        except Exception as e:  # noqa: BLE001 - reported in the line
            log(f"SM partition unavailable: {e}")
    ep.ep_set_num_sms(args.budget_sms)
    fused_budget = time_fused_steps(step, args.steps, args.warmup, dist_on, stream)
    ep.ep_set_num_sms(0)
    # dispatch and combine back to back without their tail launches (one
    # persistent launch each), beside the same figures with them (main_run)
    n_b2b = max(50, min(args.steps, 500))
    tail_pct = ep.ep_get_dispatch_tail()
    ep.ep_set_dispatch_tail(0)
    no_tail_b2b_us = calls_b2b_us(lambda s: step.dispatch(step.b, s), stream, n_b2b)
    ep.ep_set_dispatch_tail(tail_pct)
    ctail_pct = ep.ep_get_combine_tail()
    ep.ep_set_combine_tail(0)
    no_ctail_b2b_us = calls_b2b_us(lambda s: step.combine(step.b, s), stream, n_b2b)
    ep.ep_set_combine_tail(ctail_pct)
    e2e = time_e2e(step, inp, max(3, min(args.steps, 200)), 3)
    ceil = per_sm_ceilings(dev, (16, args.budget_sms, 0)) if rank == 0 else {}
    decode = decode_latency(ep, dev, (16, args.budget_sms, 0), ceil) if rank == 0 else None
    st = ep.ep_get_status(step.b.status)
    if st != 0:
        raise SystemExit(f"device status {st}: {ep.ep_status_string(st)}")

    ab = algorithmic_bytes(step.T, step.H, step.K, step.E, step.R)
    peak, peak_src = peak_hbm()

    def summarize(run: dict, nsms: int) -> dict:
        ms = max_over_ranks(run["total_ms"] / args.steps, dist_on)
        d = statistics.mean(run["dispatch_ms"])
        c = statistics.mean(run["combine_ms"])
        lay = statistics.mean(run["layout_ms"])
        moved = ab["dispatch"] + ab["combine"]
        return {
            "num_sms": nsms, "ms_per_step": ms,
            "ms_per_step_kernel_events": run["total_ms_kernel_events"] / args.steps,
            "tokens_per_s": world * step.T / (ms * 1e-3),
            "dispatch_combine_gbs": moved / ((d + c) * 1e-3) / 1e9,
            "dispatch_combine_frac": moved / ((d + c) * 1e-3) / 1e9 / peak,
            "dispatch_combine_frac_of_nominal": moved / ((d + c) * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
            # the whole step (layout included, kernels overlapping) as bandwidth
            "step_gbs": (moved + ab["layout"]) / (ms * 1e-3) / 1e9,
            "step_frac": (moved + ab["layout"]) / (ms * 1e-3) / 1e9 / peak,
            "step_frac_of_nominal": (moved + ab["layout"]) / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
            "dispatch_us": 1e3 * d, "combine_us": 1e3 * c, "layout_us": 1e3 * lay,
            # what the layout adds to the step: the step minus dispatch +
            # combine alone (both K steps, no events between the kernels)
            "layout_in_step_us": 1e3 * (run["total_ms"] - run["dispatch_combine_total_ms"])
                                 / args.steps,
            "dispatch_gbs": ab["dispatch"] / (d * 1e-3) / 1e9,
            "combine_gbs": ab["combine"] / (c * 1e-3) / 1e9,
            # each copy kernel's average launch duration over K launches back
            # to back, and its bandwidth from that
            "b2b_us": {k: 1e3 * v for k, v in run["b2b_ms"].items()},
            "dispatch_gbs_b2b": ab["dispatch"] / (run["b2b_ms"]["dispatch"] * 1e-3) / 1e9,
            "combine_gbs_b2b": ab["combine"] / (run["b2b_ms"]["combine"] * 1e-3) / 1e9,
            "us_median_p10_p90": {k: spread(run[f"{k}_ms"])
                                  for k in ("layout", "dispatch", "combine")},
        }

    def summarize_fused(run: dict, nsms: int) -> dict:
        ms = max_over_ranks(run["total_ms"] / args.steps, dist_on)
        ld = statistics.mean(run["layout_dispatch_ms"])
        c = statistics.mean(run["combine_ms"])
        return {"num_sms": nsms, "ms_per_step": ms,
                "tokens_per_s": world * step.T / (ms * 1e-3),
                "layout_dispatch_us": 1e3 * ld, "combine_us": 1e3 * c,
                "layout_dispatch_gbs": (ab["dispatch"] + ab["layout"]) / (ld * 1e-3) / 1e9}

    s_all = summarize(main_run, sms_all)
    s_bud = summarize(budget_run, min(args.budget_sms, sms_all))
    dom = "dispatch" if s_all["dispatch_us"] >= s_all["combine_us"] else "combine"
    achieved = s_all[f"{dom}_gbs_b2b"]
    traffic = kernel_traffic(dom)
    e2e_ms = max_over_ranks(e2e["ms_per_step"], dist_on)

    # every summary takes a max over ranks: computed on all ranks, in order
    head = summarize_fused(fused_run, sms_all)
    fused_bud = summarize_fused(fused_budget, min(args.budget_sms, sms_all))
    part_sum = summarize(part_run, part_sms) if part_run else None
    if rank == 0:
        cpu = None if args.no_cpu_baseline else cpu_baseline(inp)
        line = {
            "metric": METRIC,
            "value": head["tokens_per_s"],
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": head["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {
                "workload": wl_desc(wl),
                "step": "ep_layout_dispatch (layout + dispatch) then ep_combine; the same "
                        "step as three calls (ep_get_dispatch_layout, ep_dispatch, "
                        "ep_combine) is hbm.all_sms",
                "num_sms": sms_all,
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                "accumulate": "fp32 (combine)",
                "l2": "no flush: inputs larger than L2 (recv/expert_out 470 MB each; x, "
                      "58.7 MB, rotated over four device copies, 235 MB, so no step reads "
                      "the previous step's x from L2)",
            },
            "hbm": {
                "all_sms": s_all,
                f"sms_{args.budget_sms}": s_bud,
                "fused_all_sms": head,
                f"fused_sms_{args.budget_sms}": fused_bud,
                f"partition_sms_{args.budget_sms}": part_sum,
                "peak_gbs": peak,
                "peak_source": peak_src,
                "nominal_peak_gbs": NOMINAL_HBM_GBS,
                "algorithmic_bytes_per_step": ab,
            },
            # dispatch's and combine's split into a persistent launch and a
            # tail launch (ep_dispatch_launches, ep_combine_launches): their
            # calls back to back with and without
            "dispatch_tail": {
                "percent": tail_pct,
                "launches_per_call": step.dispatch_launches,
                "b2b_us": s_all["b2b_us"]["dispatch"],
                "b2b_us_one_launch": no_tail_b2b_us,
            },
            "combine_tail": {
                "percent": ctail_pct,
                "launches_per_call": step.combine_launches,
                "b2b_us": s_all["b2b_us"]["combine"],
                "b2b_us_one_launch": no_ctail_b2b_us,
            },
            "roofline": {
                "bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                "algorithmic_bytes": ab[dom],
                "launch_us": s_all["b2b_us"][dom],
                "timing": f"{args.steps} {dom} launches back to back between two CUDA events "
                          "on the launching stream (the in-step figure with events around "
                          "each kernel is hbm.all_sms." + dom + "_us)",
                "in_step_frac": s_all[f"{dom}_gbs"] / peak,
            },
            # the same figures for both HBM-bound kernels (all SMs and the
            # second budget); the layout is latency-bound and has none
            "roofline_by_kernel": {
                f"{k}_{tag}": {"achieved": r[f"{k}_gbs"], "frac": r[f"{k}_gbs"] / peak,
                               "us": r[f"{k}_us"], "algorithmic_bytes": ab[k],
                               "traffic": kernel_traffic(k) if tag == "all_sms" else None}
                for k in ("dispatch", "combine")
                for tag, r in (("all_sms", s_all), (f"sms_{args.budget_sms}", s_bud))
            },
            # the budgeted kernels against what that many SMs can move at all:
            # receive-row bytes dispatch writes (combine reads) per second over
            # the write-only (read-only) rate of plain streaming kernels on the
            # same number of SMs, measured in this run
            "budget_ceiling_frac": budget_ceiling_frac(
                ceil.get(min(args.budget_sms, sms_all)), s_bud, step),
            "e2e": {
                "value": world * step.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                # host-link bytes moved per second over both directions: the
                # e2e step is bound by the CPU-GPU link (~300 GB/s with both
                # directions busy on GB300, copy engines or SMs alike)
                "host_link_gbs": (e2e["h2d_bytes_per_step"] + e2e["d2h_bytes_per_step"])
                                 / (e2e_ms * 1e-3) / 1e9,
            },
            "gpu_launches": step.launches_per_step * args.steps,
            "clocks": fused_run["clocks"],
            "cpu_baseline": cpu,
            "decode_latency": decode,
        }
        print(json.dumps(line), flush=True)
    if dist_on:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
