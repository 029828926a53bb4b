"""Benchmark of the packed (varlen) KDA forward hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic packed
input (the Ling3-tiny packed workload by default: B=4, T=8192, H=16,
D=128, bf16, lognormal documents, max_segs=128):
    kda_segids_to_cu_seqlens  -> cu_seqlens [max_segs+1]
    kda_short_conv_varlen x3  -> masked causal conv of the q, k, v projections
    kda_chunk_fwd_varlen      -> o [B*T, H, D]
Prints one JSON line. `value` is packed tokens (B*T, padding included) per
second over the whole job with inputs resident in HBM; `e2e` is the same
metric through the public API with host buffers (pinned host->device copies
of the step's inputs and a device->host read of its outputs inside the timed
region). `roofline` is for the dominant kernel, kda_chunk_fwd_varlen.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun every rank runs its own replica of the workload (rows are
independent, no collective on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "packed tokens/sec for KDA varlen fwd (1×GB300) and % of roofline"
UNIT = "tokens/s"


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def maybe_init_dist(ws: int, backend: str):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(ws: int):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, ms_local: float, ws: int, device):
    """Whole-job throughput of a weak-scaling run: every rank processes
    `units_per_rank` units; the job takes as long as its slowest rank.
    Returns (units per second over all ranks, slowest rank's ms)."""
    ms = max_over_ranks(ms_local, ws, device)
    return units_per_rank * ws / (ms / 1e3), ms


def chunk_bytes_per_token_head(wl: synth.Workload) -> int:
    """Algorithmic HBM bytes of kda_chunk_fwd_varlen per (token, head): q, k, g
    (d_qk each), v and o (d_v each) and beta, in the workload dtype."""
    s = torch.tensor([], dtype=wl.dtype).element_size()
    return (3 * wl.d_qk + 2 * wl.d_v) * s + s


def chunk_flops_per_token_head(wl: synth.Workload) -> int:
    """The four dense chunk products per token and head at chunk C=64:
    2*C*(d_qk + d_v) + 4*d_qk*d_v."""
    C = 64
    return 2 * C * (wl.d_qk + wl.d_v) + 4 * wl.d_qk * wl.d_v


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one chunk-kernel
# launch on the ling3 workload, from an ncu capture of
# `python bench.py --steps 1 --warmup 3 --no-e2e --no-cpu-baseline`. It holds only
# for the kernel sources it was taken on (SHA-1 over the three files below);
# after any change to them the bench reports null until a new capture.
UNROLL = 8                         # steps per captured graph
CHUNK_TRAFFIC = {"workload": "ling3", "sha1": "91e4696fca62c04c69a92ba55af196cb5b3482d7",
                 "read": 561_189_888, "write": 117_422_336}
CHUNK_SOURCES = ("kda_segids_cu_gb300/csrc/kda_chunk_tc.cu", "kda_segids_cu_gb300/csrc/kda_sm100.cuh",
                 "kda_segids_cu_gb300/csrc/kda_plan.cuh")


def workload_label(wl: synth.Workload) -> str:
    """The workload as both arms name it in `config`."""
    dt = "bf16" if wl.dtype == torch.bfloat16 else "fp32"
    return (f"{wl.name} packed: B={wl.B} T={wl.T} H={wl.H} D={wl.d_qk} {dt}, "
            f"max_segs={wl.max_segs}, conv width {wl.k_conv}")


def chunk_traffic(wl: synth.Workload):
    import hashlib
    if wl.name != CHUNK_TRAFFIC["workload"] or wl != synth.WORKLOADS[wl.name]:
        return None
    h = hashlib.sha1()
    for p in CHUNK_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != CHUNK_TRAFFIC["sha1"]:
        return None
    return CHUNK_TRAFFIC["read"] + CHUNK_TRAFFIC["write"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """SM clock and clock-event reasons sampled DURING the timed region.

    NVML is read through ctypes every 2 ms from a thread (the library ships with
    the driver); `mark_start`/`mark_stop` bracket the timed region on the host
    after a device synchronize, and only samples inside the bracket count. If
    NVML cannot be opened, `nvidia-smi -lms 200` is used instead (its samples
    cover the whole sampling window)."""

    # nvmlClocksEventReasons bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.cuda_index = cuda_index
        self.period = period_s
        self.samples = []          # (host time, sm MHz, reasons bitmask)
        self.t_start = self.t_stop = None
        self.thread = None
        self.stop_flag = None
        self.nvml = None
        self.dev = None
        self.max_mhz = None
        self.proc = None
        self.path = None

    def _open_nvml(self) -> bool:
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        dev = ctypes.c_void_p()
        ok = False
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.cuda_index).uuid)
            ok = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev)) == 0
        except Exception:
            ok = False
        if not ok and "CUDA_VISIBLE_DEVICES" not in os.environ:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_index), ctypes.byref(dev)) == 0
        if not ok:
            return False
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) != 0:   # NVML_CLOCK_SM = 1
            return False
        self.nvml, self.dev, self.max_mhz = lib, dev, float(mx.value)
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return True

    def _loop(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            a = self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk))
            b = self.reasons_fn(self.dev, ctypes.byref(rs))
            if a == 0 and b == 0:
                self.samples.append((time.perf_counter(), float(clk.value), int(rs.value)))
            time.sleep(self.period)

    def start(self):
        import threading
        if self._open_nvml():
            self.stop_flag = threading.Event()
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.cuda_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(1.0)        # let the first rows arrive
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_stop(self):
        self.t_stop = time.perf_counter()

    def stop(self) -> dict | None:
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=2)
            inside = [s for s in self.samples if self.t_start <= s[0] <= self.t_stop]
            if not inside:
                return None
            reasons = sorted({n for s in inside for bit, n in self.REASONS.items() if s[2] & bit})
            return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(inside), "source": "nvml, 2 ms"}
        return self._stop_smi()

    def _stop_smi(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[2]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "source": "nvidia-smi, 200 ms"}


def bench_workload(args) -> synth.Workload:
    """The workload; --heads keeps its shape and segments with fewer heads, for kernel
    profiles that must hold little device memory (its line is not the workload's number);
    --max-segs changes only the length of cu_seqlens (the no-inflation check)."""
    wl = synth.WORKLOADS[args.workload]
    if args.heads:
        wl = dataclasses.replace(wl, H=args.heads)
    if args.max_segs:
        wl = dataclasses.replace(wl, max_segs=args.max_segs)
    return wl


def make_step_inputs(wl: synth.Workload, device):
    """The forward's inputs and the three convs' (x and weights seeded apart), all masked by
    the forward's segment ids, as in one attention layer."""
    kin = synth.make_kda_inputs(wl, device=device)
    convs = [dataclasses.replace(
        synth.make_conv_inputs(wl, seed=synth.default_seed(wl.name) + 101 + i, device=device),
        segment_ids=kin.segment_ids) for i in range(3)]
    return kin, convs


def run_gb300(args):
    import kda_segids_cu_gb300 as kda

    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    maybe_init_dist(ws, "nccl")
    wl = bench_workload(args)
    N, H = wl.N, wl.H
    kin, convs = make_step_inputs(wl, dev)
    seg = kin.segment_ids
    stream = torch.cuda.current_stream()

    # outputs and workspace allocated once (the library allocates nothing)
    cu = torch.empty(wl.max_segs + 1, dtype=torch.int32, device=dev)
    nseg = torch.empty(1, dtype=torch.int32, device=dev)
    ys = [torch.empty_like(c.x) for c in convs]
    # the convs produce q, k and v for the chunked forward ([B, T, H*D] read as [B*T, H, D]),
    # as in the attention layer of [RFC-0025]; g and beta are inputs of their own
    qkv = [y.view(N, H, wl.d_qk) for y in ys]
    o = torch.empty_like(kin.v)
    wsb = kda.chunk_fwd_workspace_bytes(wl.B, wl.T, H, wl.d_qk, wl.d_v, wl.dtype)
    work = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ev_chunk, ev_seg, ev_conv = [], [], []

    def mark(record):
        if not record:
            return None
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e

    def step(record=False):
        a = mark(record)
        if seg is not None:          # without ids every row is one segment: no scan
            kda.kda_segids_to_cu_seqlens(seg, wl.max_segs, out=cu, n_segs_out=nseg)
        b = mark(record)
        for c, y in zip(convs, ys):
            kda.kda_short_conv_varlen(c.x, c.w, c.segment_ids, out=y)
        e0 = mark(record)
        kda.kda_chunk_fwd_varlen(qkv[0], qkv[1], qkv[2], kin.g, kin.beta, seg, B=wl.B, T=wl.T,
                                 out=o, workspace=work, status=status)
        e1 = mark(record)
        if record:
            ev_seg.append((a, b))
            ev_conv.append((b, e0))
            ev_chunk.append((e0, e1))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # per-op times: an eager pass of K steps with CUDA events between the calls
    for _ in range(args.steps):
        step(record=True)
    torch.cuda.synchronize()
    chunk_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_chunk)
    seg_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_seg) if seg is not None else None
    conv_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_conv) / len(convs)
    # the timed steps: one step captured in a CUDA graph (the same calls, on the same
    # buffers) and replayed K times. The calls that read only the segment ids (the
    # cu_seqlens scan and the chunk plan) run on a side stream of the graph, concurrent with
    # the convs; the forward joins it and takes the plan from the workspace.
    side = torch.cuda.Stream(device=dev)

    def graph_step(pair=None):
        cur = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(cur)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            if seg is not None:
                kda.kda_segids_to_cu_seqlens(seg, wl.max_segs, out=cu, n_segs_out=nseg)
            kda.kda_chunk_plan_varlen(seg, wl.B, wl.T, H, wl.d_qk, wl.d_v, wl.dtype, work)
        join = torch.cuda.Event()
        join.record(side)
        for c, y in zip(convs, ys):
            kda.kda_short_conv_varlen(c.x, c.w, c.segment_ids, out=y)
        cur.wait_event(join)
        if pair is not None:       # the forward may start: its inputs and plan are ready
            ready = torch.cuda.Event()
            ready.record(cur)
            tstream.wait_event(ready)
            pair[0].record(tstream)
        kda.kda_chunk_fwd_varlen(qkv[0], qkv[1], qkv[2], kin.g, kin.beta, seg, B=wl.B, T=wl.T,
                                 out=o, workspace=work, status=status, planned=True)
        if pair is not None:       # the forward is done
            done = torch.cuda.Event()
            done.record(cur)
            tstream.wait_event(done)
            pair[1].record(tstream)

    # The chunk kernel's duration inside the timed region: timing events recorded as nodes
    # of the graph, on a stream of their own that waits for the point where the forward may
    # start and for its end. No kernel depends on them (a record node in front of the
    # forward would cut its programmatic launch after the last conv, about 6 us a step).
    # One graph holds UNROLL steps (the same calls in sequence) and is replayed
    # K // UNROLL times, then a one-step graph K % UNROLL times: after the timed loop the
    # events hold the last timed launches. (Replaying one graph keeps the launch path warm;
    # alternating between many graphs cost ~5 us per step.)
    tstream = torch.cuda.Stream(device=dev)
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        timed_events = True
    except TypeError:              # a torch without graph-node events: eager timing instead
        timed_events = False

    def capture(n_steps):
        gr = torch.cuda.CUDAGraph()
        prs = [tuple(torch.cuda.Event(enable_timing=True, external=True) for _ in range(2))
               if timed_events else None for _ in range(n_steps)]
        with torch.cuda.graph(gr):
            tstream.wait_stream(torch.cuda.current_stream())
            for pr in prs:
                graph_step(pr)
            torch.cuda.current_stream().wait_stream(tstream)
        return gr, prs

    unroll = min(UNROLL, args.steps)
    g_many, pairs_many = capture(unroll)
    rem = args.steps % unroll
    g_one, pairs_one = capture(1) if rem else (None, [])
    for _ in range(max(1, -(-args.warmup // unroll))):
        g_many.replay()
    if g_one is not None:
        g_one.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    clocks.mark_start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps // unroll):
        g_many.replay()
    for _ in range(rem):
        g_one.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_stop()
    pairs = (pairs_many + pairs_one) if timed_events else []
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in pairs) if pairs else None
    barrier(ws)
    clk = clocks.stop()
    ms_local = t0.elapsed_time(t1) / args.steps
    value, ms = job_throughput(N, ms_local, ws, dev)
    real_tokens = int((seg != 0).sum().item()) if seg is not None else N
    if int(status.item()) != 0:       # outputs of the timed calls are unreliable: no number
        raise RuntimeError(f"device status {int(status.item()):#x} after the timed steps")

    # ---- the step with the convs fused into the chunk kernel (kda_chunk_fwd_varlen_conv),
    # timed apart: the same graph shape (scan and plan on the side stream), K replays ----
    fused = None
    if wl.dtype == torch.bfloat16 and wl.d_qk == 128 and wl.k_conv <= 4:
        o_f = torch.empty_like(o)

        def fused_step():
            cur = torch.cuda.current_stream()
            fork = torch.cuda.Event()
            fork.record(cur)
            side.wait_event(fork)
            with torch.cuda.stream(side):
                if seg is not None:
                    kda.kda_segids_to_cu_seqlens(seg, wl.max_segs, out=cu, n_segs_out=nseg)
                kda.kda_chunk_plan_varlen(seg, wl.B, wl.T, H, wl.d_qk, wl.d_v, wl.dtype, work)
            join = torch.cuda.Event()
            join.record(side)
            cur.wait_event(join)
            kda.kda_chunk_fwd_varlen_conv(*(c.x for c in convs), *(c.w for c in convs), kin.g,
                                          kin.beta, seg, B=wl.B, T=wl.T, out=o_f,
                                          workspace=work, status=status, planned=True)

        g_f = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_f):
            fused_step()
        for _ in range(max(3, args.warmup)):
            g_f.replay()
        torch.cuda.synchronize()
        fa = torch.cuda.Event(enable_timing=True)
        fb = torch.cuda.Event(enable_timing=True)
        fa.record(stream)
        for _ in range(args.steps):
            g_f.replay()
        fb.record(stream)
        torch.cuda.synchronize()
        fused_ms = fa.elapsed_time(fb) / args.steps
        # the unfused forward on the last step's conv outputs, for the comparison
        o_u = kda.kda_chunk_fwd_varlen(qkv[0], qkv[1], qkv[2], kin.g, kin.beta, seg, B=wl.B,
                                       T=wl.T, workspace=work, status=status, planned=True)
        torch.cuda.synchronize()
        fused = {"ms_per_step": fused_ms, "value": N / (fused_ms / 1e3),
                 "vs_unfused_step": ms_local / fused_ms,
                 "equal_to_unfused": bool(torch.equal(o_f, o_u)),
                 "step": "segids->cu_seqlens and the chunk plan (side stream) + "
                         "kda_chunk_fwd_varlen_conv (the 3 masked convs inside the chunk kernel)"}
        del o_f, o_u

    # ---- per-segment state in and out (kda_chunk_fwd_varlen_state), timed apart ----
    n_state = int(nseg.item()) if seg is not None else wl.B
    st_gen = torch.Generator(device=dev).manual_seed(11)
    init = torch.randn(n_state, H, wl.d_qk, wl.d_v, device=dev, generator=st_gen) * 0.1
    state_ms = None
    if n_state > 0:
        def state_call():
            kda.kda_chunk_fwd_varlen_state(kin.q, kin.k, kin.v, kin.g, kin.beta, seg, B=wl.B,
                                           T=wl.T, initial_state=init, output_final_state=True,
                                           out=o, workspace=work, status=status)

        for _ in range(2):
            state_call()
        torch.cuda.synchronize()
        sa = torch.cuda.Event(enable_timing=True)
        sb = torch.cuda.Event(enable_timing=True)
        n_rep = 5
        sa.record(stream)
        for _ in range(n_rep):
            state_call()
        sb.record(stream)
        torch.cuda.synchronize()
        state_ms = sa.elapsed_time(sb) / n_rep

    # ---- gradients (kda_chunk_bwd_varlen) for a random upstream gradient, timed apart ----
    do_gen = torch.Generator(device=dev).manual_seed(13)
    d_o = torch.randn(kin.v.shape, device=dev, generator=do_gen).to(kin.v.dtype)
    bwd_ws = torch.empty(max(256, int(kda.load_library().kda_chunk_bwd_varlen_workspace_size(
        wl.B, wl.T, H, wl.d_qk, wl.d_v, 1 if kin.q.dtype == torch.bfloat16 else 0))),
        dtype=torch.uint8, device=dev)
    bwd_out = None

    bwd_status = torch.zeros(1, dtype=torch.int32, device=dev)

    def bwd_call(method="auto"):
        # the status word is read once, after the timing (not after every call)
        return kda.kda_chunk_bwd_varlen(kin.q, kin.k, kin.v, kin.g, kin.beta, d_o, seg, B=wl.B,
                                        T=wl.T, workspace=bwd_ws, method=method,
                                        status=bwd_status)

    bwd_out = bwd_call()
    torch.cuda.synchronize()
    ba = torch.cuda.Event(enable_timing=True)
    bb = torch.cuda.Event(enable_timing=True)
    n_bwd = 3
    ba.record(stream)
    for _ in range(n_bwd):
        bwd_out = bwd_call()
    bb.record(stream)
    torch.cuda.synchronize()
    bwd_ms = ba.elapsed_time(bb) / n_bwd
    # the fp32 walks (method "walk"), once, for comparison
    bwd_walk_ms = None
    if kin.q.dtype == torch.bfloat16:
        bwd_out = bwd_call("walk")
        ba.record(stream)
        bwd_out = bwd_call("walk")
        bb.record(stream)
        torch.cuda.synchronize()
        bwd_walk_ms = ba.elapsed_time(bb)
    if int(bwd_status.item()) != 0:
        raise RuntimeError(f"kda_chunk_bwd_varlen: device status {int(bwd_status.item()):#x}")
    del bwd_out, bwd_ws

    # ---- e2e through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        # the step's inputs come from pinned host memory; its result, o, goes back. The conv
        # outputs (q, k, v) stay on the device, as intermediates of the step.
        host_in = {"seg": seg.cpu().pin_memory()} if seg is not None else {}
        for n in ("g", "beta"):
            host_in[n] = getattr(kin, n).cpu().pin_memory()
        for i, c in enumerate(convs):
            host_in[f"x{i}"] = c.x.cpu().pin_memory()
            host_in[f"w{i}"] = c.w.cpu().pin_memory()
        host_out = {"o": torch.empty(o.shape, dtype=o.dtype).pin_memory()}
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in host_out.values())
        # Steps are pipelined: two copy streams bring step i's inputs in while the
        # compute stream runs step i-1 and a third stream copies step i-1's outputs
        # out; device inputs and outputs are double-buffered, ordered by events.
        nb = 2
        dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host_in.items()} for _ in range(nb)]
        dev_out = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in host_out.items()}
                   for _ in range(nb)]
        dev_mid = [[torch.empty_like(y) for y in ys] for _ in range(nb)]
        s_in = [torch.cuda.Stream(device=dev) for _ in range(2)]
        s_out = torch.cuda.Stream(device=dev)
        keys = sorted(host_in, key=lambda k: -host_in[k].numel() * host_in[k].element_size())
        ev_comp = [None] * nb       # kernels of the step that last used buffer b are done
        ev_out = [None] * nb        # outputs of the step that last used buffer b are copied out

        def e2e_step(i):
            b = i % nb
            for si in s_in:
                if ev_comp[b] is not None:
                    si.wait_event(ev_comp[b])
            for j, k in enumerate(keys):
                with torch.cuda.stream(s_in[j % len(s_in)]):
                    dev_in[b][k].copy_(host_in[k], non_blocking=True)
            for si in s_in:
                e = torch.cuda.Event()
                e.record(si)
                stream.wait_event(e)
            if ev_out[b] is not None:
                stream.wait_event(ev_out[b])
            d_in, d_out = dev_in[b], dev_out[b]
            sd = d_in.get("seg")
            if sd is not None:
                kda.kda_segids_to_cu_seqlens(sd, wl.max_segs, out=cu, n_segs_out=nseg)
            mid = dev_mid[b]
            for c in range(3):
                kda.kda_short_conv_varlen(d_in[f"x{c}"], d_in[f"w{c}"], sd, out=mid[c])
            kda.kda_chunk_fwd_varlen(*[y.view(N, H, wl.d_qk) for y in mid], d_in["g"],
                                     d_in["beta"], sd, B=wl.B, T=wl.T, out=d_out["o"],
                                     workspace=work, status=status)
            ev_comp[b] = torch.cuda.Event()
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                for k, v in host_out.items():
                    v.copy_(d_out[k], non_blocking=True)
            ev_out[b] = torch.cuda.Event()
            ev_out[b].record(s_out)

        for i in range(min(args.warmup, 3)):
            e2e_step(i)
        torch.cuda.synchronize()
        ev_comp, ev_out = [None] * nb, [None] * nb
        barrier(ws)
        a = torch.cuda.Event(enable_timing=True)
        b_ev = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for si in s_in + [s_out]:
            si.wait_event(a)
        for i in range(args.steps):
            e2e_step(i)
        stream.wait_event(ev_out[(args.steps - 1) % nb])
        b_ev.record(stream)
        torch.cuda.synchronize()
        e_value, e_ms = job_throughput(N, a.elapsed_time(b_ev) / args.steps, ws, dev)
        e2e = {"value": e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}

    if rank != 0:
        return None
    hbm, tf, tf_sus, peak_src = load_peaks()
    bytes_launch = chunk_bytes_per_token_head(wl) * N * H
    flops_launch = chunk_flops_per_token_head(wl) * N * H
    # the dominant kernel's duration: timed in the graph when the events could be captured,
    # else the eager call (planner + kernel)
    dom_ms = kernel_ms if kernel_ms is not None else chunk_ms
    achieved = bytes_launch / (dom_ms / 1e3) / 1e9
    tc_path = wl.dtype == torch.bfloat16 and wl.d_qk == 128
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; Ling3-tiny packed shape, lognormal EOD-separated documents)",
        "config": {"workload": workload_label(wl),
                   "step": ("segids->cu_seqlens + 3 masked short convs (producing q, k, v) + "
                            "chunked KDA fwd" if seg is not None else
                            "3 causal short convs (producing q, k, v) + chunked KDA fwd "
                            "(segment_ids=None: no scan)"),
                   "timing": ("the step's calls captured in a CUDA graph (the scan and the chunk "
                              "plan on a side stream of the graph, beside the convs; 8 steps per "
                              "graph, each with timing events around the forward), K steps "
                              "replayed between CUDA events; per-op times from an eager pass of "
                              "the plain calls with events between them"),
                   "l2": (f"inputs larger than L2 (conv inputs "
                          f"{sum(c.x.numel() * c.x.element_size() for c in convs) / 1e6:.0f} MB, "
                          f"g and beta "
                          f"{(kin.g.numel() + kin.beta.numel()) * kin.g.element_size() / 1e6:.0f}"
                          f" MB)"),
                   "parallelism": f"replicas x{ws} (rows independent)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": chunk_traffic(wl),
                     "kernel": (("tc::chunk_kernel (fast and safe instantiations)" if tc_path
                                 else "the token-recurrence kernels") +
                                " (kda_chunk_fwd_varlen_planned), timed by events in the graph, "
                                f"mean of the last {len(pairs)} timed steps"
                                if kernel_ms is not None else
                                "kda_chunk_fwd_varlen (planner + chunk kernel), eager pass"),
                     "kernel_ms": dom_ms, "chunk_ms": chunk_ms,
                     "bytes_per_launch": bytes_launch, "flops_per_launch": flops_launch,
                     "tensor_frac": flops_launch / (dom_ms / 1e3) / (tf * 1e12),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"},
        "ops": {
            name: {"us_per_call": ms_ * 1e3, "algorithmic_bytes": nbytes,
                   "gbs": nbytes / (ms_ / 1e3) / 1e9, "frac_hbm": nbytes / (ms_ / 1e3) / 1e9 / hbm}
            for name, ms_, nbytes in (
                ("kda_segids_to_cu_seqlens", seg_ms, 4 * N),
                ("kda_short_conv_varlen", conv_ms, 2 * N * wl.F * convs[0].x.element_size()),
                ("kda_chunk_fwd_varlen", chunk_ms, bytes_launch),
                ("kda_chunk_fwd_varlen_state", state_ms,
                 bytes_launch + 2 * n_state * H * wl.d_qk * wl.d_v * 4),
                # reads q, k, g, v, beta, d_o; writes dq, dk, dg, dv, dbeta (the default
                # method: the tensor-core path for bf16 with 128-wide heads)
                ("kda_chunk_bwd_varlen", bwd_ms,
                 N * H * (6 * wl.d_qk + 4 * wl.d_v + 2) * kin.q.element_size()),
                ("kda_chunk_bwd_varlen (fp32 walks)", bwd_walk_ms,
                 N * H * (6 * wl.d_qk + 4 * wl.d_v + 2) * kin.q.element_size()))
            if ms_ is not None
        },
        "real_tokens_per_s": real_tokens * ws / (ms / 1e3),
        "fused_conv_step": fused,
        # per step: the scan (with ids), 3 convs, 2 planner kernels and the forward's two
        # chunk kernels (fast, then safe, which exits at once when nothing is out of range or
        # split); the token-recurrence path launches one forward kernel
        "gpu_launches": args.steps * ((8 if tc_path else 7) if seg is not None else
                                      (7 if tc_path else 6)),
        "clocks": clk,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline(wl, seconds=args.cpu_seconds)
    else:
        line["cpu_baseline"] = None
    return line


def cpu_baseline(wl: synth.Workload, seconds: float = 15.0, seed_heads: int | None = None) -> dict:
    """The fp64 oracle as it stands, on the host cores, on a bounded sample of
    the workload, scaled to packed tokens/s of the full step."""
    import oracle

    nt = oracle.default_threads()
    seg_np, _ = synth.make_segment_ids(wl, synth.default_seed(wl.name))
    seg = torch.from_numpy(seg_np)
    # sample: h heads of the recurrence (all tokens), f features of each conv
    h = seed_heads or wl.H
    f = 512
    kin = synth.make_kda_inputs(wl, heads=h)
    ci = synth.make_conv_inputs(wl, features=f)
    # repeat the sample until `seconds` of CPU work have been timed (at least once)
    reps, t_cu, t_conv, t_kda = 0, 0.0, 0.0, 0.0
    while reps == 0 or (t_cu + t_conv + t_kda < seconds and reps < 100):
        t = time.perf_counter()
        oracle.cu_seqlens(seg_np, wl.max_segs)
        t_cu += time.perf_counter() - t
        t = time.perf_counter()
        oracle.short_conv(ci.x, ci.w, ci.segment_ids)
        t_conv += time.perf_counter() - t
        t = time.perf_counter()
        oracle.kda_fwd(kin.q, kin.k, kin.v, kin.g, kin.beta, seg, wl.B, wl.T, n_threads=nt)
        t_kda += time.perf_counter() - t
        reps += 1
    measured = t_cu + t_conv + t_kda
    t_cu, t_conv, t_kda = t_cu / reps, t_conv / reps, t_kda / reps
    full = t_cu + 3 * t_conv * (wl.F / f) + t_kda * (wl.H / h)
    out = {"value": wl.N / full, "unit": UNIT, "cores": nt, "kind": "oracle",
           "sample": f"{wl.name}: cu_seqlens in full; 1 conv on {f} of {wl.F} features "
                     f"(x3 convs, scaled by features); recurrence on {h} of {wl.H} heads "
                     f"(all {wl.N} tokens, {nt} threads, scaled by heads); "
                     f"{reps} repetitions, measured {measured:.1f} s",
           "seconds_full_step_estimate": full}
    if wl.name in ("tiny", "b2"):          # the two small workloads also on one thread
        t = time.perf_counter()
        oracle.kda_fwd(kin.q, kin.k, kin.v, kin.g, kin.beta, seg, wl.B, wl.T, n_threads=1)
        t1 = time.perf_counter() - t
        out["single_thread"] = {"value": wl.N / (t_cu + 3 * t_conv * (wl.F / f) + t1 * (wl.H / h)),
                                "unit": UNIT, "cores": 1,
                                "sample": "the same step, the recurrence on one thread (once)"}
    return out


def run_reference(args, budget_s: float = 150.0):
    """The reference arm: the fp64 CPU oracle, as it stands, timed on the host cores on
    the full step of the workload (cu_seqlens, the three masked convs on all features,
    the recurrence on all heads). When --steps + --warmup full steps would not finish
    within `budget_s`, each step runs a fixed subset of heads and conv features instead,
    scaled to the full step, and `sample` says so."""
    ws, rank, _ = dist_info()
    if rank != 0:
        return None
    import oracle

    wl = bench_workload(args)
    nt = oracle.default_threads()
    seg_np, _ = synth.make_segment_ids(wl, synth.default_seed(wl.name))
    seg = torch.from_numpy(seg_np)
    kin, convs = make_step_inputs(wl, "cpu")

    def step(h=wl.H, f=wl.F):
        ks = [t[:, :h].contiguous() for t in (kin.q, kin.k, kin.v, kin.g, kin.beta)] \
            if h < wl.H else [kin.q, kin.k, kin.v, kin.g, kin.beta]
        xs = [(c.x[..., :f].contiguous(), c.w[:, :f].contiguous()) for c in convs] \
            if f < wl.F else [(c.x, c.w) for c in convs]
        t = time.perf_counter()
        oracle.cu_seqlens(seg_np, wl.max_segs)
        a = time.perf_counter() - t
        t = time.perf_counter()
        for x, w in xs:
            oracle.short_conv(x, w, convs[0].segment_ids)
        b = time.perf_counter() - t
        t = time.perf_counter()
        oracle.kda_fwd(*ks, seg if wl.segmented else None, wl.B, wl.T, n_threads=nt)
        c = time.perf_counter() - t
        return a + b * (wl.F / f) + c * (wl.H / h)

    first = step()                               # the first warm-up step, full size
    h, f = wl.H, wl.F
    if (args.steps + args.warmup) * first > budget_s:
        frac = budget_s / ((args.steps + args.warmup) * first)
        h = max(1, int(wl.H * frac))
        f = max(8, int(wl.F * frac) // 8 * 8)
    for _ in range(args.warmup - 1):
        step(h, f)
    full = [step(h, f) for _ in range(args.steps)]
    s = statistics.mean(full)
    value = wl.N / s
    if h == wl.H and f == wl.F:
        sample = (f"{wl.name}: the full step, measured: cu_seqlens, 3 masked convs on all "
                  f"{wl.F} features, recurrence on all {wl.H} heads ({nt} threads)")
    else:
        sample = (f"{wl.name}: per step cu_seqlens in full, 3 convs on {f} of {wl.F} features "
                  f"and the recurrence on {h} of {wl.H} heads, scaled (a full step takes "
                  f"{first:.2f} s; {args.steps + args.warmup} of them exceed {budget_s:.0f} s)")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "impl": "reference",
            "config": {"workload": workload_label(wl),
                       "step": "fp64 CPU oracle: cu_seqlens + 3 masked convs + recurrence"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="ling3", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--heads", type=int, default=0,
                    help="profiling only: the workload with this many heads")
    ap.add_argument("--max-segs", type=int, default=0,
                    help="the cu_seqlens length (max_segs + 1) instead of the workload's; the "
                         "forward does not read cu_seqlens, so only the scan's writes change")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    line = run_reference(args) if args.impl == "reference" else run_gb300(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
