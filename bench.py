#!/usr/bin/env python3
"""Benchmark of the local MoE forward chain (route -> dispatch -> SwiGLU experts
-> combine) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the whole chain over one batch of the coarse BF16
prefill workload (T=8192, H=4096, I=14336, E=8, top_k=2, renormalize; the
GEMM-bound case and the largest one that fits one GPU), inputs resident in
HBM. One moe_forward call is captured once in a CUDA graph; each timed step is
one replay bracketed by CUDA events on the launching stream, and L2 is
flushed between steps outside the events (a 256 MiB write, then a 256 MiB
read so the flush's dirty lines are written back before the step). The
per-stage times come from a second run that launches the C-ABI stage calls
(route + dispatch as one launch, the experts' GEMMs, combine: the kernels
moe_forward runs) directly with events between the stages, and a third with
the routing and the dispatch as separate calls. Under torchrun each rank runs its own T-token shard of an
N*T-token global batch (weak scaling, replicated experts, no collective on
the data path); the time is the maximum over ranks.

Printed (rank 0, one JSON line): tokens/s, grouped-GEMM TFLOP/s against the
measured BF16 peak, route+dispatch microseconds, the roofline of the dominant
kernel (the experts' GEMMs), the end-to-end number through moe_forward_host
with host buffers (two streams pipelined, and one batch at a time), the CPU
oracle baseline, kernel launches and the SM clocks seen during the run; then,
as extra keys, the fine-grained BF16 prefill (T=4096, E=128, top_k=8) step
with its GEMM roofline, the decode workload's HBM GB/s over the touched
expert weights, the Zipf-skewed F16 prefill's GEMMs, the grouped sigmoid
routing on the fine-grained prefill, and one first-order training step on the
fine-grained and on the coarse prefill.

--impl reference times the CPU oracle (the only reference this path has) on
bounded samples of the headline workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "MoE fwd tokens/s + grouped-GEMM TFLOP/s vs bf16 peak; decode HBM GB/s"
HEADLINE = workloads.CONFIGS[2]  # coarse BF16 prefill
FINE = workloads.CONFIGS[1]      # fine-grained BF16 prefill
DECODE = workloads.CONFIGS[3]
ZIPF = workloads.CONFIGS[4]
FLUSH_BYTES = 256 << 20
KERNELS_PER_STEP = 3  # route + dispatch (one launch), gate/up + down GEMMs (one launch), combine
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (timing only; no data-path collective)."""
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(cfg, n_gpus):
    return {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "top_k": cfg.top_k,
            "renormalize": cfg.renormalize, "tokens_per_gpu": cfg.T,
            "global_batch_tokens": cfg.T * n_gpus,
            "parallelism": f"dp{n_gpus}: each rank runs its own {cfg.T}-token shard of a {cfg.T * n_gpus}-token "
                           "global batch (rank-seeded tokens), experts replicated, no collective on the data path",
            "l2": "flushed between timed steps (256 MiB write, then a 256 MiB read so the written lines "
                  "are written back before the step)"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.path = Path(os.environ.get("TMPDIR", "/tmp")) / f"moe_bench_clocks_{os.getpid()}.csv"
        try:
            props = torch.cuda.get_device_properties(device_index)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
            sel = ["-i", bus]
        except Exception:
            sel = []
        cmd = ["nvidia-smi", *sel, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
               "-lms", "50"]
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in self.path.read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                rows.append(parts)
        self.path.unlink(missing_ok=True)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        loaded = [s for s, p in zip(sm, pw) if p is not None and p > 200.0] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------- our arm

class Chain:
    """Pre-allocated buffers and the raw C-ABI calls of one forward step."""

    def __init__(self, moe, cfg, dev, shard=0):
        self.moe, self.lib, self.cfg, self.dev = moe, moe.load_library(), cfg, dev
        inp = workloads.generate(cfg, shard=shard)
        self.host = inp
        d = {k: v.to(dev) for k, v in inp.items()}
        self.d = d
        self.ex = moe.Experts(d["gate"], d["up"], d["down"])
        T, k, E, H, I = cfg.T, cfg.top_k, cfg.E, cfg.H, cfg.I
        n = T * k
        e = dict(device=dev)
        self.idx = torch.empty(T, k, dtype=torch.int32, **e)
        self.w = torch.empty(T, k, dtype=cfg.torch_dtype, **e)
        self.counts = torch.empty(E, dtype=torch.int32, **e)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, **e)
        self.row_src = torch.empty(n, dtype=torch.int32, **e)
        self.inv = torch.empty(n, dtype=torch.int32, **e)
        # moe_forward's choice: gather x rows in the gate/up GEMM for
        # decode-sized batches, else materialise x_dispatched.
        self.gather = n <= 8 * E
        self.xd = None if self.gather else torch.empty(n, H, dtype=cfg.torch_dtype, **e)
        self.h = torch.empty(n, I, dtype=cfg.torch_dtype, **e)
        self.yd = torch.empty(n, H, dtype=cfg.torch_dtype, **e)
        self.out = torch.empty(T, H, dtype=cfg.torch_dtype, **e)
        self.dws = torch.empty(max(1, self.lib.moe_dispatch_workspace_size(T, E, k)), dtype=torch.uint8, **e)
        self.fws = torch.empty(max(1, self.lib.moe_forward_workspace_size(self.ex.handle, T, k)),
                               dtype=torch.uint8, **e)
        self.sws = torch.empty(moe.STAGE_WORKSPACE_BYTES, dtype=torch.uint8, **e)
        self.cws = torch.empty(max(1, self.lib.moe_experts_forward_combine_workspace_size(self.ex.handle, T, k)),
                               dtype=torch.uint8, **e)
        self.uws = torch.empty(max(1, self.lib.moe_experts_forward_dispatched_workspace_size(self.ex.handle, n)),
                               dtype=torch.uint8, **e)
        self.rdws = torch.empty(max(1, self.lib.moe_route_dispatch_workspace_size(T, E)), dtype=torch.uint8, **e)
        self.fused = False  # prefill staged run: True = the experts and the combine in one launch
        self.split_route = False  # staged run: True = moe_route then moe_dispatch instead of the one launch
        self.dt = moe._dt(d["x"])
        self.grouped = None  # (bias device tensor or None, GroupRoutingOptions) to route by sigmoid groups

    def use_grouped_routing(self, routing):
        """Route by the grouped sigmoid routing from now on (routing: workloads.GroupedRouting)."""
        assert routing.top_k == self.cfg.top_k
        bias = workloads.grouped_bias(self.cfg.E, routing)
        opts = self.moe.GroupRoutingOptions(routing.top_k, routing.groups, routing.selected_groups,
                                            routing.group_top_two, routing.renormalize, routing.scale)
        self.grouped = (None if bias is None else bias.to(self.dev), opts)

    def step(self, stream, ev=None):
        """route | dispatch | experts | combine, events between: the calls
        moe_forward makes. Route and dispatch as the one launch the forward
        calls run (moe_route_dispatch, or moe_route_sigmoid_grouped_dispatch
        with grouped routing; the dispatch stage is then empty), or with
        self.split_route the routing call then moe_dispatch.
        Prefill: the chained gate/up + down launch over
        x_dispatched (moe_experts_forward_dispatched, the kernel moe_forward
        runs), then moe_combine; with self.fused, the experts and the
        combine in one launch (moe_experts_forward_combine; the combine
        stage is then empty). Decode-sized batches: x rows gathered in the
        gate/up GEMM (moe_experts_gate_up_gather), then moe_experts_down and
        moe_combine."""
        c, lib, P = self.cfg, self.lib, self.moe._ptr
        s = ctypes.c_void_p(stream.cuda_stream)
        T, k, E, H = c.T, c.top_k, c.E, c.H
        rec = (lambda i: ev[i].record(stream)) if ev is not None else (lambda i: None)
        rc = 0
        rec(0)
        fused_rd = not self.split_route
        xd = None if self.gather else self.xd
        xp = None if xd is None else P(self.d["x"])
        if fused_rd and self.grouped is None:
            rc |= lib.moe_route_dispatch(P(self.d["logits"]), self.dt, T, E, k, int(c.renormalize), P(self.idx),
                                         P(self.w), None, xp, self.dt, H, P(self.counts), P(self.offsets),
                                         P(self.row_src), P(self.inv), P(xd), P(self.rdws), self.rdws.numel(), s)
        elif fused_rd:
            bias, opts = self.grouped
            rc |= lib.moe_route_sigmoid_grouped_dispatch(P(self.d["logits"]), self.dt, T, E, P(bias),
                                                         ctypes.byref(opts), P(self.idx), P(self.w), None, xp,
                                                         self.dt, H, P(self.counts), P(self.offsets),
                                                         P(self.row_src), P(self.inv), P(xd), P(self.rdws),
                                                         self.rdws.numel(), s)
        elif self.grouped is None:
            rc |= lib.moe_route(P(self.d["logits"]), self.dt, T, E, k, int(c.renormalize), P(self.idx),
                                P(self.w), None, s)
        else:
            bias, opts = self.grouped
            rc |= lib.moe_route_sigmoid_grouped(P(self.d["logits"]), self.dt, T, E, P(bias), ctypes.byref(opts),
                                                P(self.idx), P(self.w), None, s)
        rec(1)
        if self.gather:
            if not fused_rd:
                rc |= lib.moe_dispatch(P(self.idx), T, E, k, None, self.dt, H, P(self.counts), P(self.offsets),
                                       P(self.row_src), P(self.inv), None, P(self.dws), self.dws.numel(), s)
            rec(2)
            rc |= lib.moe_experts_gate_up_gather(self.ex.handle, P(self.d["x"]), T, P(self.row_src), k,
                                                 P(self.offsets), T * k, P(self.h), P(self.sws), self.sws.numel(), s)
            rc |= lib.moe_experts_down(self.ex.handle, P(self.h), P(self.offsets), T * k, P(self.yd), P(self.sws),
                                       self.sws.numel(), s)
        else:
            if not fused_rd:
                rc |= lib.moe_dispatch(P(self.idx), T, E, k, P(self.d["x"]), self.dt, H, P(self.counts),
                                       P(self.offsets), P(self.row_src), P(self.inv), P(self.xd), P(self.dws),
                                       self.dws.numel(), s)
            rec(2)
            if self.fused:
                rc |= lib.moe_experts_forward_combine(self.ex.handle, P(self.xd), P(self.offsets), P(self.inv),
                                                      P(self.w), self.dt, T, k, P(self.out), P(self.cws),
                                                      self.cws.numel(), s)
            else:
                rc |= lib.moe_experts_forward_dispatched(self.ex.handle, P(self.xd), P(self.offsets), T * k,
                                                         P(self.yd), P(self.uws), self.uws.numel(), s)
        rec(3)
        if self.gather or not self.fused:
            rc |= lib.moe_combine(P(self.yd), self.dt, P(self.inv), P(self.w), self.dt, T, k, H, P(self.out), s)
        rec(4)
        if rc:
            raise RuntimeError("a C-ABI call failed: " + lib.moe_last_error().decode())

    def route_dispatch_maps(self, stream):
        """The one route + dispatch launch without the x copy (indices,
        weights and the dispatch maps only)."""
        c, lib, P = self.cfg, self.lib, self.moe._ptr
        rc = lib.moe_route_dispatch(P(self.d["logits"]), self.dt, c.T, c.E, c.top_k, int(c.renormalize),
                                    P(self.idx), P(self.w), None, None, self.dt, c.H, P(self.counts),
                                    P(self.offsets), P(self.row_src), P(self.inv), None, P(self.rdws),
                                    self.rdws.numel(), ctypes.c_void_p(stream.cuda_stream))
        if rc:
            raise RuntimeError("moe_route_dispatch failed: " + lib.moe_last_error().decode())

    def forward(self, stream):
        """The whole chain as one moe_forward call (what a user runs)."""
        c, lib, P = self.cfg, self.lib, self.moe._ptr
        rc = lib.moe_forward(self.ex.handle, P(self.d["x"]), P(self.d["logits"]), self.dt, c.T, c.top_k,
                             int(c.renormalize), P(self.out), P(self.idx), P(self.w), P(self.fws), self.fws.numel(),
                             ctypes.c_void_p(stream.cuda_stream))
        if rc:
            raise RuntimeError("moe_forward failed: " + lib.moe_last_error().decode())

    def touched_experts(self) -> int:
        return int((self.counts.cpu() > 0).sum())

    def free(self):
        """Drop the device buffers (the next workload's chain needs the room)."""
        for name in list(vars(self)):
            if isinstance(getattr(self, name), torch.Tensor) or name in ("d", "ex", "host"):
                setattr(self, name, None)
        torch.cuda.empty_cache()


N_STAGES = 4  # route | dispatch | experts | combine


class L2Flush:
    """Between timed steps: write a 256 MiB buffer (evicts everything the
    last step left in the 126 MB L2), then read a second one so that the
    written lines are written back to HBM before the next step starts rather
    than inside it. Runs outside the timed events."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.amax(self.r)  # a pure read (no converted copy), one small result


def timed_steps(chain, stream, flush, steps, warmup):
    """Warmup + timed steps with CUDA events between the stages; returns the
    per-stage mean seconds and the total."""
    for _ in range(warmup):
        flush()
        chain.step(stream)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(N_STAGES + 1)] for _ in range(steps)]
    for i in range(steps):
        flush()
        chain.step(stream, evs[i])
    torch.cuda.synchronize()
    stages = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(N_STAGES)]
                       for i in range(steps)]) / 1e3
    total = float(sum(evs[i][0].elapsed_time(evs[i][N_STAGES]) for i in range(steps))) / 1e3
    return stages.mean(axis=0), total


def timed_calls(fn, stream, flush, steps, warmup):
    """Mean seconds of fn(stream) between CUDA events, L2 flushed before each."""
    for _ in range(warmup):
        flush()
        fn(stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(stream)
        fn(stream)
        b.record(stream)
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in evs])) / 1e3


def capture_step(chain):
    """One moe_forward call captured into a CUDA graph (the same kernels,
    replayed without host launch overhead)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            chain.forward(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain.forward(torch.cuda.current_stream())
    torch.cuda.synchronize()
    return g


def timed_graph_steps(graph, stream, flush, steps, warmup):
    """Warmup + timed replays of the captured step, one pair of CUDA events
    around each replay; returns the total seconds over the timed steps."""
    for _ in range(warmup):
        flush()
        graph.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return float(sum(a.elapsed_time(b) for a, b in evs)) / 1e3


def e2e_steps(chain, stream, flush, steps):
    """One batch at a time: moe_forward_host with pinned host x/logits in and
    the output back to pinned host memory, then wait for it; L2 flushed
    before each batch, outside the events. Returns (seconds per batch, H2D
    bytes, D2H bytes)."""
    moe, c = chain.moe, chain.cfg
    hx, hl = chain.host["x"].pin_memory(), chain.host["logits"].pin_memory()
    hout = torch.empty(c.T, c.H, dtype=c.torch_dtype).pin_memory()
    lib = moe.load_library()
    ws = torch.empty(lib.moe_forward_host_workspace_size(chain.ex.handle, c.T, c.top_k, moe._dt(hl)),
                     dtype=torch.uint8, device=chain.dev)
    ms = []
    with torch.cuda.stream(stream):
        for i in range(steps + 2):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            moe.moe_forward_host(chain.ex, hx, hl, c.top_k, c.renormalize, out=hout, workspace=ws, stream=stream)
            b.record(stream)
            b.synchronize()
            if i >= 2:
                ms.append(a.elapsed_time(b))
    h2d = hx.numel() * hx.element_size() + hl.numel() * hl.element_size()
    d2h = hout.numel() * hout.element_size()
    return float(np.mean(ms)) / 1e3, h2d, d2h


def e2e_pipelined(chain, steps):
    """`steps` batches through moe_forward_host (pinned host inputs in, the
    output back to pinned host memory) alternating over two streams with two
    workspaces, so that one batch's copies overlap the other's kernels; the
    expert weights (1.2 GB) are larger than L2, so there is no flush between
    batches. Returns seconds per batch: from an event before the first batch
    to the later of the two streams' final events."""
    moe, c = chain.moe, chain.cfg
    lib = moe.load_library()
    hx, hl = chain.host["x"].pin_memory(), chain.host["logits"].pin_memory()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    nbytes = lib.moe_forward_host_workspace_size(chain.ex.handle, c.T, c.top_k, moe._dt(hl))
    wss = [torch.empty(nbytes, dtype=torch.uint8, device=chain.dev) for _ in range(2)]
    outs = [torch.empty(c.T, c.H, dtype=c.torch_dtype).pin_memory() for _ in range(2)]

    def run(n, start=None):
        if start is not None:
            for s in streams:
                s.wait_event(start)
        for i in range(n):
            s = streams[i % 2]
            moe.moe_forward_host(chain.ex, hx, hl, c.top_k, c.renormalize, out=outs[i % 2], workspace=wss[i % 2],
                                 stream=s)

    run(4)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    ends = [torch.cuda.Event(enable_timing=True) for _ in streams]
    start.record(torch.cuda.current_stream())
    run(steps, start)
    for e, s in zip(ends, streams):
        e.record(s)
    torch.cuda.synchronize()
    return max(start.elapsed_time(e) for e in ends) / 1e3 / steps


def traffic_record(kernel_source: Path, workload: str):
    """ncu DRAM bytes per launch of the dominant kernel on one workload, if
    they were taken on the current kernel source (else None)."""
    p = ROOT / "profiles" / "ncu_traffic.json"
    if not p.exists():
        return None
    rec = json.loads(p.read_text())
    sha = hashlib.sha256(kernel_source.read_bytes()).hexdigest()
    if rec.get("source_sha256") != sha:
        return None
    return rec.get("workloads", {}).get(workload)


def gemm_stage_times(moe, cfg, dev, stream, flush, steps):
    """Mean seconds of the gate/up and down GEMM stages on one workload, each
    launched on its own, and of the chained launch of both (the one
    moe_forward runs; moe_experts_forward_dispatched). Routing and dispatch
    done once beforehand; L2 flushed before each timed call."""
    inp = workloads.generate(cfg)
    d = {k: v.to(dev) for k, v in inp.items()}
    del inp
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, _ = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    h = moe.moe_experts_gate_up(ex, disp.x_dispatched, disp.offsets)
    y = moe.moe_experts_down(ex, h, disp.offsets)
    ws = torch.empty(moe.STAGE_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
    rows = disp.x_dispatched.shape[0]
    cws = torch.empty(moe.load_library().moe_experts_forward_dispatched_workspace_size(ex.handle, rows),
                      dtype=torch.uint8, device=dev)
    y2 = torch.empty_like(y)
    times = {"gate_up": [], "down": [], "chain": []}
    for i in range(steps + 2):
        for name in ("gate_up", "down", "chain"):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if name == "gate_up":
                moe.moe_experts_gate_up(ex, disp.x_dispatched, disp.offsets, out=h, workspace=ws)
            elif name == "down":
                moe.moe_experts_down(ex, h, disp.offsets, out=y, workspace=ws)
            else:
                moe.moe_experts_forward_dispatched(ex, disp.x_dispatched, disp.offsets, out=y2, workspace=cws)
            b.record(stream)
            b.synchronize()
            if i >= 2:
                times[name].append(a.elapsed_time(b) / 1e3)
    assert moe.moe_device_status() == 0
    assert torch.equal(y.view(torch.uint8), y2.view(torch.uint8)), "chained and split expert GEMMs differ"
    del ex, d, h, y, y2, disp, cws
    torch.cuda.empty_cache()
    return float(np.mean(times["gate_up"])), float(np.mean(times["down"])), float(np.mean(times["chain"]))


def training_step_times(moe, cfg, dev, stream, flush, steps):
    """One first-order training step on a workload (ruDNN user guide, section
    12): forward (route + dispatch in one launch, training forward of the
    experts, combine)
    then backward (combine backward, experts backward, dispatch backward,
    router backward of the softmax weights). Returns mean seconds per stage
    (forward, combine_backward, experts_backward, dispatch_backward,
    router_backward)."""
    inp = workloads.generate(cfg)
    d = {k: v.to(dev) for k, v in inp.items()}
    del inp
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    g = torch.Generator().manual_seed(7)
    grad_out = torch.randn(cfg.T, cfg.H, generator=g).to(cfg.torch_dtype).to(dev)
    opts = moe.RouterWeightOptions("softmax", cfg.renormalize, 1.0)

    def step(ev=None):
        rec = (lambda i: ev[i].record(stream)) if ev is not None else (lambda i: None)
        rec(0)
        idx, w, disp = moe.moe_route_dispatch(d["logits"], cfg.top_k, cfg.renormalize, d["x"])
        y, cache = moe.moe_experts_forward_training(ex, disp.x_dispatched, disp.offsets)
        moe.moe_combine(y, disp.inv, w)
        rec(1)
        dexp, dw = moe.moe_combine_backward(y, disp.inv, disp.row_src, w, grad_out)
        rec(2)
        gr = moe.moe_experts_backward(ex, cache, dexp)
        rec(3)
        moe.moe_dispatch_backward(gr.dx_dispatched, disp.inv, cfg.T, cfg.top_k)
        rec(4)
        moe.moe_router_backward(d["logits"], idx, dw, opts)
        rec(5)

    for _ in range(2):
        flush()
        step()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        step(ev)
        torch.cuda.synchronize()
        times.append([ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(5)])
    assert moe.moe_device_status() == 0
    del ex, d
    torch.cuda.empty_cache()
    return [float(x) for x in np.mean(np.array(times), axis=0)]


def widened_weights(inp):
    """The expert weights as f64 CPU tensors: exact copies of the dtype values
    (the oracle computes the experts in f64), made once so that a timed oracle
    call does not convert the expert weights again."""
    return {k: inp[k].to(torch.float64) for k in ("gate", "up", "down")}


def cpu_baseline(cfg, inp, target_s=15.0):
    """The oracle, as it stands, on the first n tokens of the batch, n sized
    from a 256-token probe (after a 32-token warm-up call) so that the timed
    call takes about ``target_s`` seconds of CPU work; the weights are
    widened to f64 before the timed calls."""
    from oracle import moe_oracle

    w64 = widened_weights(inp)

    def run(n):
        t0 = time.perf_counter()
        moe_oracle.forward(inp["x"][:n], inp["logits"][:n], w64["gate"], w64["up"], w64["down"],
                           cfg.top_k, cfg.renormalize)
        return time.perf_counter() - t0

    run(min(32, cfg.T))
    probe = min(256, cfg.T)
    t_probe = run(probe)
    n = int(min(cfg.T, max(probe, (target_s / max(t_probe, 1e-6)) * probe)))
    n = max(probe, (n // 32) * 32) if n < cfg.T else cfg.T
    dt = run(n)
    return {"value": n / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"the first {n} of {cfg.T} tokens of {cfg.name} (one call, sized from a {probe}-token probe "
                      f"of {t_probe:.2f} s): FP32 routing, dispatch, f64 SwiGLU experts and combine, {dt:.1f} s "
                      "(expert weights widened to f64 once, before the timed call)"}


def gemm_roofline(cfg, t_chain, touched, peaks, peaks_src, traffic, timing):
    """Roofline of the chained gate/up + down launch on one workload.
    Algorithmic work per launch (the method's, not the kernel's): flops
    6*T*k*H*I; bytes = the touched experts' gate, up and down weights, x read
    once and the output written once (T*H each)."""
    es = 2
    flops = cfg.expert_flops
    nbytes = touched * 3 * cfg.I * cfg.H * es + 2 * cfg.T * cfg.H * es
    tflops = flops / t_chain / 1e12
    gbs = nbytes / t_chain / 1e9
    bound = "hbm" if nbytes / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops"] * 1e12) else "tensor"
    dram = traffic["dram_bytes_per_launch"] if traffic else None
    # A tensor-bound launch is timed inside seconds of back-to-back steps, at
    # the GPU's power cap: its peak is the sustained BF16 figure (the burst
    # fraction is reported beside it).
    return {"kernel": "experts_tc_kernel, chained gate/up + SwiGLU and down (K3 + K4), one launch",
            "workload": cfg.name, "bound": bound,
            "achieved": round(gbs if bound == "hbm" else tflops, 2),
            "peak": peaks["hbm_gbs"] if bound == "hbm" else peaks["bf16_tflops_sustained"],
            "peak_kind": "measured HBM copy" if bound == "hbm" else "measured sustained BF16 (seconds-long loop)",
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": round(gbs / peaks["hbm_gbs"] if bound == "hbm" else tflops / peaks["bf16_tflops_sustained"], 4),
            "traffic": dram, "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
            "traffic_over_algorithmic": round(dram / nbytes, 4) if dram else None,
            "us": round(t_chain * 1e6, 2), "tflops": round(tflops, 1),
            "tensor_frac": round(tflops / peaks["bf16_tflops"], 4),  # of the burst peak
            "tensor_frac_sustained": round(tflops / peaks["bf16_tflops_sustained"], 4),
            "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": peaks_src, "timing": timing}


def forward_measure(moe, cfg, dev, stream, flush, steps, warmup, world, shard=0, stage_steps=None):
    """The whole chain on one workload: CUDA-graph replays of one moe_forward
    call (tokens/s, max over ranks), then the staged run (route | dispatch |
    experts | combine with events between), and for prefill the same staged
    run with the experts and the combine in one launch
    (moe_experts_forward_combine: an A/B of the fused combine). Returns
    (chain, result dict)."""
    chain = Chain(moe, cfg, dev, shard=shard)
    graph = capture_step(chain)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize()
    total = timed_graph_steps(graph, stream, flush, steps, warmup)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total = max_over_ranks(total, world, dev)
    del graph
    n_stage = stage_steps or min(steps, 200)
    stages, stage_total = timed_steps(chain, stream, flush, n_stage, warmup)
    stages = [float(x) for x in stages]
    chain.split_route = True
    split, _ = timed_steps(chain, stream, flush, n_stage, warmup)
    chain.split_route = False
    split = [float(x) for x in split]
    maps_only = timed_calls(chain.route_dispatch_maps, stream, flush, n_stage, warmup)
    fused = None
    if not chain.gather:
        chain.fused = True
        f_stages, f_total = timed_steps(chain, stream, flush, n_stage, warmup)
        chain.fused = False
        fused = {"fused_experts_combine_us": round(float(f_stages[2]) * 1e6, 2),
                 "experts_us": round(stages[2] * 1e6, 2), "combine_us": round(stages[3] * 1e6, 2),
                 "experts_plus_combine_us": round((stages[2] + stages[3]) * 1e6, 2),
                 "fused_staged_step_us": round(f_total / n_stage * 1e6, 2),
                 "staged_step_us": round(stage_total / n_stage * 1e6, 2)}
    return chain, {"total_s": total, "steps": steps, "stages_s": stages, "split_stages_s": split,
                   "maps_only_s": maps_only,
                   "stage_steps": n_stage,
                   "stage_total_s": stage_total, "touched": chain.touched_experts(), "fused_ab": fused}


def run_ours(args, rank, world, local_rank):
    import moe_routing_swiglu_gb300 as moe
    from moe_routing_swiglu_gb300 import _build

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if local_rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    moe.load_library()
    peaks, peaks_src = load_peaks()
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    kernel_src = ROOT / "moe_routing_swiglu_gb300" / "csrc" / "experts_tc.cu"
    clocks = ClockSampler(local_rank)

    # ---- headline: the coarse BF16 prefill, this rank's token shard
    c = HEADLINE
    chain, hr = forward_measure(moe, c, dev, stream, flush, args.steps, args.warmup, world, shard=rank)
    t_exp = hr["stages_s"][2]
    e2e_serial_s, h2d, d2h = e2e_steps(chain, stream, flush, min(args.steps, 20))
    e2e_serial_s = max_over_ranks(e2e_serial_s, world, dev)
    e2e_steps_n = min(args.steps, 100)
    if world > 1:
        dist.barrier()
    e2e_s = max_over_ranks(e2e_pipelined(chain, e2e_steps_n), world, dev)
    host_inp = chain.host if rank == 0 and world == 1 else None
    chain.free()
    del chain
    t_gu, t_dn, _ = gemm_stage_times(moe, c, dev, stream, flush, 5)
    trc = training_step_times(moe, c, dev, stream, flush, 3)

    # ---- fine-grained BF16 prefill (E=128, top_k=8): step, GEMM roofline, grouped routing, training
    f = FINE
    fchain, fr = forward_measure(moe, f, dev, stream, flush, min(args.steps, 1000), args.warmup, world)
    grouped_cfg, grouped_routing = workloads.GROUPED["bf16_prefill_grouped"]
    assert grouped_cfg is FINE
    fchain.use_grouped_routing(grouped_routing)
    g_steps = min(args.steps, 200)
    g_stages, g_total = timed_steps(fchain, stream, flush, g_steps, args.warmup)
    g_total = max_over_ranks(g_total, world, dev)
    fchain.split_route = True
    g_split, _ = timed_steps(fchain, stream, flush, g_steps, args.warmup)
    fchain.split_route = False
    fchain.free()
    del fchain
    f_gu, f_dn, _ = gemm_stage_times(moe, f, dev, stream, flush, 5)
    tr = training_step_times(moe, f, dev, stream, flush, 5)

    # ---- decode
    dchain, dr = forward_measure(moe, DECODE, dev, stream, flush, min(args.steps, 1000), args.warmup, world,
                                 stage_steps=min(args.steps, 50))
    dchain.free()
    del dchain

    # ---- Zipf-skewed F16 prefill: the expert GEMMs
    z_gu, z_dn, z_ch = gemm_stage_times(moe, ZIPF, dev, stream, flush, 5)
    clk = clocks.stop()
    assert moe.moe_device_status() == 0, "a device-side wait timed out during the benchmark"

    ms_per_step = hr["total_s"] / args.steps * 1e3
    tokens_per_s = world * c.T * args.steps / hr["total_s"]
    stage_note = ("the staged run's experts stage: the chained gate/up + down launch "
                  "(moe_experts_forward_dispatched, the kernel moe_forward runs), CUDA events on the launching "
                  "stream around it in each of {n} steps, L2 flushed before each step")
    roof = gemm_roofline(c, t_exp, hr["touched"], peaks, peaks_src, traffic_record(kernel_src, c.name),
                         stage_note.format(n=hr["stage_steps"]))
    froof = gemm_roofline(f, fr["stages_s"][2], fr["touched"], peaks, peaks_src, traffic_record(kernel_src, f.name),
                          stage_note.format(n=fr["stage_steps"]))
    def training_line(cfg, tr):
        bwd_flops = 2 * cfg.expert_flops  # dgrad + wgrad: twice the forward's 6*T*k*H*I
        tf = bwd_flops / tr[2] / 1e12
        return {"workload": cfg.name, "us_per_step": round(sum(tr) * 1e6, 1),
                "tokens_per_s": round(world * cfg.T / sum(tr), 1),
                "forward_us": round(tr[0] * 1e6, 1), "combine_backward_us": round(tr[1] * 1e6, 1),
                "experts_backward_us": round(tr[2] * 1e6, 1), "dispatch_backward_us": round(tr[3] * 1e6, 1),
                "router_backward_us": round(tr[4] * 1e6, 1), "experts_backward_tflops": round(tf, 1),
                "experts_backward_frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                "experts_backward_frac_bf16_sustained": round(tf / peaks["bf16_tflops_sustained"], 4)}

    training = training_line(f, tr)
    training_coarse = training_line(c, trc)
    d = DECODE
    es = 2
    dec_bytes = dr["touched"] * 3 * d.I * d.H * es
    dec_fwd = dr["total_s"] / dr["steps"]
    dec_exp = dr["stages_s"][2]
    ztf = ZIPF.expert_flops / z_ch / 1e12

    def route_dispatch(r):
        """The one route + dispatch launch moe_forward runs, and beside it
        moe_route then moe_dispatch (the split API's kernels)."""
        st, sp = r["stages_s"], r["split_stages_s"]
        return {"total": round((st[0] + st[1]) * 1e6, 2),
                "maps_only": round(r["maps_only_s"] * 1e6, 2),  # the same launch without the x copy
                "split_route": round(sp[0] * 1e6, 2),
                "split_dispatch": round(sp[1] * 1e6, 2), "split_total": round((sp[0] + sp[1]) * 1e6, 2)}

    line = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) logits and x, N(0, 1/sqrt(fan_in)) expert weights (random init)",
        "config": workload_config(c, world),
        "grouped_gemm": {"tflops": roof["tflops"], "frac_bf16_peak": roof["tensor_frac"],
                         "frac_bf16_sustained": roof["tensor_frac_sustained"], "flops_per_step": c.expert_flops,
                         "chained_us": roof["us"], "gate_up_alone_us": round(t_gu * 1e6, 2),
                         "down_alone_us": round(t_dn * 1e6, 2)},
        "route_dispatch_us": route_dispatch(hr),
        "combine_us": round(hr["stages_s"][3] * 1e6, 2),
        "fused_combine_ab": hr["fused_ab"],
        "timing": {"value": f"{args.steps} CUDA-graph replays of one moe_forward call (its {KERNELS_PER_STEP} "
                            "kernels), one event pair around each replay",
                   "stages": f"{hr['stage_steps']} steps launched stage by stage with events between "
                             f"({hr['stage_total_s'] / hr['stage_steps'] * 1e6:.1f} us per step including the "
                             "events)"},
        "roofline": roof,
        "e2e": {"value": round(world * c.T / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "api": "moe_forward_host (C ABI, pinned host buffers)",
                "timing": f"{e2e_steps_n} batches alternating over two streams with two workspaces (one batch's "
                          "copies overlap the other's kernels); weights larger than L2, no flush between "
                          "batches; from an event before the first batch to the last batch's end",
                "serial": {"value": round(world * c.T / e2e_serial_s, 1), "unit": "tokens/s",
                           "timing": "one batch at a time (copy in, chain, copy out, wait), L2 flushed before "
                                     "each, outside the events; the cost of one call"}},
        "fine_prefill": {
            "workload": f.name, "tokens_per_s": round(world * f.T * fr["steps"] / fr["total_s"], 1),
            "us_per_step": round(fr["total_s"] / fr["steps"] * 1e6, 2),
            "route_dispatch_us": route_dispatch(fr),
            "experts_us": round(fr["stages_s"][2] * 1e6, 2), "combine_us": round(fr["stages_s"][3] * 1e6, 2),
            "fused_combine_ab": fr["fused_ab"],
            "gate_up_alone_us": round(f_gu * 1e6, 2), "down_alone_us": round(f_dn * 1e6, 2),
            "roofline": froof},
        "decode": {"workload": d.name, "us_per_step": round(dec_fwd * 1e6, 2),
                   "timing": "CUDA-graph replays of the decode step (forward, gate/up and down chained in one "
                             "launch); experts_us from the staged run (the two GEMMs launched apart)",
                   "route_dispatch_us": route_dispatch(dr),
                   "frac_hbm_forward": round(dec_bytes / dec_fwd / 1e9 / peaks["hbm_gbs"], 4),
                   "experts_us": round(dec_exp * 1e6, 2), "touched_experts": dr["touched"],
                   "touched_weight_bytes": dec_bytes,
                   "gbs_over_forward": round(dec_bytes / dec_fwd / 1e9, 1),
                   "gbs_over_experts": round(dec_bytes / dec_exp / 1e9, 1),
                   "frac_hbm_experts": round(dec_bytes / dec_exp / 1e9 / peaks["hbm_gbs"], 4)},
        "zipf_prefill_gemms": {"workload": ZIPF.name, "tflops": round(ztf, 1),
                               "frac_peak": round(ztf / peaks["bf16_tflops"], 4),
                               "chained_us": round(z_ch * 1e6, 1), "gate_up_alone_us": round(z_gu * 1e6, 1),
                               "down_alone_us": round(z_dn * 1e6, 1), "flops": ZIPF.expert_flops,
                               "note": "F16 and BF16 share the dense tensor rate"},
        "training_step": training,
        "training_step_coarse": training_coarse,
        "sigmoid_grouped": {
            "workload": f"{f.name} with grouped sigmoid routing: {grouped_routing.groups} groups, "
                        f"{grouped_routing.selected_groups} selected, top-two group scores, scale "
                        f"{grouped_routing.scale}, FP32 bias N(0, {grouped_routing.bias_std}^2)",
            "tokens_per_s": round(world * f.T * g_steps / g_total, 1),
            "us_per_step": round(g_total / g_steps * 1e6, 2),
            "route_dispatch_us": round(float(g_stages[0] + g_stages[1]) * 1e6, 2),
            "split_route_us": round(float(g_split[0]) * 1e6, 2),
            "split_dispatch_us": round(float(g_split[1]) * 1e6, 2),
            "softmax_split_route_us": round(fr["split_stages_s"][0] * 1e6, 2)},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clk,
    }
    if world > 1:
        dist.barrier()
    if host_inp is not None:
        line["cpu_baseline"] = cpu_baseline(c, host_inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The CPU oracle on bounded samples of the headline batch (rank 0 only)."""
    if rank != 0:
        return
    from oracle import moe_oracle

    c = HEADLINE
    n_tok = 32
    inp = workloads.generate(c)
    w64 = widened_weights(inp)
    times = []
    for i in range(args.warmup + args.steps):
        lo = (i * n_tok) % c.T
        t0 = time.perf_counter()
        moe_oracle.forward(inp["x"][lo:lo + n_tok], inp["logits"][lo:lo + n_tok], w64["gate"], w64["up"],
                           w64["down"], c.top_k, c.renormalize)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = n_tok * args.steps / total
    cores = len(os.sched_getaffinity(0))
    sample = (f"{n_tok} consecutive tokens of {c.name} per step through the whole oracle chain (expert weights "
              "widened to f64 once, before the timed steps)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) logits and x, N(0, 1/sqrt(fan_in)) expert weights (random init)",
        "config": workload_config(c, world),
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
