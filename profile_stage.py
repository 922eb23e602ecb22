"""Run one stage of the MoE chain a few times on one workload, for profilers.

    python profile_stage.py --workload cfg1 --stage gate_up --reps 3

Workloads: cfg0..cfg4 (the five configurations, numbered from 0: F32
routing contract, fine-grained BF16 prefill, coarse BF16 prefill, BF16
decode, Zipf-skewed F16 prefill), a reduced workload's name, or
coarse_E2 (the coarse prefill's expert shape, H=4096, I=14336 and 2048 rows
per expert, on 2 experts and 2048 tokens: the same kernel on 0.9 GB instead
of 3.7 GB, for captures that replay a launch many times). The inputs
are the seeded synthetic workloads of ``workloads.py``; routing and
dispatch run once to set up the stage's inputs, then the chosen stage runs
``--reps`` times back to back (stream-ordered) and the device is synchronised.
Stages: route, dispatch, route_dispatch (routing and dispatch in one
launch, as moe_forward runs them), gate_up, gate_up_gather (x rows read
through row_src), down, experts (gate/up and down chained in one launch),
experts_combine (gate/up, down and the weighted combine in one launch:
moe_experts_forward_combine), combine, forward (moe_forward), and
route_grouped (the grouped sigmoid routing, on workloads that have a grouped
variant in ``workloads.GROUPED``), route_grouped_dispatch (the same routing
with the dispatch in one launch), backward (the experts' backward of
first-order training on a random output gradient) and combine_backward (the
combine's backward on a random output gradient).
"""
from __future__ import annotations

import argparse
import sys
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import workloads  # noqa: E402

import moe_routing_swiglu_gb300 as moe  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    names = {f"cfg{i}": c for i, c in workloads.CONFIGS.items()}
    names.update(workloads.SMALL_CONFIGS)
    names["coarse_E2"] = workloads.CONFIGS[2].scaled("bf16_prefill_T2048_H4096_I14336_E2_k2", T=2048, E=2)
    ap.add_argument("--workload", default="cfg1", choices=sorted(names))
    ap.add_argument("--stage", default="gate_up",
                    choices=["route", "dispatch", "route_dispatch", "route_grouped_dispatch", "gate_up", "gate_up_gather", "down", "experts", "experts_combine",
                             "combine", "forward", "route_grouped", "backward", "combine_backward"])
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    cfg = names[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    moe.load_library()
    d = {k: v.to(dev) for k, v in workloads.generate(cfg).items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, w = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    h = moe.moe_experts_gate_up(ex, disp.x_dispatched, disp.offsets)
    y = moe.moe_experts_down(ex, h, disp.offsets)
    grouped = [r for c, r in workloads.GROUPED.values() if c is cfg]
    if args.stage in ("route_grouped", "route_grouped_dispatch"):
        if not grouped:
            ap.error(f"{args.workload} has no grouped-routing variant")
        r = grouped[0]
        bias = workloads.grouped_bias(cfg.E, r)
        bias = None if bias is None else bias.to(dev)
        opts = moe.GroupRoutingOptions(r.top_k, r.groups, r.selected_groups, r.group_top_two, r.renormalize,
                                       r.scale)
    if args.stage == "backward":
        _, cache = moe.moe_experts_forward_training(ex, disp.x_dispatched, disp.offsets)
        g = torch.Generator().manual_seed(7)
        dy = torch.randn(cfg.T * cfg.top_k, cfg.H, generator=g).to(cfg.torch_dtype).to(dev)
    if args.stage == "combine_backward":
        g = torch.Generator().manual_seed(7)
        grad_out = torch.randn(cfg.T, cfg.H, generator=g).to(cfg.torch_dtype).to(dev)
    if args.stage == "experts_combine":
        comb_out = torch.empty(cfg.T, cfg.H, dtype=cfg.torch_dtype, device=dev)
        comb_ws = torch.empty(moe.load_library().moe_experts_forward_combine_workspace_size(ex.handle, cfg.T,
                                                                                             cfg.top_k),
                              dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    for _ in range(args.reps):
        if args.stage == "route":
            moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize, indices=idx, weights=w)
        elif args.stage == "dispatch":
            moe.moe_dispatch(idx, cfg.E, d["x"])
        elif args.stage == "route_dispatch":  # one launch, as moe_forward runs it
            gather = cfg.T * cfg.top_k <= 8 * cfg.E
            moe.moe_route_dispatch(d["logits"], cfg.top_k, cfg.renormalize, None if gather else d["x"])
        elif args.stage == "gate_up":
            moe.moe_experts_gate_up(ex, disp.x_dispatched, disp.offsets, out=h)
        elif args.stage == "gate_up_gather":
            moe.moe_experts_gate_up_gather(ex, d["x"], disp.row_src, cfg.top_k, disp.offsets, out=h)
        elif args.stage == "down":
            moe.moe_experts_down(ex, h, disp.offsets, out=y)
        elif args.stage == "experts":  # gate/up and down chained in one launch
            moe.moe_experts_forward_dispatched(ex, disp.x_dispatched, disp.offsets, out=y)
        elif args.stage == "experts_combine":  # gate/up, down and combine in one launch
            moe.moe_experts_forward_combine(ex, disp.x_dispatched, disp.offsets, disp.inv, w, out=comb_out,
                                            workspace=comb_ws)
        elif args.stage == "route_grouped":
            moe.moe_route_sigmoid_grouped(d["logits"], bias, opts, indices=idx, weights=w)
        elif args.stage == "route_grouped_dispatch":  # one launch, as moe_forward_sigmoid_grouped runs it
            gather = cfg.T * cfg.top_k <= 8 * cfg.E
            moe.moe_route_sigmoid_grouped_dispatch(d["logits"], bias, opts, None if gather else d["x"])
        elif args.stage == "backward":
            moe.moe_experts_backward(ex, cache, dy)
        elif args.stage == "combine":
            moe.moe_combine(y, disp.inv, w)
        elif args.stage == "combine_backward":
            moe.moe_combine_backward(y, disp.inv, disp.row_src, w, grad_out)
        else:
            moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    print(f"{args.stage} x{args.reps} on {cfg.name}: ok")


if __name__ == "__main__":
    main()
