"""Expert-parallel exchange plan (moe_routing_swiglu_gb300.expert_parallel) on
CPU ranks (gloo, world sizes 2, 3 and 4): every rank routes and dispatches its
own token shard, the dispatched rows travel to the ranks that own their
experts and back, and the locally combined result must equal the single-rank
oracle chain on the same tokens. The experts and the combine here are the
oracle's (the library's kernels need a GPU); what is under test is the plan:
counts exchange, splits, the expert-major permutation and the return into
each source's dispatched order."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import workloads
from moe_routing_swiglu_gb300 import expert_parallel as ep

CFG = workloads.SMALL_CONFIGS["bf16_fine"].scaled("ep_T48_H64_I40_E10_k3", T=48, H=64, I=40, E=10, top_k=3,
                                                  seed=5101)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_expert_ranges_cover_every_expert_once():
    for E in (1, 5, 8, 10, 128):
        for world in (1, 2, 3, 4, 8):
            if world > E:
                continue
            spans = [ep.expert_range(E, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == E
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    with pytest.raises(ValueError):
        ep.expert_range(4, 2, 2)


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    from oracle import moe_oracle

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = CFG
        inp = workloads.generate(c, shard=rank)
        rt = moe_oracle.route(inp["logits"], c.top_k, c.renormalize)
        disp = moe_oracle.dispatch(rt.indices, c.E)
        x64 = torch.from_numpy(moe_oracle.widen(inp["x"]))
        x_d = x64[torch.from_numpy(disp.row_src.astype(np.int64)) // c.top_k]
        counts = torch.from_numpy(disp.counts.astype(np.int64))

        def experts_fn(x_local, local_offsets, span):
            lo, hi = span
            n = x_local.shape[0]
            local = moe_oracle.DispatchResult(
                counts=np.diff(local_offsets.numpy()).astype(np.uint32),
                offsets=local_offsets.numpy().astype(np.uint32),
                row_src=(np.arange(n, dtype=np.int64) * c.top_k).astype(np.uint32),
                inv=np.zeros(n, dtype=np.uint32))
            y = moe_oracle.experts_forward_dispatched(x_local.numpy(), inp["gate"][lo:hi], inp["up"][lo:hi],
                                                      inp["down"][lo:hi], local, c.top_k)
            return torch.from_numpy(y)

        plan = ep.ep_plan(counts, c.E)
        y_d = ep.ep_experts_forward(x_d, counts, c.E, experts_fn).numpy()
        out = moe_oracle.combine(y_d, disp.inv, rt.weights, c.T, c.top_k)
        ref = moe_oracle.forward(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], c.top_k,
                                 c.renormalize)
        y_ref = moe_oracle.experts_forward_dispatched(inp["x"], inp["gate"], inp["up"], inp["down"], disp, c.top_k)
        rows_in = torch.tensor([sum(plan.recv_splits)], dtype=torch.int64)
        rows_out = torch.tensor([sum(plan.send_splits)], dtype=torch.int64)
        dist.all_reduce(rows_in)
        dist.all_reduce(rows_out)
        perm_ok = bool(torch.equal(torch.sort(plan.perm).values, torch.arange(plan.perm.numel())))
        scale = np.abs(ref.out).max()
        q.put((rank, {
            "y_err": float(np.abs(y_d - y_ref).max() / max(np.abs(y_ref).max(), 1e-300)),
            "out_err": float(np.abs(out - ref.out).max() / scale),
            "rows_balance": int(rows_in.item()) == int(rows_out.item()) == world * c.T * c.top_k,
            "perm_ok": perm_ok,
            "offsets_ok": int(plan.local_offsets[-1]) == sum(plan.recv_splits),
            "send_ok": plan.send_splits == [int(counts[a:b].sum()) for a, b in
                                            (ep.expert_range(c.E, world, r) for r in range(world))],
            "tokens_differ": world == 1 or rank == 0 or not torch.equal(
                inp["x"], workloads.generate(c, shard=0, weights=False)["x"]),
        }))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3, 4])
def test_ep_chain_equals_single_rank_oracle(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, v in res.items():
        # f64 oracle experts on other row groupings: equal up to the BLAS's summation order.
        assert v["y_err"] <= 1e-12, (r, v)
        assert v["out_err"] <= 1e-12, (r, v)
        assert v["rows_balance"] and v["perm_ok"] and v["offsets_ok"] and v["send_ok"] and v["tokens_differ"], (r, v)
