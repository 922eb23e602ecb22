"""Data-parallel sharding of the benchmark (bench.py --gpus N): rank r runs
its own token shard (workloads.generate(cfg, shard=r)) with the same expert
weights, and no collective touches the data. Two gloo ranks on the CPU each
run the oracle chain on their shard; the shards' outputs, concatenated, must
equal the oracle chain on the concatenated global batch (tokens are
independent: routing, dispatch and the combine are per token, and each
expert row depends on its own token only)."""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

import workloads

CFG = workloads.SMALL_CONFIGS["bf16_fine"].scaled("dp_T40_H96_I64_E12_k4", T=40, H=96, I=64, E=12, top_k=4,
                                                  seed=5201)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    from oracle import moe_oracle

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = workloads.generate(CFG, shard=rank)
        res = moe_oracle.forward(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], CFG.top_k,
                                 CFG.renormalize)
        # Gathered for the check only (the chain itself exchanges nothing).
        outs = [torch.empty(CFG.T, CFG.H, dtype=torch.float64) for _ in range(world)]
        idxs = [torch.empty(CFG.T, CFG.top_k, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(outs, torch.from_numpy(res.out))
        dist.all_gather(idxs, torch.from_numpy(res.route.indices.astype(np.int64)))
        wsum = torch.tensor([float(inp["gate"].float().sum() + inp["down"].float().sum())], dtype=torch.float64)
        wall = [torch.empty(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(wall, wsum)
        if rank == 0:
            shards = [workloads.generate(CFG, shard=r) for r in range(world)]
            x = torch.cat([s["x"] for s in shards])
            lg = torch.cat([s["logits"] for s in shards])
            ref = moe_oracle.forward(x, lg, inp["gate"], inp["up"], inp["down"], CFG.top_k, CFG.renormalize)
            got = torch.cat(outs).numpy()
            q.put({
                "indices_equal": bool(np.array_equal(torch.cat(idxs).numpy(), ref.route.indices.astype(np.int64))),
                "out_err": float(np.abs(got - ref.out).max() / np.abs(ref.out).max()),
                "weights_replicated": all(float(w) == float(wall[0]) for w in wall),
                "shards_differ": not torch.equal(shards[0]["x"], shards[1]["x"]),
            })
    finally:
        dist.destroy_process_group()


def test_two_token_shards_concatenate_to_the_global_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res["indices_equal"] and res["weights_replicated"] and res["shards_differ"], res
    # f64 expert rows grouped differently in the two runs: equal up to the BLAS's summation order.
    assert res["out_err"] <= 1e-12, res


def test_shard_zero_is_the_workload_itself():
    a = workloads.generate(CFG, weights=False)
    b = workloads.generate(CFG, shard=0, weights=False)
    assert torch.equal(a["x"], b["x"]) and torch.equal(a["logits"], b["logits"])
