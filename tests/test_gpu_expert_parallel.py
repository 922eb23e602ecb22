"""The expert-parallel exchange on the GPU path, one rank (NCCL, world size 1):
the plan, the all-to-all-v of dispatched rows and their return, with the
library's own kernels for the experts and the combine, must give moe_forward's
output bit for bit. (More ranks need more GPUs; the plan itself is tested
with 2-4 CPU ranks in tests/test_expert_parallel.py.)"""
import socket

import numpy as np
import pytest
import torch

import workloads
from moe_routing_swiglu_gb300 import expert_parallel as ep

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture(scope="module")
def nccl_group():
    import torch.distributed as dist

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            device_id=torch.device(DEV, 0))
    yield dist.group.WORLD
    dist.destroy_process_group()


@pytest.mark.parametrize("name", ["bf16_fine", "f16_zipf", "bf16_coarse"])
def test_ep_one_rank_equals_forward(cuda_lib, nccl_group, name):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    d = {k: v.to(DEV) for k, v in workloads.generate(cfg).items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, w = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])

    def experts_fn(x_local, local_offsets, span):
        lo, hi = span
        sub = moe.Experts(d["gate"][lo:hi], d["up"][lo:hi], d["down"][lo:hi])
        offs = local_offsets.to(torch.int32).to(DEV)
        return moe.moe_experts_forward_dispatched(sub, x_local.contiguous(), offs)

    y = ep.ep_experts_forward(disp.x_dispatched, disp.counts, cfg.E, experts_fn, group=nccl_group)
    out = moe.moe_combine(y, disp.inv, w)
    ref = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))
    plan = ep.ep_plan(disp.counts, cfg.E, group=nccl_group)
    assert plan.send_splits == plan.recv_splits == [int(disp.offsets[-1])]
    assert np.array_equal(plan.perm.cpu().numpy(), np.arange(int(disp.offsets[-1])))
    assert moe.moe_device_status() == 0
