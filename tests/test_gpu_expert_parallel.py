"""The expert-parallel exchange on the GPU path, one rank (NCCL, world size 1):
the plan, the all-to-all-v of dispatched rows and their return, with the
library's own kernels for the reorders (moe_permute_rows), the experts and
the combine, must give moe_forward's output bit for bit. (More ranks need
more GPUs; the plan itself is tested with 2-4 CPU ranks in
tests/test_expert_parallel.py.) Then moe_permute_rows against torch indexing
of the same rows."""
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


@pytest.mark.parametrize("dtype,width", [(torch.bfloat16, 64), (torch.float32, 3), (torch.float16, 6),
                                         (torch.uint8, 5), (torch.bfloat16, 2048)])
def test_permute_rows_matches_indexing(cuda_lib, dtype, width):
    """moe_permute_rows (the exchange's reorders) against torch indexing of
    the same rows: gather and scatter by a random permutation, rows of 16-byte
    multiples and of odd byte counts."""
    moe = cuda_lib
    g = torch.Generator().manual_seed(width)
    rows = 1000
    src = (torch.randn(rows, width, generator=g) * 100).to(dtype)
    perm = torch.randperm(rows, generator=g)
    got = moe.moe_permute_rows(src.to(DEV), perm.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(got.cpu().view(torch.uint8), src[perm].view(torch.uint8))
    got = moe.moe_permute_rows(src.to(DEV), perm.to(DEV), scatter=True)
    ref = torch.empty_like(src)
    ref[perm] = src
    torch.cuda.synchronize()
    assert torch.equal(got.cpu().view(torch.uint8), ref.view(torch.uint8))


def test_permute_rows_out_of_range_indexes(cuda_lib):
    """Gather writes a zero row for an index outside the source; scatter
    skips a row whose index is outside the destination."""
    moe = cuda_lib
    src = torch.arange(1, 1 + 8 * 16, dtype=torch.float32).reshape(8, 16).to(DEV)
    idx = torch.tensor([3, -1, 8, 0, 7, 100, 2, 1], dtype=torch.int64, device=DEV)
    got = moe.moe_permute_rows(src, idx).cpu()
    s = src.cpu()
    for r, i in enumerate(idx.tolist()):
        assert torch.equal(got[r], s[i] if 0 <= i < 8 else torch.zeros(16))
    dst = torch.full((8, 16), -5.0, device=DEV)
    moe.moe_permute_rows(src, idx, scatter=True, out=dst)
    d = dst.cpu()
    for r, i in enumerate(idx.tolist()):
        if 0 <= i < 8:
            assert torch.equal(d[i], s[r])
    assert torch.equal(d[4], torch.full((16,), -5.0)) and torch.equal(d[5], torch.full((16,), -5.0))
    assert moe.moe_device_status() == 0
