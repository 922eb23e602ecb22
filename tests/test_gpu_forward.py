"""The whole chain on the GPU (moe_forward) against the oracle: full oracle on
the reduced workloads, sampled tokens on the full-size workloads (the launch
configuration the benchmark times), plus split-API equality, determinism and
degenerate sizes."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle
from tests.parity import assert_output_close, assert_route_matches, f64, u32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _device_inputs(inp):
    return {k: v.to(DEV) for k, v in inp.items()}


def _forward(moe, cfg, d, ex=None):
    ex = ex or moe.Experts(d["gate"], d["up"], d["down"])
    idx = torch.empty(cfg.T, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, cfg.top_k, dtype=d["logits"].dtype, device=DEV)
    out = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize, indices=idx, weights=w)
    torch.cuda.synchronize()
    return out, idx, w, ex


@pytest.mark.parametrize("name", sorted(workloads.SMALL_CONFIGS))
def test_forward_full_oracle(cuda_lib, name):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    inp = workloads.generate(cfg)
    out, idx, w, _ = _forward(moe, cfg, _device_inputs(inp))
    ref = moe_oracle.forward(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], cfg.top_k,
                             cfg.renormalize)
    assert np.array_equal(u32(idx), ref.route.indices)
    assert_output_close(f64(out), ref.out, cfg.torch_dtype)
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("cfg_id,n_sample", [(1, 192), (2, 48), (3, 16), (4, 192)])
def test_forward_full_size_sampled(cuda_lib, cfg_id, n_sample):
    """Full-size workloads in the benchmark's launch configuration: routing
    and dispatch compared in full, outputs on sampled tokens (first, last and
    a seeded sample)."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[cfg_id]
    inp = workloads.generate(cfg)
    d = _device_inputs(inp)
    out, idx, w, ex = _forward(moe, cfg, d)
    rt = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    assert np.array_equal(u32(idx), rt.indices)
    _, _, w32 = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize, weights_fp32=True)
    assert_route_matches(idx, w, w32, rt, cfg.torch_dtype)
    rng = np.random.default_rng(cfg_id)
    toks = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, size=min(n_sample, cfg.T), replace=False)]))
    ref = moe_oracle.forward_tokens(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], cfg.top_k,
                                    cfg.renormalize, toks)
    got = f64(out)[toks]
    assert_output_close(got, ref, cfg.torch_dtype, f"out[sampled {len(toks)} tokens]")
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("name", ["f32_contract", "bf16_fine", "f16_zipf", "bf16_ragged"])
def test_forward_equals_split_api(cuda_lib, name):
    """moe_forward is bit-identical to route -> dispatch -> forward_dispatched -> combine."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    d = _device_inputs(workloads.generate(cfg))
    out, idx, w, ex = _forward(moe, cfg, d)
    idx2, w2 = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx2, cfg.E, d["x"])
    y = moe.moe_experts_forward_dispatched(ex, disp.x_dispatched, disp.offsets)
    out2 = moe.moe_combine(y, disp.inv, w2)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
    assert torch.equal(w.view(torch.uint8), w2.view(torch.uint8))  # bitwise, NaN rows included
    assert torch.equal(out.view(torch.uint8), out2.view(torch.uint8))


@pytest.mark.parametrize("cfg_id", [1, 4])
def test_forward_equals_split_api_full_size(cuda_lib, cfg_id):
    """At full size (thousands of tiles): moe_forward is bit-identical, three
    times in a row, to the split route -> dispatch -> experts -> combine path."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[cfg_id]
    d = _device_inputs(workloads.generate(cfg))
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx2, w2 = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx2, cfg.E, d["x"])
    y = moe.moe_experts_forward_dispatched(ex, disp.x_dispatched, disp.offsets)
    ref = moe.moe_combine(y, disp.inv, w2)
    for _ in range(3):
        out, _, _, _ = _forward(moe, cfg, d, ex)
        assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("name", ["bf16_fine", "f16_zipf"])
def test_forward_deterministic(cuda_lib, name):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    d = _device_inputs(workloads.generate(cfg))
    a, _, _, ex = _forward(moe, cfg, d)
    b, _, _, _ = _forward(moe, cfg, d, ex)
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("T", [0, 1, 3])
def test_forward_tiny_token_counts(cuda_lib, T):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_fine"].scaled("tiny", T=max(T, 1), seed=99)
    inp = workloads.generate(cfg)
    inp["x"], inp["logits"] = inp["x"][:T], inp["logits"][:T]
    d = _device_inputs(inp)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    out = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert out.shape == (T, cfg.H)
    if T:
        ref = moe_oracle.forward(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], cfg.top_k,
                                 cfg.renormalize)
        assert_output_close(f64(out), ref.out, cfg.torch_dtype)


def test_forward_workspace_too_small_is_rejected(cuda_lib):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_ragged"]
    d = _device_inputs(workloads.generate(cfg))
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    need = moe.moe_forward_workspace_size(ex, cfg.T, cfg.top_k)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, True, workspace=ws)
    assert err.value.status == 6
    with pytest.raises(moe.MoeError) as err:
        moe.moe_forward(ex, d["x"], d["logits"], cfg.E + 1, True)
    assert err.value.status == 4


@pytest.mark.parametrize("name", ["bf16_fine", "f16_zipf", "f32_contract"])
@pytest.mark.parametrize("pinned", [True, False])
def test_forward_host_equals_forward(cuda_lib, name, pinned):
    """moe_forward_host (host x/logits in, host out back) gives moe_forward's
    outputs bit for bit, with pinned and with pageable host memory."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    inp = workloads.generate(cfg)
    out, idx, w, ex = _forward(moe, cfg, _device_inputs(inp))
    hx, hl = inp["x"].contiguous(), inp["logits"].contiguous()
    if pinned:
        hx, hl = hx.pin_memory(), hl.pin_memory()
    hout = torch.empty(cfg.T, cfg.H, dtype=cfg.torch_dtype)
    if pinned:
        hout = hout.pin_memory()
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    moe.moe_forward_host(ex, hx, hl, cfg.top_k, cfg.renormalize, out=hout, indices=idx2, weights=w2)
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.uint8), out.cpu().view(torch.uint8))
    assert torch.equal(idx2, idx) and torch.equal(w2.view(torch.uint8), w.view(torch.uint8))
    assert moe.moe_device_status() == 0


def test_forward_host_two_streams_pipelined(cuda_lib):
    """Consecutive batches alternating over two streams and two workspaces
    (one batch's copies overlapping the other's kernels), the prefill
    workload at full size: every batch's host output equals moe_forward's."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[1]
    base = workloads.generate(cfg)
    d = _device_inputs(base)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    batches = []
    for b in range(4):
        g = torch.Generator().manual_seed(100 + b)
        x = (torch.randn(cfg.T, cfg.H, generator=g)).to(cfg.torch_dtype).pin_memory()
        lg = (torch.randn(cfg.T, cfg.E, generator=g)).to(cfg.torch_dtype).pin_memory()
        batches.append((x, lg))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    nbytes = moe.load_library().moe_forward_host_workspace_size(ex.handle, cfg.T, cfg.top_k, moe._dt(batches[0][1]))
    wss = [torch.empty(nbytes, dtype=torch.uint8, device=DEV) for _ in range(2)]
    outs = [torch.empty(cfg.T, cfg.H, dtype=cfg.torch_dtype).pin_memory() for _ in range(4)]
    for b, (x, lg) in enumerate(batches):
        moe.moe_forward_host(ex, x, lg, cfg.top_k, cfg.renormalize, out=outs[b], workspace=wss[b % 2],
                             stream=streams[b % 2])
    torch.cuda.synchronize()
    for b, (x, lg) in enumerate(batches):
        ref = moe.moe_forward(ex, x.to(DEV), lg.to(DEV), cfg.top_k, cfg.renormalize)
        torch.cuda.synchronize()
        assert torch.equal(outs[b].view(torch.uint8), ref.cpu().view(torch.uint8)), f"batch {b}"
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("T", [0, 1, 3])
def test_forward_host_tiny_token_counts(cuda_lib, T):
    """moe_forward_host on 0, 1 and 3 tokens equals moe_forward (T = 0: an
    empty output, no copies)."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_fine"].scaled("tiny", T=max(T, 1), seed=99)
    inp = workloads.generate(cfg)
    hx, hl = inp["x"][:T].contiguous().pin_memory(), inp["logits"][:T].contiguous().pin_memory()
    d = _device_inputs(inp)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    out = moe.moe_forward_host(ex, hx, hl, cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert out.shape == (T, cfg.H) and not out.is_cuda
    if T:
        ref = moe.moe_forward(ex, hx.to(DEV), hl.to(DEV), cfg.top_k, cfg.renormalize)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.uint8), ref.cpu().view(torch.uint8))


def test_forward_host_rejects_bad_arguments(cuda_lib):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_ragged"]
    inp = workloads.generate(cfg)
    d = _device_inputs(inp)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    hx, hl = inp["x"].contiguous().pin_memory(), inp["logits"].contiguous().pin_memory()
    lib = moe.load_library()
    need = lib.moe_forward_host_workspace_size(ex.handle, cfg.T, cfg.top_k, moe._dt(hl))
    assert need >= lib.moe_forward_workspace_size(ex.handle, cfg.T, cfg.top_k)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_forward_host(ex, hx, hl, cfg.top_k, True, workspace=ws)
    assert err.value.status == 6
    with pytest.raises(moe.MoeError) as err:
        moe.moe_forward_host(ex, hx, hl, cfg.E + 1, True)
    assert err.value.status == 4
    with pytest.raises(moe.MoeError):
        moe.moe_forward_host(ex, d["x"], hl, cfg.top_k, True)      # a device tensor where host memory belongs
    assert lib.moe_forward_host_workspace_size(ex.handle, cfg.T, cfg.top_k, 7) == 0


@pytest.mark.parametrize("cfg_id", [1, 2])
def test_token_shards_equal_the_global_batch(cuda_lib, cfg_id):
    """Data-parallel sharding on the GPU path: moe_forward on two token shards
    (workloads.generate shard=0 and shard=1, the same experts) equals, row
    for row and bit for bit, moe_forward on their concatenation. A row's
    expert outputs do not depend on which other rows share its tiles."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[cfg_id]
    full = workloads.generate(cfg)
    other = workloads.generate(cfg, weights=False, shard=1)
    d = _device_inputs(full)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    x1, l1 = other["x"].to(DEV), other["logits"].to(DEV)
    out0 = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    out1 = moe.moe_forward(ex, x1, l1, cfg.top_k, cfg.renormalize)
    both = moe.moe_forward(ex, torch.cat([d["x"], x1]), torch.cat([d["logits"], l1]), cfg.top_k,
                           cfg.renormalize)
    torch.cuda.synchronize()
    assert torch.equal(both.view(torch.uint8), torch.cat([out0, out1]).view(torch.uint8))
    assert moe.moe_device_status() == 0
