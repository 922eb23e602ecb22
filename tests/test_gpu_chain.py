"""GPU parity of routing, dispatch, combine and the FP32 experts against the
CPU oracle, through the C ABI (Python binding), plus the bounded-wait check."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle
from tests.parity import assert_output_close, assert_route_matches, f64, u32

pytestmark = pytest.mark.gpu
DEV = "cuda"

ALL = {f"cfg{i}": c for i, c in workloads.CONFIGS.items()}
ALL.update(workloads.SMALL_CONFIGS)


@pytest.mark.parametrize("name", sorted(ALL))
def test_route_parity(cuda_lib, name):
    moe = cuda_lib
    cfg = ALL[name]
    inp = workloads.generate(cfg, weights=False)
    ref = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    idx, w, w32 = moe.moe_route(inp["logits"].to(DEV), cfg.top_k, cfg.renormalize, weights_fp32=True)
    torch.cuda.synchronize()
    assert_route_matches(idx, w, w32, ref, cfg.torch_dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("E,k,renorm", [(1, 1, True), (3, 3, False), (33, 5, True), (64, 64, True),
                                        (1000, 7, False), (1024, 1, True)])
def test_route_edge_shapes(cuda_lib, dtype, E, k, renorm):
    """E not a multiple of 32, k = E, E = 1, the largest E, many exact ties
    (logits quantised to quarters), -inf entries and non-finite rows."""
    moe = cuda_lib
    g = torch.Generator().manual_seed(E * 131 + k)
    T = 157
    l = torch.round(torch.randn(T, E, generator=g) * 4) / 4
    l[torch.rand(T, E, generator=g) < 0.1] = float("-inf")
    l[5] = float("nan") if E > 1 else l[5]
    l[6, 0] = float("inf")
    l[7] = float("-inf")
    l = l.to(dtype)
    ref = moe_oracle.route(l, k, renorm)
    idx, w, w32 = moe.moe_route(l.to(DEV), k, renorm, weights_fp32=True)
    torch.cuda.synchronize()
    assert_route_matches(idx, w, w32, ref, dtype)


def _check_dispatch(moe, indices_np, T, E, k, x):
    ref = moe_oracle.dispatch(indices_np, E)
    idx = torch.from_numpy(indices_np.astype(np.int64)).to(torch.int32).to(DEV)
    d = moe.moe_dispatch(idx, E, x.to(DEV) if x is not None else None)
    torch.cuda.synchronize()
    assert np.array_equal(u32(d.counts), ref.counts)
    assert np.array_equal(u32(d.offsets), ref.offsets)
    n = int(ref.offsets[-1])
    assert np.array_equal(u32(d.row_src)[:n], ref.row_src)
    assert np.array_equal(u32(d.inv), ref.inv)
    if x is not None:
        rows = ref.row_src.astype(np.int64) // k
        assert torch.equal(d.x_dispatched[:n].cpu(), x[torch.from_numpy(rows)])
    return d


@pytest.mark.parametrize("name", sorted(ALL))
def test_dispatch_parity(cuda_lib, name):
    cfg = ALL[name]
    inp = workloads.generate(cfg, weights=False)
    ref = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    _check_dispatch(cuda_lib, ref.indices, cfg.T, cfg.E, cfg.top_k, inp["x"])


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (2049, 3, 2), (5000, 1024, 9), (700, 64, 64), (4097, 8, 1),
                                   (70000, 64, 2), (33000, 1000, 4)])
def test_dispatch_skewed_and_edge(cuda_lib, T, E, k):
    """Chunk boundaries (2048 slots), one hot expert, many empty experts, E = 1024, k = E;
    the last two exceed the one-block limit (131072 slots) and take the
    three-kernel path."""
    rng = np.random.default_rng(T + E + k)
    p = rng.random(E) ** 8
    p[0] += 5
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.uint32)
    x = torch.randn(T, 24, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    _check_dispatch(cuda_lib, idx, T, E, k, x)


def test_dispatch_rejects_out_of_range_index_on_device(cuda_lib):
    """An index >= E is not dispatched (no out-of-range access): its inv entry
    is 0xFFFFFFFF, counts exclude it, and combine gives that token a NaN row."""
    moe = cuda_lib
    T, E, k, H = 40, 6, 2, 16
    rng = np.random.default_rng(3)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.uint32)
    idx[7, 1] = E + 3
    idx[20, 0] = 0xFFFFFFF0
    d = moe.moe_dispatch(torch.from_numpy(idx.astype(np.int64)).to(torch.int32).to(DEV), E)
    torch.cuda.synchronize()
    inv = u32(d.inv)
    assert inv[7 * k + 1] == 0xFFFFFFFF and inv[20 * k] == 0xFFFFFFFF
    assert int(u32(d.counts).sum()) == T * k - 2 and int(u32(d.offsets)[-1]) == T * k - 2
    valid = np.ones(T * k, bool)
    valid[[7 * k + 1, 20 * k]] = False
    assert np.array_equal(np.sort(inv[valid]), np.arange(T * k - 2))
    y = torch.randn(T * k, H, device=DEV)
    w = torch.full((T, k), 0.5, device=DEV)
    out = moe.moe_combine(y, d.inv, w).cpu().numpy()
    assert np.isnan(out[[7, 20]]).all() and not np.isnan(np.delete(out, [7, 20], axis=0)).any()


@pytest.mark.parametrize("dtype,wdtype", [(torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
                                          (torch.float16, torch.float16), (torch.bfloat16, torch.float32)])
@pytest.mark.parametrize("T,k,H", [(1, 1, 8), (300, 3, 200), (64, 8, 2048), (33, 2, 4100)])
def test_combine_parity(cuda_lib, dtype, wdtype, T, k, H):
    moe = cuda_lib
    g = torch.Generator().manual_seed(T * k + H)
    y = torch.randn(T * k, H, generator=g).to(dtype)
    inv = torch.randperm(T * k, generator=g).to(torch.int32)
    w = torch.rand(T, k, generator=g).to(wdtype)
    w[0, 0] = float("nan") if T > 1 else w[0, 0]
    out = moe.moe_combine(y.to(DEV), inv.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    ref = moe_oracle.combine(f64(y), inv.numpy().view(np.uint32), f64(w), T, k)
    assert_output_close(f64(out), ref, dtype)


@pytest.mark.parametrize("name", ["f32_contract", "f32_ragged"])
def test_f32_experts_parity(cuda_lib, name):
    """FP32 SwiGLU experts on CUDA cores (no TF32) against the f64 oracle."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    inp = workloads.generate(cfg)
    rt = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    dp = moe_oracle.dispatch(rt.indices, cfg.E)
    yref = moe_oracle.experts_forward_dispatched(inp["x"], inp["gate"], inp["up"], inp["down"], dp, cfg.top_k)
    xd = inp["x"][torch.from_numpy(dp.row_src.astype(np.int64) // cfg.top_k)]
    ex = moe.Experts(inp["gate"].to(DEV), inp["up"].to(DEV), inp["down"].to(DEV))
    offs = torch.from_numpy(dp.offsets.astype(np.int64)).to(torch.int32).to(DEV)
    y = moe.moe_experts_forward_dispatched(ex, xd.to(DEV), offs)
    torch.cuda.synchronize()
    assert_output_close(f64(y), yref, torch.float32, "y_dispatched")


def test_bounded_wait_gives_up_and_reports(cuda_lib):
    """A wait on a barrier nothing arrives on runs out, records its code and
    returns; the context stays usable afterwards."""
    moe = cuda_lib
    assert moe.moe_device_status(clear=True) in (0, 0x100)
    moe.moe_selftest_bounded_wait(20_000)
    assert moe.moe_device_status(clear=True) == 0x100
    assert moe.moe_device_status(clear=True) == 0
    l = torch.randn(4, 8, device=DEV)
    idx, w = moe.moe_route(l, 2, True)
    torch.cuda.synchronize()
    assert u32(idx).shape == (4, 2)
