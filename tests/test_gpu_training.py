"""GPU parity of first-order training (ruDNN user guide, section 12) against
the training oracle, through the C ABI: router weights and their gradient,
the training forward's cache, combine backward, the experts' backward and
dispatch backward."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import moe_oracle
from tests.grad_bounds import ACC, UNIT, assert_within_bound, expert_error_bounds
from tests.parity import assert_nan_positions_equal, f64, u32

pytestmark = pytest.mark.gpu
DEV = "cuda"
Opt = oracle.RouterWeightOptions
VARIANTS = [Opt("softmax", False, 1.0), Opt("softmax", True, 1.0), Opt("sigmoid", False, 1.5),
            Opt("sigmoid", True, 2.5)]
_ULP = {torch.float32: 2.0 ** -23, torch.float16: 2.0 ** -10, torch.bfloat16: 2.0 ** -7}


def _router_inputs(T, E, k, dtype, seed, idx_dtype=torch.int32):
    g = torch.Generator().manual_seed(seed)
    l = (torch.randn(T, E, generator=g) * 2).to(dtype)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)])
    idx[1, 1] = idx[1, 0]                      # a repeated index gathers twice
    idx[2, 0] = E + 3                          # an invalid index: NaN row
    gw = torch.randn(T, k, generator=g)
    return l, idx.to(idx_dtype), gw


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("E,k", [(8, 2), (64, 6), (128, 8), (200, 64), (1024, 7)])
def test_router_weights_and_backward_parity(cuda_lib, dtype, E, k):
    moe = cuda_lib
    T = 97
    l, idx, gw = _router_inputs(T, E, k, dtype, E * 31 + k)
    for i, o in enumerate(VARIANTS):
        it = [torch.int32, torch.int64, torch.int32, torch.int64][i]
        w = moe.moe_router_weights(l.to(DEV), idx.to(it).to(DEV), o)
        d = moe.moe_router_backward(l.to(DEV), idx.to(it).to(DEV), gw.to(DEV), o)
        torch.cuda.synchronize()
        w32, _ = oracle.selected_router_weights(l, idx.numpy(), o)
        d64, _ = oracle.selected_router_backward(l, idx.numpy(), gw, o)
        gwv = f64(w)
        assert_nan_positions_equal(gwv, w32.astype(np.float64), "router weights")
        fin = np.isfinite(w32)
        rel = np.abs(gwv[fin] - w32[fin]) / np.maximum(np.abs(w32[fin]), 1e-30)
        assert rel.max() <= 1e-6, f"{o}: weight rel error {rel.max():.3e}"
        gd = f64(d)
        assert_nan_positions_equal(gd, d64, "dlogits")
        rows = np.isfinite(d64).all(axis=1)
        bound = 4e-6 * o.scale * np.abs(gw.numpy().astype(np.float64)).sum(axis=1)[rows][:, None]
        err = np.abs(gd[rows] - d64[rows])
        assert (err <= _ULP[dtype] * np.abs(d64[rows]) + bound + 1e-30).all(), \
            f"{o}: dlogits error {err.max():.3e} (bound {bound.max():.3e})"


def test_router_sigmoid_backward_is_local(cuda_lib):
    """Sigmoid scoring: logits outside the selection get an exact zero gradient."""
    moe = cuda_lib
    l, idx, gw = _router_inputs(64, 40, 5, torch.float32, 3)
    idx[2, 0] = 0
    d = moe.moe_router_backward(l.to(DEV), idx.to(DEV), gw.to(DEV), Opt("sigmoid", True, 1.0)).cpu()
    mask = torch.zeros(64, 40, dtype=torch.bool)
    mask.scatter_(1, idx.long(), True)
    assert (d[~mask] == 0).all()


def _small_training_case(name, seed=5):
    cfg = workloads.SMALL_CONFIGS[name]
    inp = workloads.generate(cfg)
    rt = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    dp = moe_oracle.dispatch(rt.indices, cfg.E)
    xd = inp["x"][torch.from_numpy(dp.row_src.astype(np.int64) // cfg.top_k)]
    g = torch.Generator().manual_seed(seed)
    dy = (torch.randn(cfg.T * cfg.top_k, cfg.H, generator=g) * 0.5).to(cfg.torch_dtype)
    return cfg, inp, rt, dp, xd, dy


def check_experts_training(cache, gr, xd, gate, up, down, offsets, dy, dtype, what=""):
    """The training forward's cache (g, u, h) and the experts' backward
    against the oracle, which recomputes the cache itself in f64 from x (it
    never sees the GPU's cache), each entry within its rounding bound
    (tests/grad_bounds.py). Only the dispatched rows [0, offsets[E]) count."""
    n = int(offsets[-1])
    bounds = expert_error_bounds(xd, gate, up, down, offsets, dy, dtype)
    g_ref, u_ref, h_ref = oracle.training_forward_cache(xd, gate, up, offsets)
    for name, got, ref in (("g", cache.g, g_ref), ("u", cache.u, u_ref), ("h", cache.h, h_ref)):
        assert_within_bound(f64(got)[:n], ref[:n], bounds[name][:n], f"{what}cache {name}")
    ref = oracle.experts_backward(xd, gate, up, down, offsets, dy)
    assert_within_bound(f64(gr.dx_dispatched)[:n], ref.dx_dispatched[:n], bounds["dx"][:n], f"{what}dx_dispatched")
    for name in ("dgate", "dup", "ddown"):
        assert_within_bound(f64(getattr(gr, name)), getattr(ref, name), bounds[name], f"{what}{name}")


@pytest.mark.parametrize("name", ["f32_ragged", "bf16_ragged", "bf16_fine", "f16_zipf", "bf16_decode"])
def test_experts_training_forward_and_backward_parity(cuda_lib, name):
    moe = cuda_lib
    cfg, inp, rt, dp, xd, dy = _small_training_case(name)
    d = {k: v.to(DEV) for k, v in inp.items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    offs = torch.from_numpy(dp.offsets.astype(np.int64)).to(torch.int32).to(DEV)
    xdd = xd.to(DEV).contiguous()
    y, cache = moe.moe_experts_forward_training(ex, xdd, offs)
    y_ref = moe.moe_experts_forward_dispatched(ex, xdd, offs)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.uint8), y_ref.view(torch.uint8))
    gr = moe.moe_experts_backward(ex, cache, dy.to(DEV))
    torch.cuda.synchronize()
    check_experts_training(cache, gr, xd, inp["gate"], inp["up"], inp["down"], dp.offsets, dy, cfg.torch_dtype)
    assert moe.moe_device_status() == 0


def test_experts_training_coarse_expert_shape(cuda_lib):
    """The coarse prefill's expert shape (H = 4096, I = 14336) on two experts
    with 300 and 300 rows (every token on both): the training forward's cache
    and the tensor-core backward against the oracle, entry by entry."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[2].scaled("coarse_shape_T300_E2_k2", T=300, E=2, seed=5301)
    inp = workloads.generate(cfg)
    rt = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    dp = moe_oracle.dispatch(rt.indices, cfg.E)
    xd = inp["x"][torch.from_numpy(dp.row_src.astype(np.int64) // cfg.top_k)]
    g = torch.Generator().manual_seed(17)
    dy = (torch.randn(cfg.T * cfg.top_k, cfg.H, generator=g) * 0.5).to(cfg.torch_dtype)
    d = {k: v.to(DEV) for k, v in inp.items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    offs = torch.from_numpy(dp.offsets.astype(np.int64)).to(torch.int32).to(DEV)
    xdd = xd.to(DEV).contiguous()
    y, cache = moe.moe_experts_forward_training(ex, xdd, offs)
    gr = moe.moe_experts_backward(ex, cache, dy.to(DEV))
    torch.cuda.synchronize()
    check_experts_training(cache, gr, xd, inp["gate"], inp["up"], inp["down"], dp.offsets, dy, cfg.torch_dtype)
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("which", ["u_is_g", "h_is_u"])
def test_planted_wrong_cache_entry_is_caught(cuda_lib, which):
    """A cache whose u holds the gate pre-activation (or whose h holds u),
    planted by overwriting the cached tensor from the host before the
    backward, fails the parity check of the cache and of the gradients the
    backward computes from it: the oracle recomputes g, u and h from x."""
    moe = cuda_lib
    cfg, inp, rt, dp, xd, dy = _small_training_case("bf16_fine")
    d = {k: v.to(DEV) for k, v in inp.items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    offs = torch.from_numpy(dp.offsets.astype(np.int64)).to(torch.int32).to(DEV)
    _, cache = moe.moe_experts_forward_training(ex, xd.to(DEV).contiguous(), offs)
    if which == "u_is_g":
        cache.u.copy_(cache.g)
    else:
        cache.h.copy_(cache.u)
    gr = moe.moe_experts_backward(ex, cache, dy.to(DEV))
    torch.cuda.synchronize()
    with pytest.raises(AssertionError, match="cache u" if which == "u_is_g" else "cache h"):
        check_experts_training(cache, gr, xd, inp["gate"], inp["up"], inp["down"], dp.offsets, dy, cfg.torch_dtype)
    # The gradients alone catch it too (the cache check is not what fails them).
    ref = oracle.experts_backward(xd, inp["gate"], inp["up"], inp["down"], dp.offsets, dy)
    bounds = expert_error_bounds(xd, inp["gate"], inp["up"], inp["down"], dp.offsets, dy, cfg.torch_dtype)
    with pytest.raises(AssertionError):
        for name in ("dgate", "dup", "ddown"):
            assert_within_bound(f64(getattr(gr, name)), getattr(ref, name), bounds[name], name)
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("name", ["f32_contract", "bf16_fine", "f16_zipf", "bf16_ragged"])
def test_combine_and_dispatch_backward_parity(cuda_lib, name):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    inp = workloads.generate(cfg, weights=False)
    rt = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    dp = moe_oracle.dispatch(rt.indices, cfg.E)
    g = torch.Generator().manual_seed(17)
    n = cfg.T * cfg.top_k
    y = torch.randn(n, cfg.H, generator=g).to(cfg.torch_dtype)
    go = torch.randn(cfg.T, cfg.H, generator=g).to(cfg.torch_dtype)
    w = torch.from_numpy(rt.weights).to(cfg.torch_dtype)
    inv = torch.from_numpy(dp.inv.astype(np.int64)).to(torch.int32)
    # row -> slot for the dispatched rows; the entries past them hold an
    # invalid slot (the kernel only trusts rows with inv[row_src[r]] == r)
    rs = np.full(n, 0xFFFFFFFF, dtype=np.uint32)
    rs[:dp.row_src.size] = dp.row_src
    row_src = torch.from_numpy(rs.view(np.int32).copy())
    dexp, dw = moe.moe_combine_backward(y.to(DEV), inv.to(DEV), row_src.to(DEV), w.to(DEV), go.to(DEV))
    torch.cuda.synchronize()
    ref_dexp, ref_dw = oracle.combine_backward(y, dp.inv, f64(w), go, cfg.T, cfg.top_k)
    used = int(dp.offsets[-1])
    got = f64(dexp)[:used]
    ref = ref_dexp[:used]
    assert_nan_positions_equal(got, ref, "dexpert")
    fin = np.isfinite(ref)
    # one rounding of the exact FP32 product to the dtype (half a subnormal
    # step near zero for f16)
    tiny = 2.0 ** -25 if cfg.torch_dtype == torch.float16 else 1e-30
    assert (np.abs(got[fin] - ref[fin]) <= _ULP[cfg.torch_dtype] * np.abs(ref[fin]) + tiny).all()
    gdw = f64(dw)
    assert_nan_positions_equal(gdw, ref_dw, "dweights")
    fin = np.isfinite(ref_dw)
    scale = (np.abs(f64(go))[:, None, :] * np.abs(f64(y))[dp.inv.astype(np.int64).reshape(cfg.T, cfg.top_k) % n]).sum(-1)
    assert (np.abs(gdw[fin] - ref_dw[fin]) <= 1e-5 * scale[fin] + 1e-30).all()

    dx = moe.moe_dispatch_backward(dexp, inv.to(DEV), cfg.T, cfg.top_k)
    torch.cuda.synchronize()
    ref_dx = oracle.dispatch_backward(dexp.cpu(), dp.inv, cfg.T, cfg.top_k)
    gdx = f64(dx)
    assert_nan_positions_equal(gdx, ref_dx, "dx")
    fin = np.isfinite(ref_dx)
    assert (np.abs(gdx[fin] - ref_dx[fin]) <= _ULP[cfg.torch_dtype] * np.abs(ref_dx[fin]) * 1.0000001 + tiny).all()


def test_dispatch_backward_invalid_slot_gives_nan_row(cuda_lib):
    moe = cuda_lib
    idx = torch.tensor([[0, 1], [1, 9], [2, 0]], dtype=torch.int32)   # token 1 holds an invalid index
    d = moe.moe_dispatch(idx.to(DEV), 3)
    dinput = torch.randn(6, 8).to(torch.bfloat16).to(DEV)
    dx = moe.moe_dispatch_backward(dinput, d.inv, 3, 2).cpu().float()
    assert torch.isnan(dx[1]).all() and torch.isfinite(dx[0]).all() and torch.isfinite(dx[2]).all()


def test_whole_training_step_matches_oracle(cuda_lib):
    """One whole first-order step on the reduced fine-grained workload:
    route -> dispatch -> training forward; then combine backward -> experts
    backward -> dispatch backward, and the router gradient of the FP32
    dweights (softmax, renormalize); every stage checked against the oracle
    on the inputs that stage received on the GPU (the experts' cache
    excepted: the oracle recomputes it from x), within rounding bounds
    derived from the documented roundings."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_fine"]
    inp = workloads.generate(cfg)
    d = {k: v.to(DEV) for k, v in inp.items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, w = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    y, cache = moe.moe_experts_forward_training(ex, disp.x_dispatched, disp.offsets)
    g = torch.Generator().manual_seed(23)
    go = (torch.randn(cfg.T, cfg.H, generator=g)).to(cfg.torch_dtype)
    dexp, dw = moe.moe_combine_backward(y, disp.inv, disp.row_src, w, go.to(DEV))
    gr = moe.moe_experts_backward(ex, cache, dexp)
    dx = moe.moe_dispatch_backward(gr.dx_dispatched, disp.inv, cfg.T, cfg.top_k)
    o = Opt("softmax", True, 1.0)
    dl = moe.moe_router_backward(d["logits"], idx, dw, o)
    torch.cuda.synchronize()

    rt = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    dp = moe_oracle.dispatch(rt.indices, cfg.E)
    assert np.array_equal(u32(idx), rt.indices)
    assert np.array_equal(u32(disp.inv), dp.inv)
    xd = inp["x"][torch.from_numpy(dp.row_src.astype(np.int64) // cfg.top_k)]
    assert torch.equal(disp.x_dispatched.cpu().view(torch.int16), xd.view(torch.int16))
    T, k, H = cfg.T, cfg.top_k, cfg.H
    # Combine backward on the forward's y; dweights is an FP32 dot over H.
    ref_dexp, ref_dw = oracle.combine_backward(y.cpu(), dp.inv, rt.weights, go, T, k)
    dw_abs = (np.abs(f64(go))[:, None, :] * np.abs(f64(y))[dp.inv.astype(np.int64).reshape(T, k)]).sum(-1)
    assert_within_bound(dw, ref_dw, H * ACC * dw_abs + 2.0 ** -24 * np.abs(ref_dw), "dweights")
    # The experts' cache and backward: the oracle recomputes g, u and h from x.
    check_experts_training(cache, gr, xd, inp["gate"], inp["up"], inp["down"], dp.offsets, dexp.cpu(),
                           cfg.torch_dtype)
    # Dispatch backward: k rows added in FP32, rounded once to the dtype.
    ref_dx = oracle.dispatch_backward(gr.dx_dispatched.cpu(), dp.inv, T, k)
    dx_abs = oracle.dispatch_backward(np.abs(f64(gr.dx_dispatched)), dp.inv, T, k)
    assert_within_bound(dx, ref_dx, UNIT[cfg.torch_dtype] * np.abs(ref_dx) + k * ACC * dx_abs, "dx")
    # Router gradient: FP32 evaluation (the router test's bound), rounded to the logits dtype.
    ref_dl, _ = oracle.selected_router_backward(inp["logits"], rt.indices, dw.cpu(), o)
    dl_bound = UNIT[cfg.torch_dtype] * np.abs(ref_dl) + 4e-6 * o.scale * np.abs(f64(dw)).sum(axis=1, keepdims=True)
    assert_within_bound(dl, ref_dl, dl_bound, "dlogits")
    assert moe.moe_device_status() == 0


def test_experts_backward_full_size_sampled_experts(cuda_lib):
    """The fine-grained prefill workload at full size (the benchmark's launch
    configuration): the tensor-core backward against the oracle on three
    sampled experts (their rows, weights and gradients cut out of the full
    problem), including the expert with the most rows."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[1]
    inp = workloads.generate(cfg)
    d = {k: v.to(DEV) for k, v in inp.items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, w = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    y, cache = moe.moe_experts_forward_training(ex, disp.x_dispatched, disp.offsets)
    g = torch.Generator().manual_seed(29)
    dy = (torch.randn(cfg.T * cfg.top_k, cfg.H, generator=g) * 0.5).to(cfg.torch_dtype)
    gr = moe.moe_experts_backward(ex, cache, dy.to(DEV))
    torch.cuda.synchronize()
    offs = u32(disp.offsets).astype(np.int64)
    counts = np.diff(offs)
    xd_all = disp.x_dispatched.cpu()
    for e in sorted({0, 77, int(np.argmax(counts))}):
        lo, hi = int(offs[e]), int(offs[e + 1])
        sub = _Sub(cache, lo, hi)
        sub_gr = _Sub(gr, lo, hi, e)
        check_experts_training(sub, sub_gr, xd_all[lo:hi], inp["gate"][e:e + 1], inp["up"][e:e + 1],
                               inp["down"][e:e + 1], np.array([0, hi - lo]), dy[lo:hi], cfg.torch_dtype,
                               what=f"expert {e}: ")
    assert moe.moe_device_status() == 0


class _Sub:
    """The rows [lo, hi) of a cache or of the row gradients, and expert e's
    weight gradients (one expert cut out of the full problem)."""

    def __init__(self, src, lo, hi, e=None):
        for name in ("g", "u", "h", "dx_dispatched"):
            if hasattr(src, name):
                setattr(self, name, getattr(src, name)[lo:hi])
        if e is not None:
            for name in ("dgate", "dup", "ddown"):
                setattr(self, name, getattr(src, name)[e:e + 1])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_experts_backward_expert_row_counts_around_the_k_steps(cuda_lib, dtype):
    """The weight-gradient GEMMs take K over an expert's rows in blocks of 64,
    16 rows per MMA: counts on both sides of 16 and 64 (and 0, 1, 130) check
    that the MMAs past an expert's end are skipped and the rows of the next
    expert inside the last one are zeroed (each expert's rows here are the
    next expert's garbage). Ragged H and I clip the tiles too."""
    moe = cuda_lib
    counts = [0, 1, 15, 16, 17, 63, 64, 65, 127, 130, 3]
    E, H, I = len(counts), 136, 200
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(41)
    gate = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dtype)
    up = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dtype)
    down = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(dtype)
    xd = torch.randn(rows, H, generator=g).to(dtype)
    dy = (torch.randn(rows, H, generator=g) * 0.5).to(dtype)
    ex = moe.Experts(gate.to(DEV), up.to(DEV), down.to(DEV))
    offs = torch.from_numpy(offsets).to(torch.int32).to(DEV)
    y, cache = moe.moe_experts_forward_training(ex, xd.to(DEV), offs)
    gr = moe.moe_experts_backward(ex, cache, dy.to(DEV))
    torch.cuda.synchronize()
    check_experts_training(cache, gr, xd, gate, up, down, offsets, dy, dtype)
    assert (gr.dgate[0] == 0).all() and (gr.ddown[0] == 0).all()  # the expert without rows
    assert moe.moe_device_status() == 0


def test_combine_backward_ignores_row_src_past_the_dispatched_rows(cuda_lib):
    """row_src entries past the dispatched rows (here: a token with an invalid
    index, so one row fewer than slots) may hold anything, even a valid slot:
    the results equal those with a clean row_src."""
    moe = cuda_lib
    idx = torch.tensor([[0, 1], [1, 9], [2, 0]], dtype=torch.int32)   # slot 3 is invalid: 5 rows for 6 slots
    d = moe.moe_dispatch(idx.to(DEV), 3)
    g = torch.Generator().manual_seed(3)
    y = torch.randn(6, 64, generator=g).to(torch.bfloat16).to(DEV)
    go = torch.randn(3, 64, generator=g).to(torch.bfloat16).to(DEV)
    w = torch.rand(3, 2, generator=g).to(torch.bfloat16).to(DEV)
    clean = d.row_src.clone()
    clean[5] = -1
    dirty = d.row_src.clone()
    dirty[5] = 0                                                      # a valid slot, not this row's
    e1, w1 = moe.moe_combine_backward(y, d.inv, clean, w, go)
    e2, w2 = moe.moe_combine_backward(y, d.inv, dirty, w, go)
    torch.cuda.synchronize()
    assert torch.equal(e1[:5].view(torch.uint8), e2[:5].view(torch.uint8))
    assert torch.equal(w1.view(torch.int32), w2.view(torch.int32))
    assert torch.isnan(w1[1, 1]) and torch.isfinite(w1[0]).all()


def test_training_forward_workspace_holds_the_counters(cuda_lib):
    """The chained training forward keeps a tile counter and one ready counter
    per expert in its workspace: the documented size is 256 + 4 E bytes, and
    anything smaller is rejected before any launch."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_ragged"]
    inp = workloads.generate(cfg)
    d = {k: v.to(DEV) for k, v in inp.items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    lib = moe.load_library()
    need = lib.moe_experts_forward_training_workspace_size(ex.handle)
    assert need == 256 + 4 * cfg.E
    idx, _ = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    with pytest.raises(moe.MoeError) as err:
        moe.moe_experts_forward_training(ex, disp.x_dispatched, disp.offsets,
                                         workspace=torch.empty(need - 4, dtype=torch.uint8, device=DEV))
    assert err.value.status == 6
    y, _ = moe.moe_experts_forward_training(ex, disp.x_dispatched, disp.offsets,
                                            workspace=torch.empty(need, dtype=torch.uint8, device=DEV))
    y_ref = moe.moe_experts_forward_dispatched(ex, disp.x_dispatched, disp.offsets)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.uint8), y_ref.view(torch.uint8))
    assert moe.moe_device_status() == 0
