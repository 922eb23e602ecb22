"""GPU parity of the grouped, bias-corrected sigmoid routing and of the whole
chain with it (route_sigmoid_grouped / forward_sigmoid_grouped, ruDNN user
guide section 10) against the oracle, through the C ABI: indices bit-exact,
FP32 weights within 1e-6 relative, outputs within the chain's tolerances."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle
from tests.parity import assert_output_close, assert_route_matches, f64, u32

pytestmark = pytest.mark.gpu
DEV = "cuda"
Opt = moe_oracle.GroupRoutingOptions


def _opts(r):
    return Opt(r.top_k, r.groups, r.selected_groups, r.group_top_two, r.renormalize, r.scale)


def _route_both(moe, logits, bias, o):
    ref = moe_oracle.route_sigmoid_grouped(logits, bias, o)
    idx, w, w32 = moe.moe_route_sigmoid_grouped(logits.to(DEV), None if bias is None else bias.to(DEV), o,
                                                weights_fp32=True)
    torch.cuda.synchronize()
    return ref, idx, w, w32


@pytest.mark.parametrize("name", sorted(workloads.GROUPED))
def test_grouped_route_parity(cuda_lib, name):
    cfg, r = workloads.GROUPED[name]
    inp = workloads.generate(cfg, weights=False)
    ref, idx, w, w32 = _route_both(cuda_lib, inp["logits"], workloads.grouped_bias(cfg.E, r), _opts(r))
    assert_route_matches(idx, w, w32, ref, cfg.torch_dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_grouped_route_deepseek_sized(cuda_lib, dtype):
    """256 experts in 8 groups, 4 groups kept, top-8 by top-two group scores,
    a small correction bias, 4096 tokens."""
    g = torch.Generator().manual_seed(71)
    l = torch.randn(4096, 256, generator=g).to(dtype)
    b = (torch.randn(256, generator=g) * 0.01).float()
    ref, idx, w, w32 = _route_both(cuda_lib, l, b, Opt(8, 8, 4, True, True, 2.5))
    assert_route_matches(idx, w, w32, ref, dtype)


EDGE = [  # E, groups, selected, top_k, top_two
    (1, 1, 1, 1, False),
    (7, 7, 3, 3, False),        # one expert per group
    (33, 3, 2, 5, True),        # 11 experts per group, E just above a warp
    (96, 32, 5, 10, True),      # groups of 3
    (200, 8, 3, 9, True),       # groups of 25 (one lane per group)
    (256, 8, 4, 8, True),       # groups of 32 (the warp scans each group)
    (256, 4, 2, 16, False),     # groups of 64
    (1024, 128, 128, 64, True),  # every limit at once
    (1024, 1, 1, 64, False),    # one group of 1024
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("E,groups,sel,k,top_two", EDGE)
def test_grouped_route_edge_shapes(cuda_lib, dtype, E, groups, sel, k, top_two):
    """Group layouts at both branches of the group scan, many exact ties
    (logits in quarters, bias in 1/64ths), -inf and +inf logits, a NaN row,
    renormalize on and off."""
    g = torch.Generator().manual_seed(E * 7 + groups * 3 + k)
    T = 157
    l = torch.round(torch.randn(T, E, generator=g) * 4) / 4
    l[torch.rand(T, E, generator=g) < 0.05] = float("-inf")
    l[torch.rand(T, E, generator=g) < 0.02] = float("inf")
    l[5, E // 2] = float("nan")
    l[7] = float("-inf")
    b = torch.round(torch.randn(E, generator=g) * 4) / 256
    for renorm, scale in [(True, 1.0), (False, 2.5)]:
        ref, idx, w, w32 = _route_both(cuda_lib, l.to(dtype), b.float(), Opt(k, groups, sel, top_two, renorm,
                                                                               scale))
        assert_route_matches(idx, w, w32, ref, dtype)
        ref, idx, w, w32 = _route_both(cuda_lib, l.to(dtype), None, Opt(k, groups, sel, top_two, renorm, scale))
        assert_route_matches(idx, w, w32, ref, dtype)


def test_grouped_route_near_ties(cuda_lib):
    """Corrected scores one or two FP32 ulps apart: logits a few 2^-22 apart
    around 0.3, and biases that cancel the sigmoid differences of unrelated
    logits to within an ulp. The selection must still be the oracle's."""
    rng = np.random.default_rng(5)
    T, E = 2048, 64
    base = rng.choice(np.arange(-8, 9), size=(T, E)) * 2.0 ** -22 + 0.3
    l = torch.from_numpy(base.astype(np.float32))
    ref, idx, w, w32 = _route_both(cuda_lib, l, None, Opt(6, 8, 3, True, True, 1.0))
    assert_route_matches(idx, w, w32, ref, torch.float32)
    l2 = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32))
    s = 1.0 / (1.0 + np.exp(-l2.numpy().astype(np.float64)))
    b = (s[0, 0] - s[0] + rng.choice([-1, 0, 1], size=E) * 2.0 ** -24).astype(np.float32)
    ref, idx, w, w32 = _route_both(cuda_lib, l2, torch.from_numpy(b), Opt(4, 4, 2, False, True, 1.0))
    assert_route_matches(idx, w, w32, ref, torch.float32)


def test_grouped_route_special_biases(cuda_lib):
    """A -inf bias inside a selected group, +inf and -inf in one group's top
    two (a NaN group score, ranked last), and a NaN bias (every row NaN)."""
    g = torch.Generator().manual_seed(9)
    l = torch.randn(300, 16, generator=g)
    b = torch.zeros(16)
    b[3], b[8], b[9] = float("-inf"), float("inf"), float("-inf")
    for o in [Opt(4, 8, 2, True, True, 1.0), Opt(4, 8, 3, False, False, 1.0), Opt(2, 4, 1, True, True, 1.0)]:
        ref, idx, w, w32 = _route_both(cuda_lib, l, b, o)
        assert_route_matches(idx, w, w32, ref, torch.float32)
    b[5] = float("nan")
    ref, idx, w, w32 = _route_both(cuda_lib, l, b, Opt(4, 8, 2, True, True, 1.0))
    assert np.isnan(f64(w32)).all()
    assert_route_matches(idx, w, w32, ref, torch.float32)


def _device(inp):
    return {k: v.to(DEV) for k, v in inp.items()}


def _grouped_forward(moe, cfg, r, d, bias, ex=None):
    ex = ex or moe.Experts(d["gate"], d["up"], d["down"])
    idx = torch.empty(cfg.T, r.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(cfg.T, r.top_k, dtype=d["logits"].dtype, device=DEV)
    out = moe.moe_forward_sigmoid_grouped(ex, d["x"], d["logits"], bias, _opts(r), indices=idx, weights=w)
    torch.cuda.synchronize()
    return out, idx, w, ex


@pytest.mark.parametrize("name", ["bf16_fine_grouped", "f16_zipf_grouped", "f32_ragged_grouped",
                                  "bf16_ragged_grouped", "bf16_decode_grouped"])
def test_grouped_forward_full_oracle(cuda_lib, name):
    moe = cuda_lib
    cfg, r = workloads.GROUPED[name]
    inp = workloads.generate(cfg)
    bias = workloads.grouped_bias(cfg.E, r)
    out, idx, w, _ = _grouped_forward(moe, cfg, r, _device(inp), None if bias is None else bias.to(DEV))
    rt = moe_oracle.route_sigmoid_grouped(inp["logits"], bias, _opts(r))
    ref = moe_oracle.forward_with_routing(inp["x"], inp["gate"], inp["up"], inp["down"], rt)
    assert np.array_equal(u32(idx), rt.indices)
    assert_output_close(f64(out), ref.out, cfg.torch_dtype)
    assert moe.moe_device_status() == 0


def test_grouped_forward_full_size_sampled(cuda_lib):
    """The fine-grained prefill shape with grouped routing: routing in full,
    outputs on sampled tokens, and bit-identical to the split path."""
    moe = cuda_lib
    cfg, r = workloads.GROUPED["bf16_prefill_grouped"]
    inp = workloads.generate(cfg)
    bias = workloads.grouped_bias(cfg.E, r)
    d = _device(inp)
    bd = bias.to(DEV)
    out, idx, w, ex = _grouped_forward(moe, cfg, r, d, bd)
    rt = moe_oracle.route_sigmoid_grouped(inp["logits"], bias, _opts(r))
    assert np.array_equal(u32(idx), rt.indices)
    rng = np.random.default_rng(12)
    toks = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, size=192, replace=False)]))
    rt_s = moe_oracle.route_sigmoid_grouped(inp["logits"][torch.from_numpy(toks)], bias, _opts(r))
    ref = moe_oracle.forward_tokens_routed(inp["x"], inp["gate"], inp["up"], inp["down"], rt_s, toks)
    assert_output_close(f64(out)[toks], ref, cfg.torch_dtype, f"out[sampled {len(toks)} tokens]")

    idx2, w2 = moe.moe_route_sigmoid_grouped(d["logits"], bd, _opts(r))
    disp = moe.moe_dispatch(idx2, cfg.E, d["x"])
    y = moe.moe_experts_forward_dispatched(ex, disp.x_dispatched, disp.offsets)
    out2 = moe.moe_combine(y, disp.inv, w2)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
    assert torch.equal(w.view(torch.uint8), w2.view(torch.uint8))
    assert torch.equal(out.view(torch.uint8), out2.view(torch.uint8))
    assert moe.moe_device_status() == 0


def test_grouped_forward_rejects_bad_options(cuda_lib):
    moe = cuda_lib
    cfg, r = workloads.GROUPED["bf16_ragged_grouped"]
    d = _device(workloads.generate(cfg))
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    with pytest.raises(moe.MoeError) as err:
        moe.moe_forward_sigmoid_grouped(ex, d["x"], d["logits"], None, Opt(6, 1, 1, False, True, 1.0))
    assert err.value.status == 4
    with pytest.raises(moe.MoeError) as err:
        moe.moe_forward_sigmoid_grouped(ex, d["x"], d["logits"], None, Opt(2, 2, 1, False, True, 1.0))
    assert err.value.status == 2
