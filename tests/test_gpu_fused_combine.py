"""The combine run inside the experts' launch (moe_experts_forward_combine:
once every down tile has stored its rows, the epilogue warps of all CTAs
combine a fixed stripe of the tokens) against the separate combine
(moe_experts_forward_dispatched then moe_combine, which sums in the same slot
order with the same FP32 arithmetic) bit for bit, and against the oracle;
moe_forward (which keeps the combine as its own launch) is checked beside it.

The cases aim at the fused path's own logic: a partial last 256-column block
(H not a multiple of 256), top_k = 1, top_k = E and top_k = 64 (the largest
the fused path stages), every token on the same two experts, routing-contract
rows whose NaN weights must turn whole output rows into NaN, FP32 routing
weights with 16-bit experts, a decode-sized batch, top_k above 64 (refused by
the fused call) and repeated full-size runs (the bits must not change)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle
from tests.parity import assert_output_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(inp):
    return {k: v.to(DEV) for k, v in inp.items()}


def _split_out(moe, ex, d, cfg, logits=None):
    """route -> dispatch -> forward_dispatched -> combine (the unfused path)."""
    lg = d["logits"] if logits is None else logits
    idx, w = moe.moe_route(lg, cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    y = moe.moe_experts_forward_dispatched(ex, disp.x_dispatched, disp.offsets)
    return moe.moe_combine(y, disp.inv, w), idx, w, disp


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


CASES = {
    "bf16_fine": workloads.SMALL_CONFIGS["bf16_fine"],
    "f16_zipf": workloads.SMALL_CONFIGS["f16_zipf"],
    "bf16_coarse": workloads.SMALL_CONFIGS["bf16_coarse"],
    "bf16_ragged_H136": workloads.SMALL_CONFIGS["bf16_ragged"],
    "bf16_decode": workloads.SMALL_CONFIGS["bf16_decode"],
    "bf16_top1": workloads.SMALL_CONFIGS["bf16_fine"].scaled("top1_T700_H392_E6_k1", T=700, H=392, I=264, E=6,
                                                             top_k=1, seed=4101),
    "f16_topE": workloads.SMALL_CONFIGS["f16_zipf"].scaled("topE_T90_H520_E12_k12", T=90, H=520, I=136, E=12,
                                                           top_k=12, renormalize=True, logits_kind="normal",
                                                           seed=4102),
    "bf16_all_on_two": workloads.SMALL_CONFIGS["bf16_fine"].scaled("k_eq_E_T3000_H512_E2_k2", T=3000, H=512, I=256,
                                                                   E=2, top_k=2, seed=4103),
    "bf16_top64": workloads.SMALL_CONFIGS["bf16_fine"].scaled("top64_T40_H264_I136_E64_k64", T=40, H=264, I=136,
                                                              E=64, top_k=64, seed=4106),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_forward_combine_equals_split(cuda_lib, name):
    """moe_experts_forward_combine and moe_forward both equal the unfused
    split path bit for bit, and the oracle within the output tolerance."""
    moe = cuda_lib
    cfg = CASES[name]
    inp = workloads.generate(cfg)
    d = _dev(inp)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    ref, idx, w, disp = _split_out(moe, ex, d, cfg)
    fused = moe.moe_experts_forward_combine(ex, disp.x_dispatched, disp.offsets, disp.inv, w)
    fwd = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert _same_bits(fused, ref), "fused combine differs from forward_dispatched + combine"
    assert _same_bits(fwd, ref), "moe_forward differs from the split path"
    oref = moe_oracle.forward(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], cfg.top_k,
                              cfg.renormalize)
    assert_output_close(f64(fused), oref.out, cfg.torch_dtype)
    assert moe.moe_device_status() == 0


def test_contract_rows_in_bf16(cuda_lib):
    """The routing-contract rows (two equal maxima, a NaN, a +inf, all -inf)
    on BF16 experts with H = 128 (one partial column block): NaN weights make
    whole rows NaN in the fused combine too."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[0].scaled("bf16_contract_T64_H128_I256_E8_k2", dtype="bf16", seed=4104)
    inp = workloads.generate(cfg)
    d = _dev(inp)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    ref, _, w, disp = _split_out(moe, ex, d, cfg)
    fused = moe.moe_experts_forward_combine(ex, disp.x_dispatched, disp.offsets, disp.inv, w)
    fwd = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert _same_bits(fused, ref) and _same_bits(fwd, ref)
    got = f64(fused)
    assert np.isnan(got[1:4]).all() and not np.isnan(got[0]).any() and not np.isnan(got[4:]).any()
    oref = moe_oracle.forward(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], cfg.top_k,
                              cfg.renormalize)
    assert_output_close(got, oref.out, cfg.torch_dtype)


def test_fp32_weights_with_bf16_experts(cuda_lib):
    """FP32 logits (so FP32 routing weights) with BF16 experts: the fused
    epilogue reads the weights in their own dtype."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_fine"]
    inp = workloads.generate(cfg)
    d = _dev(inp)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    lg32 = d["logits"].float()
    ref, _, w, disp = _split_out(moe, ex, d, cfg, logits=lg32)
    assert w.dtype == torch.float32
    fused = moe.moe_experts_forward_combine(ex, disp.x_dispatched, disp.offsets, disp.inv, w)
    fwd = moe.moe_forward(ex, d["x"], lg32, cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert _same_bits(fused, ref) and _same_bits(fwd, ref)


@pytest.mark.parametrize("cfg_id", [1, 2, 4])
def test_fused_combine_deterministic_full_size(cuda_lib, cfg_id):
    """Full-size prefill workloads (fine-grained, coarse, Zipf-skewed): the
    fused call three times in a row (one workspace), and moe_forward, give
    the same bits as the unfused split path."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[cfg_id]
    d = _dev(workloads.generate(cfg))
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    ref, idx, w, disp = _split_out(moe, ex, d, cfg)
    need = moe.load_library().moe_experts_forward_combine_workspace_size(ex.handle, cfg.T, cfg.top_k)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    for _ in range(3):
        fused = moe.moe_experts_forward_combine(ex, disp.x_dispatched, disp.offsets, disp.inv, w, workspace=ws)
        torch.cuda.synchronize()
        assert _same_bits(fused, ref)
    out = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert _same_bits(out, ref)
    assert moe.moe_device_status() == 0


def test_top_k_above_64_is_refused_by_the_fused_call(cuda_lib):
    """top_k = 300 of E = 320: moe_forward equals the split path and the
    oracle; the fused call refuses (its staging holds top_k <= 64)."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_fine"].scaled("topk300_T6_H64_I64_E320_k300", T=6, H=64, I=64, E=320,
                                                      top_k=300, seed=4105)
    inp = workloads.generate(cfg)
    d = _dev(inp)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    ref, _, w, disp = _split_out(moe, ex, d, cfg)
    fwd = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert _same_bits(fwd, ref)
    oref = moe_oracle.forward(inp["x"], inp["logits"], inp["gate"], inp["up"], inp["down"], cfg.top_k,
                              cfg.renormalize)
    assert_output_close(f64(fwd), oref.out, cfg.torch_dtype)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_experts_forward_combine(ex, disp.x_dispatched, disp.offsets, disp.inv, w)
    assert err.value.status == 7


def test_forward_combine_rejects_bad_arguments(cuda_lib):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_ragged"]
    d = _dev(workloads.generate(cfg))
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, w = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    lib = moe.load_library()
    need = lib.moe_experts_forward_combine_workspace_size(ex.handle, cfg.T, cfg.top_k)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_experts_forward_combine(ex, disp.x_dispatched, disp.offsets, disp.inv, w, workspace=small)
    assert err.value.status == 6
    f32 = workloads.SMALL_CONFIGS["f32_ragged"]
    d32 = _dev(workloads.generate(f32))
    ex32 = moe.Experts(d32["gate"], d32["up"], d32["down"])
    i32, w32 = moe.moe_route(d32["logits"], f32.top_k, f32.renormalize)
    disp32 = moe.moe_dispatch(i32, f32.E, d32["x"])
    with pytest.raises(moe.MoeError) as err:
        moe.moe_experts_forward_combine(ex32, disp32.x_dispatched, disp32.offsets, disp32.inv, w32)
    assert err.value.status == 7
