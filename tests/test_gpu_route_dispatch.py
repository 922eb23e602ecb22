"""moe_route_dispatch — routing and dispatch as one cooperative launch (the
launch moe_forward runs) — against moe_route followed by moe_dispatch bit
for bit, and against the oracle's routing and dispatch.

The cases aim at the fused launch's own logic: one block (T <= 32), one token
per block (T just above 32), exactly one full round per block and one token
more (two rounds, the second almost empty), many rounds per block (T = 70000),
expert counts from 1 to 1024 with their block shapes (32, 16 and 8 warps),
top_k = E, rows of non-finite logits, quantised ties, F32 logits with BF16 x,
x rows that are not a multiple of 16 bytes, no x at all (maps only), the
full-size workloads, and moe_forward captured in a CUDA graph and replayed
(the barrier counter is zeroed on the stream every call)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle
from tests.parity import assert_route_matches, u32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    return t.contiguous().view(torch.uint8)


def _same(a, b):
    if a is None or b is None:
        return a is None and b is None
    return torch.equal(_bits(a), _bits(b))


def _compare(moe, logits, k, renorm, x, E):
    """Fused launch vs the split calls (bit for bit), then vs the oracle."""
    idx_s, w_s, w32_s = moe.moe_route(logits, k, renorm, weights_fp32=True)
    disp_s = moe.moe_dispatch(idx_s, E, x)
    idx_f, w_f, w32_f, disp_f = moe.moe_route_dispatch(logits, k, renorm, x, weights_fp32=True)
    torch.cuda.synchronize()
    n = int(disp_s.offsets[-1])
    assert _same(idx_f, idx_s) and _same(w_f, w_s) and _same(w32_f, w32_s), "routing outputs differ"
    assert _same(disp_f.counts, disp_s.counts) and _same(disp_f.offsets, disp_s.offsets)
    assert _same(disp_f.row_src[:n], disp_s.row_src[:n]) and _same(disp_f.inv, disp_s.inv)
    assert _same(disp_f.x_dispatched, disp_s.x_dispatched), "x_dispatched differs"
    ref = moe_oracle.route(logits.cpu(), k, renorm)
    assert_route_matches(idx_f, w_f, w32_f, ref, logits.dtype)
    rd = moe_oracle.dispatch(ref.indices, E)
    assert np.array_equal(u32(disp_f.counts), rd.counts)
    assert np.array_equal(u32(disp_f.offsets), rd.offsets)
    assert np.array_equal(u32(disp_f.row_src)[:n], rd.row_src)
    assert np.array_equal(u32(disp_f.inv), rd.inv)
    if x is not None:
        src = torch.from_numpy(rd.row_src.astype(np.int64) // k)
        assert torch.equal(_bits(disp_f.x_dispatched.cpu()), _bits(x.cpu()[src]))
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("name", sorted(workloads.SMALL_CONFIGS))
def test_small_workloads(cuda_lib, name):
    cfg = workloads.SMALL_CONFIGS[name]
    inp = workloads.generate(cfg)
    _compare(cuda_lib, inp["logits"].to(DEV), cfg.top_k, cfg.renormalize, inp["x"].to(DEV), cfg.E)


# (T, E, k): one block, one token per block, a full round per block and one
# token more, many rounds per block; E across the 32-, 16- and 8-warp shapes.
SHAPES = [(1, 8, 2), (17, 128, 8), (32, 128, 8), (33, 128, 8), (151, 64, 4), (4864, 128, 8), (4865, 128, 8),
          (9000, 32, 32), (70000, 8, 2), (3000, 256, 8), (1500, 512, 16), (700, 1024, 8), (400, 1000, 1000),
          (257, 1, 1)]


@pytest.mark.parametrize("T,E,k", SHAPES)
def test_block_shapes(cuda_lib, T, E, k):
    g = torch.Generator().manual_seed(T * 7 + E * 131 + k)
    logits = torch.randn(T, E, generator=g).to(torch.bfloat16)
    H = 64 if E * k <= 16000 else 16
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    _compare(cuda_lib, logits.to(DEV), k, True, x.to(DEV), E)


def test_many_rounds_per_block(cuda_lib):
    """T = 131072 (862 tokens a block, 27 rounds of 32 warps), E = 128, top_k
    = 8: a million slots, block histograms in the thousands."""
    g = torch.Generator().manual_seed(77)
    T, E, k = 131072, 128, 8
    logits = torch.randn(T, E, generator=g).to(torch.bfloat16)
    x = torch.randn(T, 64, generator=g).to(torch.bfloat16)
    _compare(cuda_lib, logits.to(DEV), k, True, x.to(DEV), E)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("E,k,renorm", [(1, 1, True), (3, 3, False), (33, 5, True), (64, 64, True),
                                        (1000, 7, False), (1024, 1, True)])
def test_contract_rows(cuda_lib, dtype, E, k, renorm):
    """Quantised ties, -inf entries, a NaN row, a +inf entry, an all -inf row."""
    g = torch.Generator().manual_seed(E * 131 + k + 7)
    T = 157
    l = torch.round(torch.randn(T, E, generator=g) * 4) / 4
    l[torch.rand(T, E, generator=g) < 0.1] = float("-inf")
    l[5] = float("nan") if E > 1 else l[5]
    l[6, 0] = float("inf")
    l[7] = float("-inf")
    x = torch.randn(T, 40, generator=g).to(dtype)
    _compare(cuda_lib, l.to(dtype).to(DEV), k, renorm, x.to(DEV), E)


@pytest.mark.parametrize("xdtype,H", [(torch.float32, 5), (torch.bfloat16, 12), (torch.float16, 8),
                                      (torch.float32, 4)])
def test_unaligned_rows_and_mixed_dtypes(cuda_lib, xdtype, H):
    """x rows of 20, 24, 16 and 16 bytes; F32 logits with 16-bit x and
    16-bit logits with F32 x."""
    g = torch.Generator().manual_seed(H * 11)
    T, E, k = 300, 48, 6
    ldt = torch.float32 if xdtype != torch.float32 else torch.bfloat16
    logits = torch.randn(T, E, generator=g).to(ldt)
    x = torch.randn(T, H, generator=g).to(xdtype)
    _compare(cuda_lib, logits.to(DEV), k, False, x.to(DEV), E)


def test_maps_only(cuda_lib):
    g = torch.Generator().manual_seed(5)
    logits = torch.randn(16, 128, generator=g).to(torch.bfloat16)
    _compare(cuda_lib, logits.to(DEV), 8, True, None, 128)


def test_empty_batch(cuda_lib):
    moe = cuda_lib
    logits = torch.empty(0, 16, dtype=torch.bfloat16, device=DEV)
    idx, w, disp = moe.moe_route_dispatch(logits, 4, True, None)
    torch.cuda.synchronize()
    assert idx.numel() == 0 and int(disp.counts.abs().sum()) == 0 and int(disp.offsets.abs().sum()) == 0


@pytest.mark.parametrize("cfg_id", [1, 2, 3, 4])
def test_full_size_workloads(cuda_lib, cfg_id):
    cfg = workloads.CONFIGS[cfg_id]
    inp = workloads.generate(cfg, weights=False)
    x = None if cfg.T * cfg.top_k <= 8 * cfg.E else inp["x"].to(DEV)
    _compare(cuda_lib, inp["logits"].to(DEV), cfg.top_k, cfg.renormalize, x, cfg.E)


def test_rejects_bad_arguments(cuda_lib):
    moe = cuda_lib
    lib = moe.load_library()
    logits = torch.randn(64, 16, device=DEV).to(torch.bfloat16)
    need = lib.moe_route_dispatch_workspace_size(64, 16)
    assert need > 0
    with pytest.raises(moe.MoeError) as err:
        moe.moe_route_dispatch(logits, 4, True, None,
                               workspace=torch.empty(need - 256, dtype=torch.uint8, device=DEV))
    assert err.value.status == 6
    with pytest.raises(moe.MoeError) as err:
        moe.moe_route_dispatch(logits, 17, True, None)
    assert err.value.status == 4


@pytest.mark.parametrize("name", ["bf16_fine", "bf16_decode"])
def test_forward_in_a_cuda_graph(cuda_lib, name):
    """moe_forward captured once and replayed three times gives the eager
    call's bits each time (the fused launch's barrier counter is zeroed on
    the stream inside the graph)."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    d = {k: v.to(DEV) for k, v in workloads.generate(cfg).items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    ref = moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize)
    lib = moe.load_library()
    ws = torch.empty(lib.moe_forward_workspace_size(ex.handle, cfg.T, cfg.top_k), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe.moe_forward(ex, d["x"], d["logits"], cfg.top_k, cfg.renormalize, out=out, workspace=ws)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert _same(out, ref)
    assert moe.moe_device_status() == 0


# ---- the grouped, bias-corrected sigmoid routing in the same launch

GOpt = moe_oracle.GroupRoutingOptions


def _gopts(r):
    return GOpt(r.top_k, r.groups, r.selected_groups, r.group_top_two, r.renormalize, r.scale)


def _compare_grouped(moe, logits, bias, o, x, E):
    """moe_route_sigmoid_grouped_dispatch vs moe_route_sigmoid_grouped then
    moe_dispatch (bit for bit), then vs the oracle."""
    b = None if bias is None else bias.to(DEV)
    idx_s, w_s, w32_s = moe.moe_route_sigmoid_grouped(logits, b, o, weights_fp32=True)
    disp_s = moe.moe_dispatch(idx_s, E, x)
    idx_f, w_f, w32_f, disp_f = moe.moe_route_sigmoid_grouped_dispatch(logits, b, o, x, weights_fp32=True)
    torch.cuda.synchronize()
    n = int(disp_s.offsets[-1])
    assert _same(idx_f, idx_s) and _same(w_f, w_s) and _same(w32_f, w32_s), "routing outputs differ"
    assert _same(disp_f.counts, disp_s.counts) and _same(disp_f.offsets, disp_s.offsets)
    assert _same(disp_f.row_src[:n], disp_s.row_src[:n]) and _same(disp_f.inv, disp_s.inv)
    assert _same(disp_f.x_dispatched, disp_s.x_dispatched), "x_dispatched differs"
    ref = moe_oracle.route_sigmoid_grouped(logits.cpu(), bias, o)
    assert_route_matches(idx_f, w_f, w32_f, ref, logits.dtype)
    rd = moe_oracle.dispatch(ref.indices, E)
    assert np.array_equal(u32(disp_f.counts), rd.counts)
    assert np.array_equal(u32(disp_f.row_src)[:n], rd.row_src)
    assert np.array_equal(u32(disp_f.inv), rd.inv)
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("name", sorted(workloads.GROUPED))
def test_grouped_workloads(cuda_lib, name):
    cfg, r = workloads.GROUPED[name]
    inp = workloads.generate(cfg, weights=False)
    x = None if cfg.T * r.top_k <= 8 * cfg.E else inp["x"].to(DEV)
    _compare_grouped(cuda_lib, inp["logits"].to(DEV), workloads.grouped_bias(cfg.E, r), _gopts(r), x, cfg.E)


# (T, E, groups, selected, top_k, top_two): one block, one token per block,
# a full round and one token more, many rounds; top_k past 32 (the second
# slot register); the largest E.
GSHAPES = [(1, 16, 4, 2, 4, True), (33, 64, 8, 3, 6, True), (4865, 128, 8, 4, 8, True), (70000, 8, 2, 1, 2, False),
           (600, 256, 8, 4, 40, True), (300, 1024, 128, 128, 64, True), (157, 1024, 1, 1, 64, False)]


@pytest.mark.parametrize("T,E,groups,sel,k,top_two", GSHAPES)
def test_grouped_block_shapes(cuda_lib, T, E, groups, sel, k, top_two):
    g = torch.Generator().manual_seed(T + E * 3 + k)
    logits = torch.randn(T, E, generator=g).to(torch.bfloat16)
    bias = (torch.randn(E, generator=g) * 0.02).float()
    H = 64 if T * k <= 400000 else 16
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    _compare_grouped(cuda_lib, logits.to(DEV), bias, GOpt(k, groups, sel, top_two, True, 2.5), x.to(DEV), E)


def test_grouped_contract_rows(cuda_lib):
    """Quantised ties, +-inf logits, a NaN row; then a NaN bias (every row NaN)."""
    g = torch.Generator().manual_seed(13)
    T, E = 157, 96
    l = torch.round(torch.randn(T, E, generator=g) * 4) / 4
    l[torch.rand(T, E, generator=g) < 0.05] = float("-inf")
    l[torch.rand(T, E, generator=g) < 0.02] = float("inf")
    l[5, 40] = float("nan")
    b = torch.round(torch.randn(E, generator=g) * 4) / 256
    x = torch.randn(T, 24, generator=g).to(torch.float32)
    _compare_grouped(cuda_lib, l.to(DEV), b.float(), GOpt(10, 32, 5, True, False, 1.0), x.to(DEV), E)
    b[3] = float("nan")
    _compare_grouped(cuda_lib, l.to(DEV), b.float(), GOpt(10, 32, 5, True, True, 1.0), x.to(DEV), E)


@pytest.mark.parametrize("name", ["bf16_fine_grouped", "f16_zipf_grouped", "bf16_decode_grouped"])
def test_grouped_forward_equals_split_calls(cuda_lib, name):
    """moe_forward_sigmoid_grouped (routing and dispatch in one launch) gives
    the bits of the split calls: grouped routing, dispatch, experts, combine."""
    moe = cuda_lib
    cfg, r = workloads.GROUPED[name]
    d = {k: v.to(DEV) for k, v in workloads.generate(cfg).items()}
    bias = workloads.grouped_bias(cfg.E, r)
    b = None if bias is None else bias.to(DEV)
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    o = _gopts(r)
    out = moe.moe_forward_sigmoid_grouped(ex, d["x"], d["logits"], b, o)
    idx, w = moe.moe_route_sigmoid_grouped(d["logits"], b, o)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    y = moe.moe_experts_forward_dispatched(ex, disp.x_dispatched, disp.offsets)
    ref = moe.moe_combine(y, disp.inv, w)
    torch.cuda.synchronize()
    assert _same(out, ref)
    assert moe.moe_device_status() == 0
