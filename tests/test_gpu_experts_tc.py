"""GPU parity of the F16/BF16 SwiGLU experts (tcgen05 grouped GEMMs) against
the f64 oracle, on dispatched rows prepared by the oracle."""
import numpy as np
import pytest
import torch

import workloads
from oracle import moe_oracle
from tests.parity import assert_output_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL_16 = ["bf16_ragged", "bf16_fine", "bf16_coarse", "f16_zipf", "bf16_decode"]


def _run_experts(moe, cfg, inp, dp):
    xd = inp["x"][torch.from_numpy(dp.row_src.astype(np.int64) // cfg.top_k)]
    ex = moe.Experts(inp["gate"].to(DEV), inp["up"].to(DEV), inp["down"].to(DEV))
    offs = torch.from_numpy(dp.offsets.astype(np.int64)).to(torch.int32).to(DEV)
    y = moe.moe_experts_forward_dispatched(ex, xd.to(DEV).contiguous(), offs)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    return y


@pytest.mark.parametrize("name", SMALL_16)
def test_tc_experts_parity(cuda_lib, name):
    cfg = workloads.SMALL_CONFIGS[name]
    inp = workloads.generate(cfg)
    rt = moe_oracle.route(inp["logits"], cfg.top_k, cfg.renormalize)
    dp = moe_oracle.dispatch(rt.indices, cfg.E)
    y = _run_experts(cuda_lib, cfg, inp, dp)
    yref = moe_oracle.experts_forward_dispatched(inp["x"], inp["gate"], inp["up"], inp["down"], dp, cfg.top_k)
    assert_output_close(f64(y), yref, cfg.torch_dtype, "y_dispatched")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_tc_single_expert_and_empty_experts(cuda_lib, dtype):
    """All rows on one expert (one long expert, the rest empty), rows not a
    multiple of the 128-row tile."""
    cfg = workloads.SMALL_CONFIGS["bf16_fine"].scaled("one_hot", T=300, H=256, I=256, E=6, top_k=1,
                                                      seed=77, dtype="bf16" if dtype == torch.bfloat16 else "f16")
    inp = workloads.generate(cfg)
    idx = np.full((cfg.T, 1), 4, dtype=np.uint32)
    dp = moe_oracle.dispatch(idx, cfg.E)
    y = _run_experts(cuda_lib, cfg, inp, dp)
    yref = moe_oracle.experts_forward_dispatched(inp["x"], inp["gate"], inp["up"], inp["down"], dp, 1)
    assert_output_close(f64(y), yref, dtype, "y_dispatched")


def test_tc_identity_experts_closed_form(cuda_lib):
    """gate = up = down = I (BF16): y = SiLU(x) * x rounded through BF16 h."""
    moe = cuda_lib
    E, n, rows = 3, 128, 200
    eye = torch.eye(n).to(torch.bfloat16)
    w = eye.repeat(E, 1, 1).contiguous()
    x = (torch.randn(rows, n, generator=torch.Generator().manual_seed(5)) * 2).to(torch.bfloat16)
    offs = torch.tensor([0, 70, 70, rows], dtype=torch.int32)
    ex = moe.Experts(w.to(DEV), w.clone().to(DEV), w.clone().to(DEV))
    y = moe.moe_experts_forward_dispatched(ex, x.to(DEV), offs.to(DEV))
    torch.cuda.synchronize()
    xf = f64(x)
    assert_output_close(f64(y), xf * xf / (1 + np.exp(-xf)), torch.bfloat16, "identity experts")


def test_tc_decode_path_with_a_hot_expert(cuda_lib):
    """Few rows per expert on average (the 32-token-block path) while one
    expert holds about 75 rows (three token blocks) and most hold none."""
    cfg = workloads.SMALL_CONFIGS["bf16_fine"].scaled("hot_decode", T=100, H=256, I=384, E=64, top_k=2, seed=91)
    inp = workloads.generate(cfg)
    rng = np.random.default_rng(4)
    idx = np.stack([rng.permutation(64)[:2] for _ in range(cfg.T)]).astype(np.uint32)
    idx[:75, 0] = 3
    idx[:75, 1] = np.where(idx[:75, 1] == 3, 7, idx[:75, 1])
    dp = moe_oracle.dispatch(idx, cfg.E)
    assert dp.counts.max() > 32 and cfg.T * cfg.top_k <= 8 * cfg.E
    y = _run_experts(cuda_lib, cfg, inp, dp)
    yref = moe_oracle.experts_forward_dispatched(inp["x"], inp["gate"], inp["up"], inp["down"], dp, cfg.top_k)
    assert_output_close(f64(y), yref, torch.bfloat16, "y_dispatched")


@pytest.mark.parametrize("name", ["bf16_fine", "f16_zipf", "bf16_ragged", "bf16_decode", "f32_ragged"])
def test_gate_up_gather_equals_dense(cuda_lib, name):
    """The gathered gate/up stage (rows read from x through row_src) is
    bit-identical to the stage on the materialised x_dispatched, and h is
    the oracle's within the chain's tolerance."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS[name]
    inp = workloads.generate(cfg)
    d = {k: v.to(DEV) for k, v in inp.items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, _ = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    h_dense = moe.moe_experts_gate_up(ex, disp.x_dispatched, disp.offsets)
    h_gather = moe.moe_experts_gate_up_gather(ex, d["x"], disp.row_src, cfg.top_k, disp.offsets)
    torch.cuda.synchronize()
    assert torch.equal(h_dense.view(torch.uint8), h_gather.view(torch.uint8))
    assert moe.moe_device_status() == 0


def test_gate_up_gather_full_size(cuda_lib):
    """The fine-grained prefill workload at full size (the benchmark's launch
    configuration): gathered and dense gate/up stages agree bit for bit."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[1]
    d = {k: v.to(DEV) for k, v in workloads.generate(cfg).items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, _ = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    h_dense = moe.moe_experts_gate_up(ex, disp.x_dispatched, disp.offsets)
    for _ in range(2):
        h_gather = moe.moe_experts_gate_up_gather(ex, d["x"], disp.row_src, cfg.top_k, disp.offsets)
        torch.cuda.synchronize()
        assert torch.equal(h_dense.view(torch.uint8), h_gather.view(torch.uint8))
    assert moe.moe_device_status() == 0


def test_gate_up_gather_bad_row_src_reads_zero_rows(cuda_lib):
    """A row_src entry past T * top_k reads as a zero row: h = SiLU(0) * 0 = 0
    for that row, no out-of-range access."""
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_ragged"]
    d = {k: v.to(DEV) for k, v in workloads.generate(cfg).items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, _ = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    rs = disp.row_src.clone()
    rs[5] = 0x7FFFFFFF
    h = moe.moe_experts_gate_up_gather(ex, d["x"], rs, cfg.top_k, disp.offsets)
    ref = moe.moe_experts_gate_up(ex, disp.x_dispatched, disp.offsets)
    torch.cuda.synchronize()
    assert torch.count_nonzero(h[5]) == 0
    keep = torch.ones(h.shape[0], dtype=torch.bool, device=DEV)
    keep[5] = False
    assert torch.equal(h[keep].view(torch.uint8), ref[keep].view(torch.uint8))


def test_gate_up_gather_bad_rows_across_a_full_tile(cuda_lib):
    """Out-of-range row_src entries spread over a 256-row token block and the
    expert's next block (first and last rows, both sides of each 32-row
    boundary) each give a zero row; every other row matches the dense stage
    bit for bit (prefill workload, full size)."""
    moe = cuda_lib
    cfg = workloads.CONFIGS[1]
    d = {k: v.to(DEV) for k, v in workloads.generate(cfg).items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, _ = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E, d["x"])
    counts = disp.counts.cpu().numpy().astype(np.int64)
    e = int(np.argmax(counts))
    assert counts[e] > 256
    o = int(disp.offsets[e].item())
    local = [0, 3, 4, 31, 32, 63, 64, 127, 128, 129, 200, 255, 256, int(counts[e]) - 1]
    bad = torch.tensor([o + j for j in local], dtype=torch.int64, device=DEV)
    rs = disp.row_src.clone()
    rs[bad] = (-16 - torch.arange(len(local), device=DEV)).to(rs.dtype)  # 2^32 - 16 - j as uint32
    h = moe.moe_experts_gate_up_gather(ex, d["x"], rs, cfg.top_k, disp.offsets)
    ref = moe.moe_experts_gate_up(ex, disp.x_dispatched, disp.offsets)
    torch.cuda.synchronize()
    assert torch.count_nonzero(h[bad]) == 0
    keep = torch.ones(h.shape[0], dtype=torch.bool, device=DEV)
    keep[bad] = False
    assert torch.equal(h[keep].view(torch.uint8), ref[keep].view(torch.uint8))
    assert moe.moe_device_status() == 0


def test_gate_up_gather_rejects_bad_arguments(cuda_lib):
    moe = cuda_lib
    cfg = workloads.SMALL_CONFIGS["bf16_ragged"]
    d = {k: v.to(DEV) for k, v in workloads.generate(cfg).items()}
    ex = moe.Experts(d["gate"], d["up"], d["down"])
    idx, _ = moe.moe_route(d["logits"], cfg.top_k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, cfg.E)
    for kw, status in [(dict(top_k=0), 2), (dict(rows=cfg.T * cfg.top_k + 1), 2)]:
        a = dict(top_k=cfg.top_k, rows=None)
        a.update(kw)
        with pytest.raises(moe.MoeError) as err:
            moe.moe_experts_gate_up_gather(ex, d["x"], disp.row_src, a["top_k"], disp.offsets, rows=a["rows"],
                                           out=torch.empty(cfg.T * cfg.top_k + 1, cfg.I, dtype=cfg.torch_dtype,
                                                           device=DEV))
        assert err.value.status == status


@pytest.mark.parametrize("E,counts", [(2, None), (3, [3000, 0, 1096]), (1, None)])
def test_chained_launch_equals_the_two_launches_under_heavy_waiting(cuda_lib, E, counts):
    """moe_experts_forward_dispatched runs gate/up and down as one launch whose
    down tiles wait for their expert's h rows. With one to three long experts
    most CTAs claim down tiles while the gate/up tiles they depend on are
    still running: the waits (and the release/acquire of h across CTAs) are
    exercised on every launch. The result must be bit-identical, three times
    over, to the two GEMMs launched apart, and parity holds against the
    oracle on sampled rows."""
    moe = cuda_lib
    rows, H, I = 4096, 2048, 768
    g = torch.Generator().manual_seed(83 + E)
    gate = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    up = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    down = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(torch.bfloat16)
    x = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    if counts is None:
        counts = [rows // E] * E
        counts[-1] += rows - sum(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    ex = moe.Experts(gate.to(DEV), up.to(DEV), down.to(DEV))
    xd = x.to(DEV)
    offs = torch.from_numpy(offsets).to(torch.int32).to(DEV)
    h = moe.moe_experts_gate_up(ex, xd, offs)
    y_split = moe.moe_experts_down(ex, h, offs)
    for _ in range(3):
        y = moe.moe_experts_forward_dispatched(ex, xd, offs)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.uint8), y_split.view(torch.uint8))
    assert moe.moe_device_status() == 0
    # Oracle parity on a few rows of each expert.
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        r = np.unique(np.array([lo, (lo + hi) // 2, hi - 1]))
        xr = f64(x[r])
        gg = xr @ f64(gate[e]).T
        uu = xr @ f64(up[e]).T
        hh = gg / (1 + np.exp(-gg)) * uu
        yref = hh @ f64(down[e]).T
        assert_output_close(f64(y[torch.from_numpy(r).to(DEV)]), yref, torch.bfloat16, f"expert {e} rows")
