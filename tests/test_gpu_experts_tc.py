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
