"""Seeded synthetic inputs for the local MoE forward chain.

This module is shared by the tests, the benchmark and the oracle's callers. It
only draws random numbers and shapes them into the configurations below; it
holds none of the routing, dispatch, expert or combine arithmetic, so neither
the CUDA path nor the CPU oracle depends on the other through it.

Recipe (identical bytes for both sides):
  * one torch CPU ``Generator`` per configuration (seed ``1001 + i`` for
    configuration i, numbered from 0) draws the logits and x, in that order
    (token shard r > 0 of a data-parallel run: seed ``1001 + i + 7919 r``);
  * gate, up and down are drawn in fixed chunks of ``_CHUNK`` elements, each
    from its own generator seeded from (config seed, tensor id, chunk index),
    so the bytes do not depend on how many threads draw them;
  * every draw is FP32 standard normal, scaled, then rounded to the working
    dtype with round-to-nearest-even (torch's cast);
  * gate and up have std 1/sqrt(H) and down std 1/sqrt(I) ("N(0, 1/sqrt(fan_in))"
    read as a standard deviation); logits and x are N(0, 1).
Special logit rows (the F32 routing-contract workload) and the Zipf-skewed
expert bias with exact-tie rows (the F16 workload) are described at
``_contract_rows`` and ``_zipf_logits``.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

_CHUNK = 1 << 22


@dataclass(frozen=True)
class MoeConfig:
    """One MoE forward workload: T tokens, E experts, top_k, hidden H, intermediate I."""

    name: str
    dtype: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    renormalize: bool
    logits_kind: str = "normal"  # "normal" | "contract_rows" | "zipf"
    seed: int = 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.dtype]

    @property
    def rows(self) -> int:
        return self.T * self.top_k

    @property
    def expert_flops(self) -> int:
        """2*M*N*K summed over gate, up and down: 6*T*k*H*I."""
        return 6 * self.T * self.top_k * self.H * self.I

    def scaled(self, name: str, **kw) -> "MoeConfig":
        return replace(self, name=name, **kw)


# The five workloads of the local MoE forward chain, numbered from 0 in the
# order they are listed: 0 the F32 routing-contract case, 1 the fine-grained
# BF16 prefill, 2 the coarse BF16 prefill (the GEMM-bound case), 3 the BF16
# decode, 4 the Zipf-skewed F16 prefill.
CONFIGS = {
    0: MoeConfig("f32_routing_contract_T64_H128_I256_E8_k2", "f32", 64, 128, 256, 8, 2, True,
                 "contract_rows", 1001),
    1: MoeConfig("bf16_prefill_T4096_H2048_I768_E128_k8", "bf16", 4096, 2048, 768, 128, 8, True,
                 "normal", 1002),
    2: MoeConfig("bf16_prefill_T8192_H4096_I14336_E8_k2", "bf16", 8192, 4096, 14336, 8, 2, True,
                 "normal", 1003),
    3: MoeConfig("bf16_decode_T16_H2048_I768_E128_k8", "bf16", 16, 2048, 768, 128, 8, True,
                 "normal", 1004),
    4: MoeConfig("f16_zipf_T16384_H2048_I1408_E64_k6", "f16", 16384, 2048, 1408, 64, 6, False,
                 "zipf", 1005),
}

# Reduced sizes of the same workloads: small enough for the full oracle in a few
# seconds, still several tiles in every dimension and ragged per-expert tails.
SMALL_CONFIGS = {
    "f32_contract": CONFIGS[0],
    "bf16_fine": CONFIGS[1].scaled("bf16_fine_small_T600_H512_I384_E24_k5", T=600, H=512, I=384,
                                   E=24, top_k=5, seed=2002),
    "bf16_coarse": CONFIGS[2].scaled("bf16_coarse_small_T520_H1024_I1280_E4_k2", T=520, H=1024,
                                     I=1280, E=4, top_k=2, seed=2003),
    "bf16_decode": CONFIGS[3],
    "f16_zipf": CONFIGS[4].scaled("f16_zipf_small_T1200_H512_I640_E16_k3", T=1200, H=512, I=640,
                                  E=16, top_k=3, seed=2005),
    "f32_ragged": CONFIGS[0].scaled("f32_ragged_T333_H200_I136_E7_k3", T=333, H=200, I=136, E=7,
                                    top_k=3, logits_kind="normal", seed=2006),
    "bf16_ragged": CONFIGS[1].scaled("bf16_ragged_T77_H136_I200_E5_k2", T=77, H=136, I=200, E=5,
                                     top_k=2, seed=2007),
}


@dataclass(frozen=True)
class GroupedRouting:
    """Options of the group-limited sigmoid routing (ruDNN user guide,
    section 10) and the recipe of its FP32 correction bias: N(0, bias_std^2)
    from a torch Generator seeded with ``bias_seed`` (no bias if bias_std is 0)."""

    groups: int
    selected_groups: int
    top_k: int
    group_top_two: bool
    renormalize: bool
    scale: float
    bias_std: float
    bias_seed: int


# Grouped sigmoid routing on the shapes of the workloads above (the pages give
# no sizes for it): 8 groups of 16 experts, 4 selected, top-8, top-two group
# scores and a 2.5 scale on the fine-grained prefill and decode shapes, and
# smaller group layouts on the reduced workloads (one expert per group,
# one group of all experts, groups of 6 and of 4).
GROUPED = {
    "bf16_prefill_grouped": (CONFIGS[1], GroupedRouting(8, 4, 8, True, True, 2.5, 0.02, 3002)),
    "bf16_decode_grouped": (CONFIGS[3], GroupedRouting(8, 4, 8, True, True, 2.5, 0.02, 3004)),
    "bf16_fine_grouped": (SMALL_CONFIGS["bf16_fine"], GroupedRouting(4, 2, 5, True, True, 1.0, 0.05, 3012)),
    "f16_zipf_grouped": (SMALL_CONFIGS["f16_zipf"], GroupedRouting(4, 2, 3, False, False, 1.5, 0.1, 3015)),
    "f32_ragged_grouped": (SMALL_CONFIGS["f32_ragged"], GroupedRouting(7, 3, 3, False, True, 1.0, 0.1, 3016)),
    "bf16_ragged_grouped": (SMALL_CONFIGS["bf16_ragged"], GroupedRouting(1, 1, 2, True, False, 2.0, 0.0, 3017)),
}


def grouped_bias(E: int, r: GroupedRouting) -> torch.Tensor | None:
    """The FP32 [E] correction bias of a grouped-routing workload, or None."""
    if r.bias_std == 0:
        return None
    g = torch.Generator().manual_seed(r.bias_seed)
    return (torch.randn(E, generator=g) * r.bias_std).to(torch.float32)


def _chunk_seed(base: int, tensor_id: int, chunk: int) -> int:
    return (base * 1_000_003 + tensor_id * 10_007 + chunk) & 0x7FFF_FFFF_FFFF


def _draw_chunk(args):
    seed, n, std, dtype = args
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, generator=g) * std).to(dtype)


def _normal_chunked(n: int, std: float, dtype: torch.dtype, base: int, tensor_id: int,
                    threads: int | None = None) -> torch.Tensor:
    """n values of N(0, std^2) rounded to dtype, drawn in fixed seeded chunks."""
    jobs = [(_chunk_seed(base, tensor_id, c), min(_CHUNK, n - c * _CHUNK), std, dtype)
            for c in range((n + _CHUNK - 1) // _CHUNK)]
    if len(jobs) <= 1:
        parts = [_draw_chunk(j) for j in jobs]
    else:
        nthreads = threads or min(32, torch.get_num_threads() * 2, len(jobs))
        prev = torch.get_num_threads()
        torch.set_num_threads(1)
        try:
            with ThreadPoolExecutor(nthreads) as ex:
                parts = list(ex.map(_draw_chunk, jobs))
        finally:
            torch.set_num_threads(prev)
    return torch.cat(parts) if parts else torch.empty(0, dtype=dtype)


def _contract_rows(logits: torch.Tensor) -> torch.Tensor:
    """Four rows that exercise the routing contract (ruDNN user guide, section 4):
    row 0 gets two equal maxima at experts 1 and 6; row 1 holds one NaN (expert 2);
    row 2 holds one +inf (expert 5); row 3 is all -inf."""
    l = logits.clone()
    E = l.shape[1]
    if l.shape[0] >= 4 and E >= 7:
        top = l[0].max() + 1.0
        l[0, 1] = top
        l[0, 6] = top
        l[1, 2] = float("nan")
        l[2, 5] = float("inf")
        l[3, :] = float("-inf")
    return l


def _zipf_logits(logits: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """Skewed expert load: add 2*ln(p_e), p_e Zipf(s=1.2) over a seeded expert
    permutation (p_e = r_e^-1.2 / sum_r r^-1.2, r_e the expert's rank), then round
    1% of rows (seeded choice) to the nearest multiple of 0.25 so that the
    working dtype holds exact ties."""
    T, E = logits.shape
    perm = torch.randperm(E, generator=g)
    rank = torch.empty(E, dtype=torch.float64)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64)
    z = sum(r ** -1.2 for r in range(1, E + 1))
    bias = 2.0 * torch.log(rank.pow(-1.2) / z)
    l = logits.to(torch.float64) + bias[None, :]
    n_tie = max(1, (T + 50) // 100)
    rows = torch.randperm(T, generator=g)[:n_tie]
    l[rows] = torch.round(l[rows] * 4.0) / 4.0
    return l.to(torch.float32)


def token_seed(cfg: MoeConfig, shard: int = 0) -> int:
    """Seed of the logits and x of token shard ``shard`` (0: the workload's own
    batch). Shards of a data-parallel run draw distinct tokens; the expert
    weights are always drawn from the workload's seed (replicated experts)."""
    return cfg.seed + 7919 * shard


def generate(cfg: MoeConfig, device: str | torch.device = "cpu", weights: bool = True,
             pin: bool = False, shard: int = 0) -> dict:
    """Draw logits [T,E], x [T,H], gate/up [E,I,H] and down [E,H,I] in cfg.dtype.

    The tensors are created on the CPU and then moved to ``device``; ``pin``
    places the CPU copies of x and logits in pinned memory (for timed
    host-to-device copies). ``shard`` > 0 draws another batch of T tokens
    (logits and x) with the same expert weights; only plain N(0,1) logits
    have shards."""
    dt = cfg.torch_dtype
    if shard and cfg.logits_kind != "normal":
        raise ValueError("token shards are defined for N(0,1) logits only")
    g = torch.Generator().manual_seed(token_seed(cfg, shard))
    logits = torch.randn(cfg.T, cfg.E, generator=g)
    x = torch.randn(cfg.T, cfg.H, generator=g)
    if cfg.logits_kind == "contract_rows":
        logits = _contract_rows(logits)
    elif cfg.logits_kind == "zipf":
        logits = _zipf_logits(logits, g)
    out = {"logits": logits.to(dt), "x": x.to(dt)}
    if weights:
        sg, sd = 1.0 / math.sqrt(cfg.H), 1.0 / math.sqrt(cfg.I)
        n = cfg.E * cfg.I * cfg.H
        out["gate"] = _normal_chunked(n, sg, dt, cfg.seed, 1).view(cfg.E, cfg.I, cfg.H)
        out["up"] = _normal_chunked(n, sg, dt, cfg.seed, 2).view(cfg.E, cfg.I, cfg.H)
        out["down"] = _normal_chunked(n, sd, dt, cfg.seed, 3).view(cfg.E, cfg.H, cfg.I)
    if pin:
        for key in ("logits", "x"):
            out[key] = out[key].pin_memory()
    if str(device) != "cpu":
        out = {k: v.to(device, non_blocking=False) for k, v in out.items()}
    return out
