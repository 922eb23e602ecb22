"""Host-side logic of bench.py on the CPU: the max-over-ranks timing with two
gloo ranks (the multi-GPU run shards tokens with no data-path collective;
only the timing is reduced), the JSON config and argument checks."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(1.5 + rank * 2.25, world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 3.75, 1: 3.75}


def test_single_rank_max_is_identity():
    assert bench.max_over_ranks(0.25, 1) == 0.25


def test_workload_config_is_weak_scaling():
    cfg = bench.workload_config(bench.HEADLINE, 4)
    assert cfg["tokens_per_gpu"] == 8192 and cfg["global_batch_tokens"] == 4 * 8192
    assert cfg["workload"] == bench.HEADLINE.name and "l2" in cfg
    assert cfg["parallelism"].startswith("dp4")


def test_headline_is_the_coarse_prefill():
    """The headline workload is the GEMM-bound coarse BF16 prefill (T=8192,
    H=4096, I=14336, E=8, top_k=2), the largest configuration on one GPU."""
    c = bench.HEADLINE
    assert (c.dtype, c.T, c.H, c.I, c.E, c.top_k, c.renormalize) == ("bf16", 8192, 4096, 14336, 8, 2, True)
    assert c.expert_flops == max(w.expert_flops for w in bench.workloads.CONFIGS.values())


def test_roofline_counts_the_methods_bytes():
    """Algorithmic bytes are the touched weights plus x in and out; the
    fraction follows from them and the peak."""
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}
    c = bench.HEADLINE
    r = bench.gemm_roofline(c, 3e-3, 8, peaks, "test", {"dram_bytes_per_launch": 4.0e9}, "t")
    want_bytes = 8 * 3 * c.I * c.H * 2 + 2 * c.T * c.H * 2
    assert r["algorithmic_bytes"] == want_bytes and r["bound"] == "tensor"
    assert abs(r["frac"] - c.expert_flops / 3e-3 / 1e12 / 1800.0) < 1e-4   # the sustained peak
    assert abs(r["tensor_frac"] - c.expert_flops / 3e-3 / 1e12 / 2000.0) < 1e-4
    assert abs(r["traffic_over_algorithmic"] - 4.0e9 / want_bytes) < 1e-4
    f = bench.FINE
    r = bench.gemm_roofline(f, 300e-6, 128, peaks, "test", None, "t")
    assert r["bound"] == "hbm" and r["traffic"] is None


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_peaks_have_all_keys():
    peaks, src = bench.load_peaks()
    assert set(peaks) == {"hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"} and src in ("measured", "fallback")
