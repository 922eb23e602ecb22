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
    cfg = bench.workload_config(bench.PREFILL, 4)
    assert cfg["tokens_per_gpu"] == 4096 and cfg["global_batch_tokens"] == 4 * 4096
    assert cfg["workload"] == bench.PREFILL.name and "l2" in cfg


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_peaks_have_all_keys():
    peaks, src = bench.load_peaks()
    assert set(peaks) == {"hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"} and src in ("measured", "fallback")
