"""The multi-rank harness of bench.py on CPU: two gloo ranks combine their
timings by the maximum and their verified tokens by the sum, and every rank
draws its own batch.  No GPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import CONFIGS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        span, tokens = bench.reduce_over_ranks(10.0 + 5.0 * rank, 100 + rank, world, torch.device("cpu"))
        cfg = bench.rank_config(CONFIGS["c3"], rank, world)
        dist.barrier()
        out[rank] = (span, tokens, cfg.seed)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_time_and_sum_tokens():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][:2] == res[1][:2] == (15.0, 201.0)
    assert res[0][2] != res[1][2]  # weak scaling: a different batch per rank


def test_single_rank_is_the_identity():
    assert bench.reduce_over_ranks(7.5, 42, 1, torch.device("cpu")) == (7.5, 42.0)
    assert bench.rank_config(CONFIGS["c3"], 0, 1) is CONFIGS["c3"]


def test_reference_arm_runs_on_rank_zero_only():
    from types import SimpleNamespace
    args = SimpleNamespace(steps=1, warmup=1, q=None)
    assert bench.run_reference(args, CONFIGS["c1"], "sample", 1, 2) is None
    line = bench.run_reference(args, CONFIGS["c1"], "sample", 0, 1)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True
    # the same config dict as the GPU arm prints for this workload
    assert line["config"] == bench.config_dict(CONFIGS["c1"], "sample", "logits", 1)
    assert line["cpu_baseline"]["host"]["nproc"] >= 1
