"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each a replica with
its own step time; the job time is the slowest rank's and the job throughput
counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 0: prefill 30 ms, decode 0.30 ms; rank 1: prefill 31 ms, decode 0.25 ms
        mine = [30.0 + rank, 0.30 - 0.05 * rank, 30.30 + 0.95 * rank]
        got = bench.reduce_max_over_ranks(mine, world, "cpu")
        out.put((rank, got, bench.job_tokens_per_s(world, 131072, got[0])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == pytest.approx([31.0, 0.30, 31.25])
        assert value == pytest.approx(2 * 131072 / 0.031)


def test_single_rank_passes_values_through():
    assert bench.reduce_max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]
    assert bench.job_tokens_per_s(1, 1000, 2.0) == pytest.approx(500000.0)


def test_tensor_peak_follows_the_clock_record():
    """The indexer's roofline denominator: the burst bf16 peak while the sampled
    clocks show no power cap, the sustained one when they do."""
    pk = {"bf16_tflops": 1755.6, "bf16_tflops_sustained": 1373.1}
    assert bench.tensor_peak_for({"reasons": []}, pk) == (1755.6, "burst")
    assert bench.tensor_peak_for({"reasons": ["sw_power_cap"]}, pk) == (1373.1, "sustained")
    assert bench.tensor_peak_for({"reasons": ["nvidia-smi unavailable"]}, pk) == (1755.6, "burst")
