"""The bench's multi-GPU path on CPU ranks (gloo, world size 2).

The decode path shards as independent replicas: no collective touches the
data; the only exchange is the host's all-reduce MAX of the ranks' step
times, after which rank 0 reports the whole job's throughput.  The reference
arm runs on rank 0 alone.
"""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 + 5.0 * rank  # rank 1 is the slower replica
        ms, tps = bench.combine_ranks(ms_local, world, dist, "cpu")
        out[rank] = (ms, tps)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step_and_sum_the_tokens():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, tps = out[r]
        assert ms == 15.0, "the job's step is the slowest rank's"
        assert tps == pytest.approx(bench.T_TOKENS * world / 15e-3), "whole-job tokens across both replicas"


def test_single_rank_is_unchanged():
    ms, tps = bench.combine_ranks(12.5, 1)
    assert ms == 12.5 and tps == pytest.approx(bench.T_TOKENS / 12.5e-3)


def test_reference_arm_runs_on_rank_0_only(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, ref_tokens, gpus = 1, 0, 2, 2

    bench.run_reference(A())
    assert capsys.readouterr().out == "", "a non-zero rank prints nothing and does no work"


def test_reference_arm_line(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "0")

    class A:
        steps, warmup, ref_tokens, gpus = 1, 0, 2, 1

    bench.run_reference(A())
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == "gsi_linear_tokens_per_s_batch1"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
