"""The benchmark's multi-process path on CPU: two gloo ranks, as torchrun
launches them (one replica per GPU, no data-path collective).  Only the host
logic runs here: the max-over-ranks step time, the aggregate rate, and the
reference arm's rank rule (rank 0 alone runs the oracle)."""

import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(values[rank], world, torch.device("cpu"))
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    values = [3.25, 7.5]
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, values, out), nprocs=world, join=True)
    assert out[0] == out[1] == max(values)


def test_aggregate_rate_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    ms = 0.152
    one = bench.aggregate_us_per_token_layer(ms, 1)
    two = bench.aggregate_us_per_token_layer(ms, 2)
    assert one == pytest.approx(ms * 1000 / bench.LAYERS)
    assert two == pytest.approx(one / 2)


def test_reference_arm_runs_on_rank_zero_only():
    """A non-zero rank of `bench.py --impl reference` exits 0 without work or
    output (no GPU, no oracle run)."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
