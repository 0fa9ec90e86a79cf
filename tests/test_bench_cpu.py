"""Host logic of bench.py: the FLOP count of the benchmark step and the
multi-rank aggregation (max over ranks, whole-job rate), the latter on two
CPU processes with the gloo backend."""
import os
import socket

import pytest

import bench
from cnn_conv3d_gb300 import flops


def test_step_flops_match_convention():
    ops = bench.op_table(8, 128, (4, 32, 64, 128, 256, 256))
    assert len(ops) == 5 + 5 + 4  # fwd, wgrad every block; dgrad for blocks 2..5
    total = sum(o[3] for o in ops)
    assert total == flops.stack_flops(8, 128, (4, 32, 64, 128, 256, 256), backward=True)
    assert abs(total / 1e9 - 1493.04) < 0.01
    # forward alone: 67.04 GFLOP per sample (conv FLOPs of the five blocks)
    fwd = sum(o[3] for o in ops if o[1] == "fwd")
    assert abs(fwd / 8 / 1e9 - 67.0418) < 1e-3


def test_whole_job_rate():
    assert bench.whole_job_rate(10.0, 1, 1000.0) == pytest.approx(10.0)
    assert bench.whole_job_rate(10.0, 4, 2000.0) == pytest.approx(20.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 3.0 + rank  # rank 1 is the slow one
        m = bench.max_over_ranks(ms, world)
        out[rank] = (m, bench.whole_job_rate(8, world, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_processes():
    import torch.multiprocessing as mp
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 4.0
    assert res[0][1] == pytest.approx(2 * 8 / 4e-3)


def test_host_step_sample_ranges():
    """The host-buffer step's input split: contiguous, non-empty, covering
    every sample once, at most `chunks` pieces whose sizes differ by <= 1."""
    from cnn_conv3d_gb300.stack import sample_ranges
    for n in range(1, 20):
        for chunks in range(1, 12):
            r = sample_ranges(n, chunks)
            assert 1 <= len(r) <= min(n, chunks)
            assert r[0][0] == 0 and r[-1][1] == n
            assert all(a < b for a, b in r)
            assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
            sizes = [b - a for a, b in r]
            assert max(sizes) - min(sizes) <= 1
