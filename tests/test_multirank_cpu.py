"""The benchmark's multi-rank path on CPU: two gloo ranks, max-over-ranks timing and
weak-scaling throughput (every rank runs its own independent sequences)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]                       # per-rank step times
    m = bench.max_over_ranks(ms, world)
    v = bench.weak_scaling_value(1000, world, m)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        m, v = res[rank]
        assert m == 5.0
        assert v == pytest.approx(2 * 1000 / 5e-3)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.weak_scaling_value(500, 1, 2.0) == pytest.approx(250000.0)
