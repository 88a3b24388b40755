"""The benchmark's multi-rank plumbing on CPU: two gloo ranks rendezvous on
127.0.0.1, time with a barrier on both sides and take the maximum over ranks
(the path runs independent replicas per GPU, so no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + r, w)          # per-rank step time in ms
    # whole-job throughput: every rank's work over the slowest rank's time
    value = 1000.0 * w / (slowest * 1e-3) / 1e9
    bench.barrier(w)
    q.put((r, w, slowest, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for _, w, slowest, value in out:
        assert w == 2
        assert slowest == pytest.approx(2.5)
        assert value == pytest.approx(2 * 1000.0 / 2.5e-3 / 1e9)
