"""bench.py's multi-rank logic on CPU ranks (gloo, world size 2).

The path shards with no exchange step: every rank runs its own replica of the
workload (weak scaling), and the only process-group traffic is the barrier
around the timed region and the max-over-ranks reduction of the timed total.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)       # rank 1 is slower
        # replicas: each rank lays out its own batch from its own seed
        from radixattention_prefix_shared_gb300 import workloads as W
        wl = W.tiny(seed=1001 + 7919 * r)
        q.put((r, w, local, slowest, int(wl.req_to_token.sum()), float(wl.extend.q.astype("int64").sum())))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction_and_replicas():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0, f"rank process failed with {p.exitcode}"
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert all(x[3] == 15.0 for x in res), "every rank reports the slowest rank's time"
    assert res[0][4:] != res[1][4:], "replicas draw different inputs per rank"


def test_single_process_needs_no_process_group():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    bench.barrier()  # no-op without a process group
