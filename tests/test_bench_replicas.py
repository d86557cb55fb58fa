"""Host logic of bench.py's multi-GPU mode on CPU: world size 2 over gloo.

Every rank runs an independent replica of the selection (there is no
data-path collective); the job's time is the slowest rank's, taken with an
all-reduce MAX, and the reported throughput counts the elements of all
ranks.  Here two CPU processes stand in for the ranks.
"""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        ms = bench.max_over_ranks(1.0 + 2.0 * rank, torch.device("cpu"), w)   # rank 1 is the slow one
        dist.barrier()
        out.put((r, w, lr, ms, bench.whole_job_gelems(1 << 20, w, ms)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_elements():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 and r[2] == r[0] for r in res)
    assert all(r[3] == 3.0 for r in res)                      # max(1 ms, 3 ms) on both ranks
    want = 2 * (1 << 20) / 3e-3 / 1e9                          # both ranks' elements over the slowest time
    assert all(abs(r[4] - want) < 1e-12 for r in res)


def test_one_rank_is_a_noop():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, None, 1) == 2.5
    assert abs(bench.whole_job_gelems(1 << 28, 1, 0.1864) - 1440.1) < 0.1
