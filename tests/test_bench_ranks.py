"""The benchmark's multi-rank logic on the CPU (gloo, two ranks): rank
discovery from the launcher's environment and the max-over-ranks time that
the whole-job throughput divides by."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    ws, r, local = bench.dist_info()
    dist.init_process_group("gloo", rank=r, world_size=ws)
    # rank r "took" 10 + r ms and its end-to-end pass 5 - r s
    mx = bench.max_over_ranks([10.0 + r, 5.0 - r], "cpu")
    dist.barrier()
    dist.destroy_process_group()
    out.put((r, ws, local, mx))


def test_two_ranks_max_over_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, ws, local, mx) in enumerate(res):
        assert (rank, ws, local) == (r, world, r)
        assert mx == [11.0, 5.0]   # every rank sees the slowest rank's time


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
