"""The benchmark's N > 1 path on CPU: world-size-2 gloo ranks (no GPU).  Each
rank is an independent replica; the harness takes the slowest rank's timed
region and divides the work of all ranks by it."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    kernel_s, e2e_s = bench.max_over_ranks(times[rank], "cpu")
    value = bench.job_tflops(world, 10 ** 12, 5, kernel_s)
    assert bench.dist_setup() == (world, rank, rank)
    dist.barrier()
    dist.destroy_process_group()
    out_q.put((rank, kernel_s, e2e_s, value))


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [[0.5, 2.0], [1.0, 1.5]]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, kernel_s, e2e_s, value in results:
        assert kernel_s == 1.0 and e2e_s == 2.0     # slowest rank per quantity
        assert value == pytest.approx(2 * 5 * 1.0)  # 2 ranks x 5 steps x 1 TFLOP / 1 s
