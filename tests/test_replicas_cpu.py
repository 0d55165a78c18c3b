"""The multi-GPU mode of the bench (replicas only: the layer has no exchange
step) on two CPU ranks with the gloo backend: every rank draws different layers
and tokens, the job time is the slowest rank's, and the whole-job time per
layer counts the layers of all ranks."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slow = bench.max_over_ranks(1.5 + 2.0 * rank, world, "cpu")  # rank 1 is the slow one
    seed = bench.replica_seed(7, rank)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slow, seed))


def test_two_replicas_share_the_slowest_time_and_draw_different_layers():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.5, 3.5]
    assert res[0][2] != res[1][2]


def test_job_time_per_layer_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_us_per_layer(10.0, 1000, 1) == 10.0
    assert bench.job_us_per_layer(10.0, 1000, 2) == 5.0
