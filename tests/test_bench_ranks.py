"""Host-side multi-rank logic of bench.py (replicas only): the max-over-ranks
timing and the whole-job token count, exercised with world_size 2 on gloo."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        elapsed = [0.25, 0.75][rank]                 # rank 1 is the straggler
        t = bench.reduce_max(elapsed)
        out[rank] = (t, bench.job_tokens_per_s(world, 1, 65536, t / 5))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        t, v = res[rank]
        assert t == 0.75                              # every rank sees the slowest rank's time
        assert abs(v - 2 * 65536 / 0.15) < 1e-6       # both replicas' tokens over that time


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(1.5) == 1.5
    assert bench.job_tokens_per_s(1, 1, 8192, 0.5) == 16384
