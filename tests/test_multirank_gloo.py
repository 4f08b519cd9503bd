"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each an
independent replica, agree on the job time (max over ranks) and report the
whole-job throughput (sum over replicas)."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    job_ms = bench.job_max(local_ms, dist, "cpu")
    q.put((r, ws, local, job_ms, bench.job_throughput(ws, 1000, job_ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_sum():
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
    for r, (rank, ws, local, job_ms, tput) in enumerate(res):
        assert (rank, ws, local) == (r, 2, r)
        assert job_ms == 15.0
        assert abs(tput - 2 * 1000 / 0.015) < 1e-6


def test_single_process_identity():
    assert bench.job_max(3.5, None, "cpu") == 3.5
    assert bench.job_throughput(1, 58465, 1.0) == 58465000.0
