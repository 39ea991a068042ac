"""The multi-GPU path of bench.py is "replicas only": every rank decodes its own
copy of the workload with no collective on the data path; the job's time is the
slowest rank's and its throughput counts every rank's tokens. Its host-side
logic (rank environment, max-over-ranks reduction, job token count) runs here
as two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, l = bench.rank_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    # rank-specific timings: the reduction must give the maximum to every rank
    got = bench.max_over_ranks([10.0 + rank, 5.0 - rank], w, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, (w, r, l), got, bench.job_tokens(w, 7, [100, 50])))


def test_two_gloo_ranks_reduce_to_the_slowest_and_count_every_replica():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, got, tokens in res:
        assert env == (2, rank, rank)
        assert got == [11.0, 5.0]               # max over ranks of each timing
        assert tokens == 2 * 7 * 150            # both replicas' context tokens


def test_single_rank_is_the_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1, None) == [3.0, 4.0]
    assert bench.job_tokens(1, 5, [10]) == 50
