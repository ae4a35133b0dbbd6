"""Multi-process host logic of bench.py on CPU (gloo, world size 2): every
rank runs an independent replica; the job's time is the slowest rank's and
its bytes are the sum over ranks."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t, u = bench.aggregate(elapsed_s=1.0 + rank, units=100.0 * (rank + 1))
    bench.barrier()
    q.put((rank, t, u, bench.dist_env()))
    dist.destroy_process_group()


def test_aggregate_max_time_sum_units_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u, env in out:
        assert t == 2.0 and u == 300.0
        assert env[0] == 2 and env[1] == rank


def test_aggregate_single_process_is_identity():
    import bench
    assert bench.aggregate(0.5, 7.0) == (0.5, 7.0)


def test_reference_arm_only_rank0_prints(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 3, 3
    assert bench.run_reference(A()) is None
