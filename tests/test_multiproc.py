"""The replica (N > 1) host logic of bench.py on CPU: world size 2 over gloo."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms_local = [2.0, 3.0][rank]            # rank 1 is the slower replica
    ms, tflops = bench.replica_throughput(ms_local, flops_per_rank=6 * 10**12, world=world, device="cpu")
    q.put((rank, ms, tflops))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, tflops in got:
        assert ms == 3.0
        assert abs(tflops - 2 * 6 / 3e-3 / 1e12 * 1e12) < 1e-9 * tflops  # 2 ranks x 6 TFLOP / 3 ms


def test_single_replica_is_plain_throughput():
    import bench

    ms, tflops = bench.replica_throughput(4.0, 8 * 10**12, 1)
    assert ms == 4.0 and abs(tflops - 2000.0) < 1e-9
