"""The multi-rank host logic of bench.py on CPU: world size 2 over gloo."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(1.5 + rank, dist, "cpu")
    cfg = bench.workload_config("bs256_kv8192", world)
    q.put((rank, got, cfg["parallelism"]))
    dist.destroy_process_group()


def test_max_over_ranks_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [2.5, 2.5]
    assert all(r[2] == "replicas x2" for r in res)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_workload_bytes_headline():
    import bench
    # 2,097,152 tokens x 576 B + 256 x 16 x (576 + 512) x 2 B + 2 x 257 x 4 B
    assert bench.workload_bytes("bs256_kv8192") == 1216874504
