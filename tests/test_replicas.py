"""The multi-GPU path is replicas only (no exchange step): check the host-side
cross-rank reduction bench.py uses, with two gloo ranks on CPU."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [0.010, 0.012][rank]      # rank 1 is the slower replica
        e2e = [100.0, 90.0][rank]
        out = bench.reduce_across_ranks(ms, e2e, 41_779_200, "cpu")
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_two_replicas_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        ms_all, value_all, e2e_all = res[r]
        assert ms_all == 0.012                       # max over ranks
        assert abs(value_all - 2 * 41_779_200 / 0.012e-3 / 1e9) < 1e-6  # both ranks' bytes
        assert e2e_all == 190.0                      # replicas add up
