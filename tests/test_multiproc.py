"""Host logic of the multi-GPU benchmark path on CPU: two gloo ranks, each with
its own replica of the workload (weak scaling, no data-path collective), and
the whole-job value taken over the slowest rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from dsa_sparse_attention_lightning_gb300 import inputs
    wl = bench.rank_workload(1, rank)
    small = inputs.Workload("t", [512, 300], [2, 1], H=16, k=64, seed=wl.seed)
    inp = inputs.make_inputs(small)
    local_ms = 10.0 * (rank + 1)
    mx = bench.reduce_max_ms(local_ms, "cpu")
    q.put((rank, wl.seed, float(inp["w"].sum()), inp["key_cache"][:, :8].sum().item(), mx))
    dist.destroy_process_group()


def test_two_rank_weak_scaling_host_logic():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, w0, k0, m0), (r1, s1, w1, k1, m1) = res
    assert s0 != s1                          # each rank has its own replica
    assert k0 != k1
    assert m0 == m1 == 20.0                  # slowest rank's time on every rank
    import bench
    assert bench.whole_job_gbs(1_000_000, 2, 10, m0) == pytest.approx(2 * 10 * 1e6 / 0.02 / 1e9)
