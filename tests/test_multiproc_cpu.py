"""World-size-2 checks (gloo, CPU) of the multi-rank benchmark logic: the
workload shards into independent replicas (each rank its own batch, no
collective on the data path), the job time is the slowest rank's and the
throughput counts the work of every rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from exact_deberta_disentangled_gb300 import synth
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=2, L=64, H=2, seed=bench.rank_seed(w.seed, rank))
    local_ms = 10.0 + 5.0 * rank
    slow = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    q.put((rank, float(x.q.float().sum()), tuple(x.q.shape), slow))
    dist.destroy_process_group()


def test_two_rank_replicas_and_max_timing():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    (_, s0, sh0, m0), (_, s1, sh1, m1) = res
    assert sh0 == sh1                 # same per-rank workload shape (weak scaling)
    assert s0 != s1                   # different batches on different ranks
    assert m0 == m1 == 15.0           # every rank reports the slowest rank's time
    assert bench.job_throughput(2, 1e12, 0.5) == pytest.approx(4.0)


def test_flop_formula_matches_pages_count():
    # BH(4L^2 D + 4LRD) forward, BH(10L^2 D + 12LRD) backward at the L=8192 point
    f = bench.flops_fwd(2, 12, 8192, 64, 512)
    b = bench.flops_bwd(2, 12, 8192, 64, 512)
    assert f == pytest.approx(4.381e11, rel=1e-3)
    assert b == pytest.approx(1.1081e12, rel=1e-3)
    assert f + b == pytest.approx(1.5462e12, rel=1e-3)
