"""The multi-rank plumbing of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs N independent replicas under torchrun (one per GPU) with a
barrier on both sides of the timed region and the maximum of the ranks'
times. This checks that plumbing without a GPU: both ranks initialise,
meet at the barrier and agree on the maximum of their values. A second test
checks the sharding reading of the GroupNorm backward on the oracle: split by
samples over two ranks, dx is local and only dgamma, dbeta need a sum
(all-reduce) to equal the unsharded result.
"""

import importlib.util
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), SWG_BENCH_BACKEND="gloo")
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    r, w = bench._dist_init(world)
    bench._barrier(w)
    m = bench._max_over_ranks(1.5 + r, w)
    bench._barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, m))


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert results == [(0, 2, 2.5), (1, 2, 2.5)]


def _gn_rank_main(rank, world, port, q):
    # the GroupNorm backward sharded by samples: dx stays local, dgamma and dbeta are all-reduced
    import numpy as np
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import oracle
    from synth import group_norm_inputs

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    N, C, HW, G, eps = 6, 12, 10, 4, 1e-5
    dy, x, gamma = (t.double().numpy() for t in group_norm_inputs(N, C, HW, G, torch.float32, seed=31))
    lo, hi = rank * N // world, (rank + 1) * N // world
    dx, dg, db = oracle.group_norm_bwd(dy[lo:hi], x[lo:hi], gamma, G, eps)
    t = torch.from_numpy(np.concatenate([dg, db]))
    dist.all_reduce(t)
    gathered = [torch.zeros(N // world, C, HW, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(np.ascontiguousarray(dx)))
    dist.destroy_process_group()
    if rank == 0:
        fdx, fdg, fdb = oracle.group_norm_bwd(dy, x, gamma, G, eps)
        ok = (np.array_equal(torch.cat(gathered).numpy(), fdx)
              and np.allclose(t[:C].numpy(), fdg, rtol=1e-13, atol=1e-13)
              and np.allclose(t[C:].numpy(), fdb, rtol=1e-13, atol=1e-13))
        q.put(ok)


@pytest.mark.timeout(120)
def test_group_norm_backward_shards_by_samples():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gn_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok = q.get(timeout=90)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert ok
