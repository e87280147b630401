"""The multi-rank plumbing of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs N independent replicas under torchrun (one per GPU) with a
barrier on both sides of the timed region and the maximum of the ranks'
times. This checks that plumbing without a GPU: both ranks initialise,
meet at the barrier and agree on the maximum of their values.
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
