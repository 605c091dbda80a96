"""The benchmark's multi-rank host logic on CPU with gloo (world size 2).

Under torchrun each rank runs its own batch (weak scaling): a rank-specific
seed, no collective on the data path, and one max-reduction of the step time.
"""
import importlib.util
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench = _bench()
    r, w, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    # each rank reports a different step time; every rank must see the max
    got = bench.max_over_ranks(1.0 + 0.5 * r, dist, torch.device("cpu"))
    from load_balanced_paged_02_gb300 import workloads as wl
    wk = bench.rank_workload(wl.WORKLOADS["mixed"], r)
    lens = wl.draw_lengths(wk)
    out[r] = (got, wk.seed, int(lens.sum()))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_weak_scaling_and_max_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == pytest.approx(1.5) and res[1][0] == pytest.approx(1.5)
    assert res[0][1] != res[1][1], "each rank draws its own batch"
    assert res[0][2] != res[1][2]


def test_single_rank_needs_no_process_group():
    bench = _bench()
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.0, None, torch.device("cpu")) == 3.0
