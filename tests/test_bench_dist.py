"""Host logic of bench.py's multi-process path, on CPU with the gloo backend (2 ranks):
the max over ranks of the per-rank timings, and the profile-traffic lookup."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_profiled_traffic_tracks_the_gemm_source():
    import bench
    t = bench.profiled_traffic("l535b_t8192", "expert_gemm1")
    # either the committed summary matches the current kernel source, or traffic is withheld
    assert t is None or abs(t - 15.33e9) < 1e6
    assert bench.profiled_traffic("small_bf16", "expert_gemm1") is None
