"""The benchmark's multi-rank plumbing on the host: two gloo ranks (launched
as processes, rendezvous on 127.0.0.1) set up the process group the way
bench.py does under torchrun, agree on the slowest rank's time, and only rank
0 runs the oracle reference arm. Replicas share nothing on the data path."""

import importlib.util
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    bench = _bench()
    r, w, local, dist = bench.dist_setup(world)
    bench.barrier(dist)
    slowest = bench.max_over_ranks(1.0 + r, dist, "cpu")
    # the reference arm: rank 0 alone runs (and prints); the others exit at once
    class Args:
        workload, steps, warmup, gpus = "llama3_8b_layer", 1, 0, world
    rc = bench.run_reference(Args) if r != 0 else None
    bench.barrier(dist)
    dist.destroy_process_group()
    q.put((r, w, slowest, rc))


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == world for o in out)
    assert all(o[2] == 2.0 for o in out)  # max over ranks of 1.0 + rank
    assert out[1][3] == 0                  # rank 1 returns 0 from the reference arm without work


def test_cpu_baseline_uses_host_threads_and_names_the_cpu():
    """The oracle baseline runs on every host thread it may use and records
    the thread count and the CPU model."""
    import workloads
    bench = _bench()
    case = workloads.build_case("cpu_base", 3, B=6, H_q=8, H_kv=2, D=64, page_size=16, seq_lens=[40, 17, 90, 5, 64, 33],
                                dtype="f32", scale=0.125)
    b = bench.cpu_baseline(case, budget_s=0.2)
    assert b["kind"] == "oracle" and b["value"] > 0
    assert 1 <= b["cores"] <= bench.host_threads() and b["cores"] == min(bench.host_threads(), 6)
    assert isinstance(b["cpu"], str) and b["cpu"]
