"""The multi-rank path of bench.py on CPU: two gloo ranks, each an
independent replica with its own batch, the time taken as the max over
ranks, throughput as the bytes of all ranks over that time, and the
reference arm run by rank 0 alone."""

import argparse
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_page_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + rank, world)  # rank 1 is the slower one
        gbs = bench.whole_job_gbs(2.0e9, 4, world, slowest)
        w = wl.paged_decode(2, 64, num_q_heads=2, num_kv_heads=2, head_dim=64, lnew=1,
                            seed=bench.replica_seed(rank), device="cpu")
        digests = [None] * world
        dist.all_gather_object(digests, float(w["q"].double().sum()))
        results.put((rank, slowest, gbs, digests))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_benchmark():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    got = []
    try:
        for _ in range(2):
            got.append(results.get(timeout=180))
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    for rank, slowest, gbs, digests in sorted(got):
        assert slowest == 11.0
        assert abs(gbs - 2.0e9 * 4 * 2 / 11.0e-3 / 1e9) < 1e-9
        assert digests[0] != digests[1]  # replicas draw different batches


def test_single_rank_keeps_its_own_time():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_gbs(1e9, 2, 1, 4.0) == 1e9 * 2 / 4.0e-3 / 1e9


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = argparse.Namespace(gpus=2, steps=1, warmup=3)
    bench.run_reference(args, 1, 2)
    assert capsys.readouterr().out == ""
