"""The multi-rank path of bench.py on CPU (gloo, world size 2).

The verify step shards by request with no exchange, so the only cross-rank
logic is the timing: a barrier, the max of the ranks' times, and the
whole-job throughput (steps of all ranks over the slowest rank).  Also checks
that request shards reproduce the single-process draws: the uniform counter
carries the global request index (b_base + b).
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from oracle import oracle_reject_sample
from synth import logits_inputs, workload


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [120.0, 300.0][rank]
    sps, ms_max = bench.aggregate(ms, 10, world, "cpu")
    bench.barrier(world)
    q.put((rank, sps, ms_max))
    dist.destroy_process_group()


def test_aggregate_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, sps, ms_max in out:
        assert ms_max == 300.0
        assert abs(sps - 2 * 10 / 0.3) < 1e-9


def test_single_rank_aggregate():
    sps, ms = bench.aggregate(50.0, 5, 1, "cpu")
    assert ms == 50.0 and abs(sps - 100.0) < 1e-12


def test_request_shards_reproduce_the_whole_batch():
    wl = workload("chain_7b").scaled(B=6, V=500)
    lg = logits_inputs(wl, seed=3)
    whole = oracle_reject_sample(lg["target"], lg["draft"], lg["tokens"], None,
                                 lg["temperature"], 17, 2)
    for lo, hi in [(0, 2), (2, 6)]:
        part = oracle_reject_sample(lg["target"][lo:hi], lg["draft"][lo:hi],
                                    lg["tokens"][lo:hi], None,
                                    lg["temperature"][lo:hi], 17, 2, b_base=lo)
        for k in ("out_tokens", "path", "accepted_len"):
            assert np.array_equal(part[k], whole[k][lo:hi])
