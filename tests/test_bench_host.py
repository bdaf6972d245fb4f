"""Host-side logic of bench.py on CPU: the whole-job reduction over ranks
(two gloo ranks), the workload scripts and the byte accounting."""

import math
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: elapsed 10+r ms, 100*(r+1) bytes, 5 tokens, e2e 20+2r ms, 7 bytes
        res = bench.reduce_over_ranks(10.0 + rank, 100.0 * (rank + 1), 5.0, 20.0 + 2 * rank, 7.0, world,
                                      torch.device("cpu"))
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            assert out[r] == (11.0, 300.0, 10.0, 22.0, 14.0)


def test_single_rank_passes_through():
    assert bench.reduce_over_ranks(1.0, 2.0, 3.0, 4.0, 5.0, 1, torch.device("cpu")) == (1.0, 2.0, 3.0, 4.0, 5.0)


def test_scenario_scripts_cover_the_workloads():
    for name in bench.WORKLOADS:
        sc = bench.Scenario(name, 0)
        assert len(sc.rids) == len(sc.lengths) > 0
        n_new = sum(1 for op in sc.ops if op[0] == "new")
        assert n_new >= len(sc.rids) - sum(1 for op in sc.ops if op[0] == "fork")
    sw = bench.Scenario("sliding_window", 0)
    # every request's history is built in 256-row chunks, each followed by a trim
    assert sum(op[2] for op in sw.ops if op[0] == "append") == sum(sw.lengths)
    ps = bench.Scenario("prefix_sharing", 0)
    assert sum(1 for op in ps.ops if op[0] == "fork") == 128


def test_attention_bytes_accounting():
    sc = bench.Scenario("gqa_decode", 0)
    lens = [512, 4096, 1000]
    got = bench.attention_bytes(sc, lens)
    kv = sum(lens) * 2 * 8 * 128 * 2               # K and V rows attended
    qo = 2 * len(lens) * 32 * 128 * 2              # q read, out written
    tab = 4 * sum(-(-L // 16) for L in lens) + 4 * len(lens)
    assert got == kv + qo + tab
    w = bench.Scenario("sliding_window", 0)
    assert bench.attention_bytes(w, [20000]) == 4096 * 4096 + 2 * 32 * 128 * 2 + 4 * (-(-20000 // 16) - 15904 // 16) + 4
