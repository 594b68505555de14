"""Multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

The benchmark runs independent replicas (one per rank, no collective on the
data path) and reports all ranks' rows over the slowest rank's time; the
context-parallel layout shards query rows (head-tail balanced, [HP-CP] DSA
CP with load_balance) against the full key side.  Both are checked here
without a GPU: the time reduction and throughput of bench.py, and that the
shards' rows, computed by the oracle on each rank and gathered, reproduce the
unsharded run bit for bit."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, port, outq):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        import oracle
        import synth
        # replica timing: the job time is the slowest rank's
        ms = [12.5, 17.0][rank]
        slow = bench.max_over_ranks(ms, WORLD, "cpu")
        value = bench.job_value(WORLD, 32768, slow)
        seeds = [None] * WORLD
        dist.all_gather_object(seeds, bench.replica_seed(rank))
        # CP shard of the tiny workload: head-tail rows of this rank
        wl = synth.WORKLOADS["tiny_fp32_S256"]
        S = wl["S"]
        x = synth.make_inputs(wl)
        rows = synth.head_tail_rows(S, WORLD, rank).numpy()
        shard = {n: (v[:, rows] if n in ("q_I", "w", "q") else v) for n, v in x.items()}
        _, idx, O, m, l = oracle.dsa_forward(shard["q_I"], shard["k_I"], shard["w"], shard["q"],
                                             shard["kv"], wl["topk"], wl["scale"], wl["d_v"],
                                             q_row_index=rows)
        parts = [None] * WORLD
        dist.all_gather_object(parts, (rows, idx, O, m, l))
        if rank == 0:
            outq.put((slow, value, seeds, parts))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas_and_cp_shards():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(WORLD)]
    for pr in procs:
        pr.start()
    slow, value, seeds, parts = q.get(timeout=300)
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    assert slow == 17.0
    assert value == pytest.approx(2 * 32768 / 17.0e-3)
    assert sorted(seeds) == [0, 1]                 # distinct replica problems

    import oracle
    import synth
    wl = synth.WORKLOADS["tiny_fp32_S256"]
    x = synth.make_inputs(wl)
    _, idx, O, m, l = oracle.dsa_forward(x["q_I"], x["k_I"], x["w"], x["q"], x["kv"], wl["topk"],
                                         wl["scale"], wl["d_v"])
    covered = np.concatenate([p[0] for p in parts])
    assert np.array_equal(np.sort(covered), np.arange(wl["S"]))   # the shards partition the rows
    for rows, sidx, sO, sm_, sl in parts:
        assert np.array_equal(sidx[0], idx[0, rows])
        assert np.array_equal(sO[0], O[0, rows])
        assert np.array_equal(sm_[0], m[0, rows])
        assert np.array_equal(sl[0], l[0, rows])
