"""Multi-rank host logic on CPU: two gloo ranks split a packed KDA batch by heads and by
sequences, each computes its share with the oracle, and the gathered result equals the
single-process result (heads and sequences are independent: no data-path collective is needed,
the gather here only checks the partition)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from hybrid_linear_attention_gb300 import inputs
from hybrid_linear_attention_gb300.sharding import head_shard, sequence_shard


def test_head_shard_covers_and_balances():
    for H in (1, 5, 64):
        for world in (1, 2, 3, 8):
            spans = [head_shard(H, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == H
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_sequence_shard_is_a_balanced_partition():
    lens, _ = inputs.varlen_lengths(seed=0)
    for world in (1, 2, 4, 8):
        parts = [sequence_shard(lens, world, r) for r in range(world)]
        assert sorted(i for p in parts for i in p) == list(range(len(lens)))
        loads = [sum(lens[i] for i in p) for p in parts]
        assert max(loads) - min(loads) <= max(lens)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle

        lens = [5, 40, 17, 64]
        H, d = 5, 8
        inp = inputs.kda_inputs(lens, H, d, seed=11, io_dtype=torch.float32, init_state="even")
        # by heads
        h0, h1 = head_shard(H, world, rank)
        mine = oracle.kda_forward(inp["q"][:, h0:h1], inp["k"][:, h0:h1], inp["v"][:, h0:h1],
                                  inp["g"][:, h0:h1], inp["beta"][:, h0:h1], inp["cu_seqlens"],
                                  init_state=inp["init_state"][:, h0:h1])
        parts = [None] * world
        dist.all_gather_object(parts, (h0, h1, mine["out"], mine["final_state"]))
        # by sequences
        seqs = sequence_shard(lens, world, rank)
        cu = inp["cu_seqlens"].tolist()
        seq_out = {}
        for n in seqs:
            sl = slice(cu[n], cu[n + 1])
            r = oracle.kda_forward(inp["q"][sl], inp["k"][sl], inp["v"][sl], inp["g"][sl],
                                   inp["beta"][sl], np.array([0, lens[n]], np.int32),
                                   init_state=inp["init_state"][n:n + 1])
            seq_out[n] = (r["out"], r["final_state"][0])
        seq_parts = [None] * world
        dist.all_gather_object(seq_parts, seq_out)
        if rank == 0:
            full = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                      inp["cu_seqlens"], init_state=inp["init_state"])
            out = np.concatenate([p[2] for p in sorted(parts, key=lambda p: p[0])], axis=1)
            fin = np.concatenate([p[3] for p in sorted(parts, key=lambda p: p[0])], axis=1)
            ok = np.array_equal(out, full["out"]) and np.array_equal(fin, full["final_state"])
            merged = {}
            for p in seq_parts:
                merged.update(p)
            ok = ok and sorted(merged) == list(range(len(lens)))
            for n, (o, f) in merged.items():
                ok = ok and np.array_equal(o, full["out"][cu[n]:cu[n + 1]])
                ok = ok and np.array_equal(f, full["final_state"][n])
            result_q.put(bool(ok))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_partition_heads_and_sequences():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get(timeout=10) is True
