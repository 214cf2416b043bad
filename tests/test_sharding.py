"""Multi-process (gloo, CPU) checks of the data-parallel split used under torchrun.

Every (sequence, layer, v-head) is independent on this path, so ranks split the
sequences and exchange nothing but the timing maximum.  Two CPU ranks each run the
oracle on their share; the gathered result must equal the single-process result, and
the shares must cover every sequence exactly once."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from tree_speculative_decoding_gated_gb300 import synth


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = head_slice(synth.make_problem("cfg3"))
        seqs = list(bench.shard_range(p.trees.B, world, rank))
        sub = synth.select_sequences(p, seqs)
        t = sub.trees
        o = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, sub.inputs.q, sub.inputs.k,
                          sub.inputs.v, sub.inputs.g, sub.inputs.b, sub.S0, nthreads=1)
        acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, sub.draft_ids,
                            sub.target_ids)
        gathered = [None] * world
        dist.all_gather_object(gathered, (seqs, o, acc["accept_node"]))
        slowest = bench.max_over_ranks(float(rank + 1), world)
        if rank == 0:
            out.put((gathered, slowest))
    finally:
        dist.destroy_process_group()


def head_slice(p):
    """Two query/key heads (four value heads) keep the oracle quick."""
    i = p.inputs
    vh = [0, 1, 2, 3]
    return synth.Problem(p.cfg, p.trees, synth.Inputs(i.q[:, :2], i.k[:, :2], i.v[:, vh],
                                                      i.g[:, vh], i.b[:, vh], i.io),
                         p.S0[:, vh], p.draft_ids, p.target_ids)


@pytest.mark.parametrize("n,world", [(16, 2), (7, 2), (32, 3), (1, 2), (0, 2)])
def test_shard_range_covers_every_unit_once(n, world):
    seen = [u for r in range(world) for u in bench.shard_range(n, world, r)]
    assert seen == list(range(n))
    sizes = [len(bench.shard_range(n, world, r)) for r in range(world)]
    assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_match_single_process():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for pr in procs:
        pr.start()
    gathered, slowest = out.get(timeout=300)
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    assert slowest == 2.0
    p = head_slice(synth.make_problem("cfg3"))
    t = p.trees
    o_ref = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, p.inputs.q, p.inputs.k,
                          p.inputs.v, p.inputs.g, p.inputs.b, p.S0)
    acc_ref = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, p.draft_ids,
                            p.target_ids)
    seqs = [s for part in gathered for s in part[0]]
    assert seqs == list(range(t.B))
    o = np.concatenate([part[1] for part in gathered])
    an = np.concatenate([part[2] for part in gathered])
    assert np.array_equal(o, o_ref)
    assert np.array_equal(an, acc_ref["accept_node"])
