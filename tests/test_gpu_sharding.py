"""The data-parallel split through the library: a rank's share of the sequences, run on
its own, gives bit for bit the rows the whole batch gives.

Under torchrun every rank of bench.py takes bench.shard_range(B, world, rank) of the
sequences and runs the whole decode step on them alone; the path exchanges nothing
(every sequence, layer and v-head is independent).  The ranks' kernels never wait on one
another, so here they run one after the other on one GPU: for each rank's share, tree
prep, verification, acceptance and the commit through the C ABI on that sub-batch alone
must reproduce the full batch's output rows, accepted nodes and committed states exactly
(same kernels, same per-item arithmetic, only the item-to-CTA assignment differs).
"""
import numpy as np
import pytest

import bench
from tree_speculative_decoding_gated_gb300 import synth
from helpers import run_step, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


def _rows(cu, seqs):
    return np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])


@pytest.mark.parametrize("name", ["cfg3", "cfg5"])
@pytest.mark.parametrize("world", [2, 3, 4])
def test_rank_shares_equal_the_whole_batch(name, world):
    p = synth.make_problem(name)
    full = run_step(*upload(p))
    cu = p.trees.cu_nodes
    covered = []
    for rank in range(world):
        seqs = list(bench.shard_range(p.trees.B, world, rank))
        covered += seqs
        if not seqs:
            continue
        sub = synth.select_sequences(p, seqs)
        got = run_step(*upload(sub))
        rows = _rows(cu, seqs)
        assert np.array_equal(got["o"], full["o"][rows]), (name, world, rank)
        assert np.array_equal(got["accept_node"], full["accept_node"][seqs])
        assert np.array_equal(got["S"], full["S"][seqs]), (name, world, rank)
        assert np.array_equal(got["status"], full["status"][seqs])
    assert covered == list(range(p.trees.B))


def _fused_two_steps(p1, p2):
    """Step 1 verify + accept, then step 2 verify with step 1's commit folded in
    (the benchmark's launch configuration); the step-2 outputs and the committed state."""
    from tree_speculative_decoding_gated_gb300 import tgdn
    (t1, dims, d1), (t2, _, d2) = upload(p1), upload(p2)
    S = d1["S0"].clone()
    for t in (t1, t2):
        tgdn.tree_prep(t)
    ws1, ws2 = tgdn.alloc_workspace(t1, dims), tgdn.alloc_workspace(t2, dims)
    o1 = torch.empty((t1.T, dims.H_v, dims.d_v), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty((t2.T, dims.H_v, dims.d_v), dtype=torch.bfloat16, device="cuda")
    tgdn.verify(t1, dims, d1["q"], d1["k"], d1["v"], d1["g"], d1["b"], S, o1, ws1)
    an = torch.empty(t1.B, dtype=torch.int32, device="cuda")
    al = torch.empty_like(an)
    path = torch.empty((t1.B, t1.depth_max + 1), dtype=torch.int32, device="cuda")
    tgdn.accept(t1, d1["draft"], d1["target"], an, al, path)
    tgdn.verify_fused(t2, dims, d2["q"], d2["k"], d2["v"], d2["g"], d2["b"], S, o2, ws2, t1, an,
                      path, d1["k"], ws1)
    torch.cuda.synchronize()
    return o2.float().cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("world", [2, 3])
def test_rank_shares_equal_the_whole_batch_fused(world):
    p1, p2 = synth.make_problem("cfg5", step=0), synth.make_problem("cfg5", step=1)
    o_full, S_full = _fused_two_steps(p1, p2)
    cu2 = p2.trees.cu_nodes
    for rank in range(world):
        seqs = list(bench.shard_range(p1.trees.B, world, rank))
        o, S = _fused_two_steps(synth.select_sequences(p1, seqs), synth.select_sequences(p2, seqs))
        assert np.array_equal(o, o_full[_rows(cu2, seqs)]), (world, rank)
        assert np.array_equal(S, S_full[seqs]), (world, rank)
