"""Mixed launches at the size where the kernels change how they deal items.

A launch with trees above 64 nodes runs the 64-node kernel on the sequences of at most
64 nodes and the 129-node kernel on the rest.  Up to 2048 sequences each kernel lists its
own sequences (a warp ballot over cu_nodes) and numbers its items over them; above that
it deals every (sequence, head) item and steps over the other kernel's.  Both ways are run
here on batches of 2048 and 2050 sequences (mostly 1-3-node trees, some 17-node chains,
a few 129-node top-8 trees rooted at node 0; one query/key and one value head, d = 128,
bf16), through verification, acceptance and the commit, and compared with the fp64
oracle on a sample of sequences that covers every kind and the ends of the batch.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, rel_fro_blocks, run_step, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
import oracle  # noqa: E402


def _batch(B, seed):
    rng = np.random.default_rng(seed)
    parents, kinds = [], []
    for s in range(B):
        if s % 512 == 3:
            parents.append(synth.top_m_tree(rng, 8, 16))
            kinds.append("tree129")
        elif s % 7 == 0:
            parents.append(synth.chain_tree(17))
            kinds.append("chain17")
        else:
            parents.append(synth.random_recursive_tree(rng, int(rng.integers(1, 4)), 2))
            kinds.append("small")
    trees = synth.pack_trees(parents, 129, 16)
    cfg = synth.Config("large", 900 + seed, B=B, H_qk=1, H_v=1, dk=128, dv=128, io="bf16",
                       tree="random", s0_sigma=0.05)
    inputs = synth.make_node_inputs(cfg, trees.T)
    draft = rng.integers(0, 2, trees.T).astype(np.int32)
    target = np.where(rng.random(trees.T) < 0.9, draft, 1 - draft).astype(np.int32)
    p = synth.Problem(cfg, trees, inputs, synth.make_state(cfg, B=B), draft, target)
    return p, kinds


@pytest.mark.parametrize("B", [2048, 2050])
def test_mixed_batch_around_the_item_list_limit(B):
    p, kinds = _batch(B, B)
    got = run_step(*upload(p))
    assert (got["status"] == 0).all()
    sample = sorted({0, 1, 3, 7, B - 1, B - 2} | {s for s in range(B) if kinds[s] == "tree129"}
                    | {s for s in range(0, B, 301)})
    sub = synth.select_sequences(p, sample)
    t, i = sub.trees, sub.inputs
    ref_o = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v, i.g, i.b,
                          sub.S0)
    acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, sub.draft_ids,
                        sub.target_ids)
    ref_S = oracle.commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b,
                          sub.S0, acc["accept_node"])
    cu = p.trees.cu_nodes
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in sample])
    eo = rel_fro_blocks(got["o"][rows], ref_o, t.cu_nodes)
    es = rel_fro_blocks(got["S"][sample], ref_S)
    print(f"B={B}: output error {eo:.3e}, committed-state error {es:.3e}")
    assert np.array_equal(got["accept_node"][sample], acc["accept_node"])
    assert eo <= TOL_BF16 and es <= TOL_BF16, (eo, es)
