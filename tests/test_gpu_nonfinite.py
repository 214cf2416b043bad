"""Non-finite node inputs stay inside their own sequence.

The library does not scan q, k, v for NaN or Inf (that would be an extra pass over the
inputs on the hot path): a non-finite value makes its own sequence's outputs, factors
and committed state meaningless, and nothing else.  Here one sequence gets a NaN query,
one a NaN value and one an infinite key; prep, verification, acceptance and the commit
run on the tensor-core kernels (trees of <= 64 nodes, and a mixed batch with 129-node
trees), and every other sequence's output rows, accepted node and committed state must
equal, bit for bit, those of the same batch without the bad values.  No status word is
raised (tree structure is fine) and nothing faults or hangs.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import run_step, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


def _problem(kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "small":
        parents = [synth.random_recursive_tree(rng, int(n), 12) for n in (64, 40, 64, 17, 64, 9,
                                                                           33, 64)]
        n_max = 64
    else:
        parents = [synth.top_m_tree(rng, 8, 16), synth.chain_tree(17), synth.top_m_tree(rng, 8, 16),
                   synth.random_recursive_tree(rng, 64, 12), synth.top_m_tree(rng, 8, 16),
                   synth.chain_tree(17), synth.random_recursive_tree(rng, 100, 16),
                   synth.chain_tree(17)]
        n_max = 129
    trees = synth.pack_trees(parents, n_max, 16)
    cfg = synth.Config("nonfinite", 700 + seed, B=len(parents), H_qk=2, H_v=4, dk=128, dv=128,
                       io="bf16", tree="random", s0_sigma=0.05)
    inputs = synth.make_node_inputs(cfg, trees.T)
    draft = rng.integers(0, 2, trees.T).astype(np.int32)
    target = np.where(rng.random(trees.T) < 0.9, draft, 1 - draft).astype(np.int32)
    return synth.Problem(cfg, trees, inputs, synth.make_state(cfg, B=len(parents)), draft, target)


@pytest.mark.parametrize("kind", ["small", "mixed"])
def test_non_finite_inputs_stay_in_their_sequence(kind):
    p = _problem(kind, 5 if kind == "small" else 6)
    clean = run_step(*upload(p))
    cu = p.trees.cu_nodes
    i = p.inputs
    q, k, v = i.q.copy(), i.k.copy(), i.v.copy()
    q[cu[1] + 3, 0, 5] = np.nan          # sequence 1: a query
    v[cu[2] + 1, 2, 7] = np.nan          # sequence 2: a value
    k[cu[6], 1, 0] = np.inf              # sequence 6: its root's key
    bad = synth.Problem(p.cfg, p.trees, synth.Inputs(q, k, v, i.g, i.b, i.io), p.S0, p.draft_ids,
                        p.target_ids)
    got = run_step(*upload(bad))
    assert (got["status"] == 0).all() and (clean["status"] == 0).all()
    for s in (0, 3, 4, 5, 7):
        rows = np.arange(cu[s], cu[s + 1])
        assert np.array_equal(got["o"][rows], clean["o"][rows]), (kind, s)
        assert np.array_equal(got["S"][s], clean["S"][s]), (kind, s)
    assert np.array_equal(got["accept_node"], clean["accept_node"])
    # the poisoned sequences' own results are not finite (nothing hides the bad value)
    assert not np.isfinite(got["o"][cu[1]:cu[2]]).all()
