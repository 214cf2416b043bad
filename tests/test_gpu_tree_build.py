"""tgdn_tree_build (top-w best-first draft-tree construction) against the CPU oracle.

Every output is an integer decision or an fp32 sum formed by the same single addition
on both sides, so the comparison is bit-exact: parent, token, depth, score, tree size
and round count, for whole batches, over budgets up to 256, K up to 16, w from 1 to
beyond the budget, exact ties, the depth cap, and trees that feed verification.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, oracle_step, rel_fro_blocks, run_step, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
from tree_speculative_decoding_gated_gb300 import tgdn  # noqa: E402
from oracle import tree_build as tb  # noqa: E402


def run(root, logp, tok, budget, w, depth_max):
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = tgdn.tree_build(d(root), d(logp), d(tok), budget, w, depth_max)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def check(root, logp, tok, budget, w, depth_max):
    got = run(root, logp, tok, budget, w, depth_max)
    ref = tb.build(root, logp, tok, budget, w, depth_max)
    for key in ("n_nodes", "rounds", "parent", "token", "depth"):
        assert np.array_equal(got[key], ref[key]), key
    assert np.array_equal(got["score"].view(np.uint32), ref["score"].view(np.uint32))
    return got


@pytest.mark.parametrize("budget,K,w,depth_max", [
    (64, 8, 1, 12), (64, 8, 4, 12), (64, 8, 8, 12), (33, 4, 4, 8), (128, 8, 16, 16),
    (129, 8, 8, 16), (256, 16, 32, 30), (256, 16, 1, 64), (256, 16, 300, 64), (100, 3, 7, 5),
])
def test_matches_oracle(budget, K, w, depth_max):
    root, logp, tok = synth.make_build_tables(32, budget, K, seed=budget * 7 + w)
    got = check(root, logp, tok, budget, w, depth_max)
    if depth_max >= budget:
        assert (got["n_nodes"] == budget).all()


@pytest.mark.parametrize("w", [1, 3, 8])
def test_exact_ties(w):
    """Log-probabilities on a 0.25 grid: many equal priorities, decided by candidate id."""
    root, logp, tok = synth.make_build_tables(16, 96, 6, seed=40 + w, tie_step=0.25)
    check(root, logp, tok, 96, w, 20)


@pytest.mark.parametrize("budget,K,w,depth_max", [(1, 4, 2, 5), (10, 1, 3, 20), (10, 4, 2, 0),
                                                  (12, 3, 2, 1), (200, 2, 64, 6)])
def test_edge_cases(budget, K, w, depth_max):
    """A lone root, chains (K = 1), no children (depth cap 0), a heap that runs dry."""
    root, logp, tok = synth.make_build_tables(5, budget, K, seed=budget + K)
    check(root, logp, tok, budget, w, depth_max)


def test_empty_batch_is_a_no_op():
    z = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = tgdn.tree_build(z, torch.zeros((0, 4, 2), device="cuda"),
                          torch.zeros((0, 4, 2), dtype=torch.int32, device="cuda"), 4, 2, 3)
    assert out["n_nodes"].numel() == 0


def test_built_trees_verify_against_the_oracle():
    """Trees from the construction kernel go straight into prep, verify, accept, commit."""
    B, budget, K, w, dmax = 8, 64, 8, 8, 12
    root, logp, tok = synth.make_build_tables(B, budget, K, seed=77)
    got = run(root, logp, tok, budget, w, dmax)
    n = got["n_nodes"]
    parents = [got["parent"][b, :n[b]] for b in range(B)]
    cfg = synth.Config("built", 400, B=B, H_qk=2, H_v=4, dk=128, dv=128, io="bf16",
                       tree="random", s0_sigma=0.02)
    trees = synth.pack_trees(parents, 64, dmax)
    draft = np.concatenate([got["token"][b, :n[b]] for b in range(B)]).astype(np.int32)
    rng = np.random.default_rng(5)
    target = np.where(rng.random(len(draft)) < 0.8, draft, -1).astype(np.int32)
    p = synth.Problem(cfg, trees, synth.make_node_inputs(cfg, trees.T), synth.make_state(cfg, B),
                      draft, target)
    tree, dims, dev = upload(p)
    res = run_step(tree, dims, dev)
    ref = oracle_step(p)
    assert (res["status"] == 0).all()
    assert np.array_equal(res["accept_node"], ref["accept_node"])
    assert rel_fro_blocks(res["o"], ref["o"], trees.cu_nodes) <= TOL_BF16
    assert rel_fro_blocks(res["S"], ref["S"]) <= TOL_BF16
