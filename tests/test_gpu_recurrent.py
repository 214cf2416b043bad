"""The per-branch recurrent baseline (tgdn_verify_recurrent) against the oracle and
against the fused single-pass verification, on the same inputs."""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, TOL_F32, oracle_step, rel_fro_blocks, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
from tree_speculative_decoding_gated_gb300 import tgdn  # noqa: E402


def run_both(p):
    tree, dims, dev = upload(p)
    tgdn.tree_prep(tree)
    shape = (tree.T, dims.H_v, dims.d_v)
    o_rec = torch.full(shape, float("nan"), dtype=dims.torch_dtype, device="cuda")
    tgdn.verify_recurrent(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"],
                          dev["S0"], o_rec)
    ws = tgdn.alloc_workspace(tree, dims)
    o_fused = torch.full(shape, float("nan"), dtype=dims.torch_dtype, device="cuda")
    tgdn.verify(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], dev["S0"],
                o_fused, ws)
    torch.cuda.synchronize()
    return o_rec.float().cpu().numpy(), o_fused.float().cpu().numpy()


@pytest.mark.parametrize("name,tol", [("toy", TOL_F32), ("cfg2", TOL_BF16), ("cfg3", TOL_BF16)])
def test_recurrent_matches_oracle_and_fused(name, tol):
    p = synth.make_problem(name)
    o_rec, o_fused = run_both(p)
    ref = oracle_step(p)["o"]
    cu = p.trees.cu_nodes
    assert rel_fro_blocks(o_rec, ref, cu) <= tol
    assert rel_fro_blocks(o_rec, o_fused, cu) <= tol


def test_recurrent_on_128_node_trees_and_invalid_sequences():
    rng = np.random.default_rng(3)
    cfg = synth.Config("rec", 120, B=4, H_qk=2, H_v=4, dk=128, dv=128, io="bf16",
                       tree="random", s0_sigma=0.02)
    parents = [synth.random_recursive_tree(rng, 128, 16), synth.chain_tree(17),
               np.array([-1, 0, -1], np.int32), synth.top_m_tree(rng, 8, 15)]
    trees = synth.pack_trees(parents, 128, 16)
    inputs = synth.make_node_inputs(cfg, trees.T)
    p = synth.Problem(cfg, trees, inputs, synth.make_state(cfg, B=4),
                      np.zeros(trees.T, np.int32), np.zeros(trees.T, np.int32))
    o_rec, o_fused = run_both(p)
    ref = oracle_step(p)["o"]
    assert rel_fro_blocks(o_rec, ref, trees.cu_nodes) <= TOL_BF16
    cu = trees.cu_nodes
    assert (o_rec[cu[2]:cu[3]] == 0).all()
