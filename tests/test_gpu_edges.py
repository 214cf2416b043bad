"""Edge values of the GDN update eq. through the GPU kernels, against the fp64 oracle.

"Trees from Marginals", Methodik 3 ("Herausforderung") writes the update as
S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T and contrasts it with
diagonal state-space models.  Its corner cases, each on the tensor-core kernels
(bf16, d = 128: trees of <= 64 nodes and of 65-129 nodes) and on the SIMT kernel
(fp32), and through the commit folded into the next verification:
  * b = 0: pure decay (the diagonal case), o_n = e^{G_n} S0^T q_n, S_n = e^{G_n} S0;
  * b = 1 and g = 0: an exact write, S_n^T k_n = v_n;
  * strongly negative gates, g in [-20, -5] per node, on depth-30 chains and deep
    random trees: e^{G} spans hundreds of decades along a path.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, TOL_F32, oracle_step, rel_fro_blocks, run_step, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
from tree_speculative_decoding_gated_gb300 import tgdn  # noqa: E402
import oracle  # noqa: E402


def make(parents, io, seed, gb, n_max=None, depth_max=None, d=128):
    """A batch of the given trees (H_qk = 2, H_v = 4) with g and b set by gb(rng, shape)."""
    cfg = synth.Config("edge", 500 + seed, B=len(parents), H_qk=2, H_v=4, dk=d, dv=d, io=io,
                       tree="random", s0_sigma=0.05)
    dmax = max(int(synth.tree_depths(np.asarray(p)).max()) for p in parents)
    trees = synth.pack_trees([np.asarray(p, np.int32) for p in parents],
                             n_max or max(len(p) for p in parents),
                             dmax if depth_max is None else depth_max)
    inputs = synth.make_node_inputs(cfg, trees.T)
    rng = np.random.default_rng(seed)
    g, b = gb(rng, inputs.g.shape)
    inputs = synth.Inputs(inputs.q, inputs.k, inputs.v, g.astype(np.float32),
                          b.astype(np.float32), inputs.io)
    draft = rng.integers(0, 2, trees.T).astype(np.int32)
    target = np.where(rng.random(trees.T) < 0.9, draft, 1 - draft).astype(np.int32)
    return synth.Problem(cfg, trees, inputs, synth.make_state(cfg, B=trees.B), draft, target)


def no_write(rng, shape):
    return -np.log1p(np.exp(rng.standard_normal(shape))), np.zeros(shape)


def exact_write(rng, shape):
    return np.zeros(shape), np.ones(shape)


def deep_decay(rng, shape):
    return rng.uniform(-20.0, -5.0, shape), 1.0 / (1.0 + np.exp(-rng.standard_normal(shape)))


def trees_small(rng):
    return [synth.random_recursive_tree(rng, 64, 12), synth.chain_tree(13),
            synth.random_recursive_tree(rng, 40, 8), synth.random_recursive_tree(rng, 64, 16)]


def trees_deep(rng):
    return [synth.chain_tree(31), synth.random_recursive_tree(rng, 64, 30),
            synth.chain_tree(25), synth.random_recursive_tree(rng, 50, 30)]


def trees_large(rng):
    return [synth.top_m_tree(rng, 8, 16), synth.chain_tree(17), synth.top_m_tree(rng, 8, 16)]


CASES = [("no_write", no_write, trees_small), ("exact_write", exact_write, trees_small),
         ("deep_decay", deep_decay, trees_deep), ("no_write_129", no_write, trees_large),
         ("deep_decay_129", deep_decay, trees_large)]


def check(p, tol):
    tree, dims, dev = upload(p)
    got = run_step(tree, dims, dev)
    ref = oracle_step(p)
    eo = rel_fro_blocks(got["o"], ref["o"], p.trees.cu_nodes)
    es = rel_fro_blocks(got["S"], ref["S"])
    assert np.array_equal(got["accept_node"], ref["accept_node"])
    assert np.isfinite(got["o"]).all() and np.isfinite(got["S"]).all()
    return eo, es


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("name,gb,shape", CASES, ids=[c[0] for c in CASES])
def test_edge_values_against_the_oracle(name, gb, shape, io):
    rng = np.random.default_rng(sum(map(ord, name)))
    p = make(shape(rng), io, 1 + len(name), gb)
    eo, es = check(p, TOL_BF16 if io == "bf16" else TOL_F32)
    print(f"{name} {io}: output error {eo:.3e}, committed-state error {es:.3e}")
    tol = TOL_BF16 if io == "bf16" else TOL_F32
    assert eo <= tol and es <= tol, (eo, es)


def test_pure_decay_closed_form():
    """b = 0: the committed state is e^{G*} S0 exactly as the oracle's closed form."""
    rng = np.random.default_rng(11)
    p = make(trees_small(rng), "bf16", 11, no_write)
    tree, dims, dev = upload(p)
    got = run_step(tree, dims, dev)
    t, i = p.trees, p.inputs
    for bi in range(t.B):
        n = got["accept_node"][bi]
        lo = t.cu_nodes[bi]
        path, j = [], n
        while j != -1:
            path.append(j)
            j = t.parent[lo + j]
        for h in range(4):
            G = sum(float(i.g[lo + s, h]) for s in path)
            ref = np.exp(G) * p.S0[bi, h].astype(np.float64)
            err = np.linalg.norm(got["S"][bi, h] - ref) / np.linalg.norm(ref)
            assert err <= 1e-5, (bi, h, err)


@pytest.mark.parametrize("name,gb,shape", [CASES[1], CASES[2]], ids=["exact_write", "deep_decay"])
def test_edge_values_through_the_fused_commit(name, gb, shape):
    """Two steps with the first step's commit folded into the second verification
    (for the deep trees the commit path holds up to 31 entries)."""
    rng = np.random.default_rng(77 + len(name))
    p1 = make(shape(rng), "bf16", 21, gb, depth_max=30)
    p2 = make(shape(rng), "bf16", 22, gb, depth_max=30)
    ups = [upload(p1), upload(p2)]
    dims = ups[0][1]
    S = ups[0][2]["S0"].clone()
    (t1, _, d1), (t2, _, d2) = ups
    tgdn.tree_prep(t1)
    tgdn.tree_prep(t2)
    ws1, ws2 = tgdn.alloc_workspace(t1, dims), tgdn.alloc_workspace(t2, dims)
    o1 = torch.empty((t1.T, 4, 128), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty((t2.T, 4, 128), dtype=torch.bfloat16, device="cuda")
    tgdn.verify(t1, dims, d1["q"], d1["k"], d1["v"], d1["g"], d1["b"], S, o1, ws1)
    an = torch.empty(t1.B, dtype=torch.int32, device="cuda")
    al = torch.empty_like(an)
    path = torch.empty((t1.B, t1.depth_max + 1), dtype=torch.int32, device="cuda")
    tgdn.accept(t1, d1["draft"], d1["target"], an, al, path)
    tgdn.verify_fused(t2, dims, d2["q"], d2["k"], d2["v"], d2["g"], d2["b"], S, o2, ws2, t1, an,
                      path, d1["k"], ws1)
    torch.cuda.synchronize()
    tr, i1 = p1.trees, p1.inputs
    acc = oracle.accept(tr.cu_nodes, tr.parent, tr.n_max, tr.depth_max, p1.draft_ids,
                        p1.target_ids)
    S1 = oracle.commit(tr.cu_nodes, tr.parent, tr.n_max, tr.depth_max, i1.k, i1.v, i1.g, i1.b,
                       p1.S0, acc["accept_node"])
    t, i2 = p2.trees, p2.inputs
    ref = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i2.q, i2.k, i2.v, i2.g,
                        i2.b, S1)
    eo = rel_fro_blocks(o2.float().cpu().numpy(), ref, t.cu_nodes)
    es = rel_fro_blocks(S.cpu().numpy(), S1)
    print(f"{name} fused: output error {eo:.3e}, committed-state error {es:.3e}")
    assert eo <= TOL_BF16 and es <= TOL_BF16, (eo, es)
