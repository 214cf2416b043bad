"""CPU checks of the seeded input recipes: every workload's tree shapes, tensor ranges and
id statistics are the ones the workload definitions state (toy: complete binary tree of
7 nodes, one 16x16 fp32 head; cfg2: top-4 tree of depth 8; cfg3: 16 random 64-node trees
of depth <= 16; cfg4: 16-token chains alternating with top-8 trees of depth 16; cfg5: 32
random 64-node trees of depth <= 12 over 36 layers).  The generators hold none of the
method's arithmetic; these tests pin what they produce, not how the method uses it."""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth


def depths(parent):
    return synth.tree_depths(np.asarray(parent))


def trees_of(name):
    t = synth.make_trees(synth.CONFIGS[name])
    return [t.parent[t.cu_nodes[i]:t.cu_nodes[i + 1]] for i in range(t.B)], t


def check_forest_order(par):
    """One root (node 0) and every parent earlier than its child."""
    assert par[0] == -1 and (par[1:] >= 0).all()
    assert (par[1:] < np.arange(1, len(par))).all()


def test_toy_tree_and_head():
    cfg = synth.CONFIGS["toy"]
    assert (cfg.B, cfg.H_qk, cfg.H_v, cfg.dk, cfg.dv, cfg.io) == (1, 1, 1, 16, 16, "f32")
    pars, t = trees_of("toy")
    assert t.sizes().tolist() == [7]
    assert pars[0].tolist() == [-1, 0, 0, 1, 1, 2, 2]
    p = synth.make_problem("toy")
    # q and k rows are unit vectors; the fp32 path is not rounded to bf16
    assert np.allclose(np.linalg.norm(p.inputs.q, axis=-1), 1.0, atol=1e-5)
    assert np.allclose(np.linalg.norm(p.inputs.k, axis=-1), 1.0, atol=1e-5)
    assert (synth.round_bf16(p.inputs.v) != p.inputs.v).any()
    assert p.draft_ids.max() < 8 and p.target_ids.max() < 8 and p.draft_ids.min() >= 0


def test_top4_tree_of_depth_8():
    pars, t = trees_of("cfg2")
    assert t.B == 1 and t.sizes().tolist() == [33]
    par = pars[0]
    check_forest_order(par)
    d = depths(par)
    assert np.bincount(d).tolist() == [1] + [4] * 8  # each depth holds M = 4 nodes
    assert (d[par[1:]] == d[1:] - 1).all()


@pytest.mark.parametrize("name,B,cap", [("cfg3", 16, 16), ("cfg5", 32, 12)])
def test_random_64_node_trees(name, B, cap):
    pars, t = trees_of(name)
    assert t.B == B and (t.sizes() == 64).all()
    assert t.n_max == 64 and t.depth_max == cap
    for par in pars:
        check_forest_order(par)
        assert depths(par).max() <= cap


def test_mixed_chains_and_top8_trees():
    pars, t = trees_of("cfg4")
    assert t.B == 64 and t.n_max == 129 and t.depth_max == 16
    for i, par in enumerate(pars):
        check_forest_order(par)
        if i % 2 == 0:  # a 16-token chain behind the root
            assert par.tolist() == list(range(-1, 16))
        else:           # a top-8 tree of depth 16
            assert len(par) == 129 and np.bincount(depths(par)).tolist() == [1] + [8] * 16


@pytest.mark.parametrize("name", ["cfg2", "cfg3", "cfg4"])
def test_bf16_inputs_gates_and_state(name):
    cfg = synth.CONFIGS[name]
    p = synth.make_problem(name)
    i = p.inputs
    T = p.trees.T
    assert i.q.shape == (T, 16, 128) and i.k.shape == (T, 16, 128) and i.v.shape == (T, 32, 128)
    assert i.g.shape == (T, 32) and i.b.shape == (T, 32)
    for x in (i.q, i.k, i.v):  # bf16-exact values held in fp32
        assert (synth.round_bf16(x) == x).all()
    # unit rows before the rounding to bf16
    assert np.allclose(np.linalg.norm(i.q, axis=-1), 1.0, atol=1e-2)
    assert (i.g <= 0).all() and (i.b > 0).all() and (i.b < 1).all()
    # g = -softplus(N(0, 1)): mean ~ -0.81; b = sigmoid(N(0, 1)): mean 0.5
    assert abs(float(i.g.mean()) + 0.81) < 0.05 and abs(float(i.b.mean()) - 0.5) < 0.02
    assert p.S0.shape == (cfg.B, 32, 128, 128) and p.S0.dtype == np.float32
    assert abs(float(p.S0.std()) - 0.02) < 1e-3


@pytest.mark.parametrize("name", ["cfg3", "cfg4"])
def test_draft_and_verifier_ids(name):
    p = synth.make_problem(name)
    t = p.trees
    assert p.draft_ids.max() < synth.VOCAB and p.target_ids.max() < synth.VOCAB
    assert p.draft_ids.min() >= 0 and p.target_ids.min() >= 0
    # the verifier's id matches the draft's with probability 0.7
    match = float((p.draft_ids == p.target_ids).mean())
    assert abs(match - 0.7) < 0.05
    # siblings (indeed any two nodes of one depth in a tree) carry distinct draft ids
    for bi in range(t.B):
        lo, hi = int(t.cu_nodes[bi]), int(t.cu_nodes[bi + 1])
        d = depths(t.parent[lo:hi])
        for level in range(int(d.max()) + 1):
            ids = p.draft_ids[lo:hi][d == level]
            assert len(np.unique(ids)) == len(ids)


def test_steps_and_layers_differ():
    """Distinct steps draw distinct trees and inputs; distinct layers distinct tensors."""
    cfg = synth.CONFIGS["cfg5"]
    a, b = synth.make_trees(cfg, 0), synth.make_trees(cfg, 1)
    assert not np.array_equal(a.parent, b.parent)
    x0 = synth.make_node_inputs(cfg, 64, step=0, layer=0)
    x1 = synth.make_node_inputs(cfg, 64, step=0, layer=1)
    assert not np.array_equal(x0.k, x1.k)
