"""tgdn_verify_fused: the previous step's commit folded into the next verify.

Decodes of several steps run through the C ABI twice — commit and verify as
separate passes, and the fused call — and both are compared with the fp64 oracle,
which commits each step by replaying the accepted root path and verifies the next
tree from that committed state.  Covers the tensor-core path, its two-pass
fallbacks (a previous tree deeper than 30, a tree above 64 nodes), invalid and
empty sequences on either side, accepted paths of the full 31 entries, and the final
separate commit.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, head_pair_subset, rel_fro_blocks, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
from tree_speculative_decoding_gated_gb300 import tgdn  # noqa: E402
import oracle  # noqa: E402


def oracle_decode(problems, S0):
    """Per step: outputs verified from the committed state, then the commit (fp64)."""
    S = np.asarray(S0, np.float64)
    outs, states = [], []
    for p in problems:
        t, i = p.trees, p.inputs
        outs.append(oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v,
                                  i.g, i.b, S))
        acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, p.draft_ids,
                            p.target_ids)
        S = oracle.commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b, S,
                          acc["accept_node"])
        states.append(S)
    return outs, states


def gpu_decode(problems, S0, fused, n_max=None):
    """The same decode on the GPU.  fused: steps after the first use tgdn_verify_fused with
    two alternating workspaces; otherwise commit and verify run as separate passes.  The
    last step is committed with tgdn_commit either way.  Returns per-step outputs, the
    state verified by each step and the final state."""
    S = torch.from_numpy(np.ascontiguousarray(S0, np.float32)).cuda()
    ups = [upload(p, n_max=n_max) for p in problems]
    dims = ups[0][1]
    outs, verified = [], []
    prev = None
    wss = []
    for s, (tree, _, dev) in enumerate(ups):
        tgdn.tree_prep(tree)
        ws = tgdn.alloc_workspace(tree, dims)
        wss.append(ws)
        o = torch.full((tree.T, dims.H_v, dims.d_v), float("nan"), dtype=dims.torch_dtype,
                       device="cuda")
        if prev is None:
            tgdn.verify(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], S, o, ws)
        elif fused:
            ptree, pdev, pws, pan, ppath = prev
            tgdn.verify_fused(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], S, o,
                              ws, ptree, pan, ppath, pdev["k"], pws)
        else:
            ptree, pdev, pws, pan, ppath = prev
            tgdn.commit(ptree, dims, pan, pdev["k"], pws, S, S)
            tgdn.verify(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], S, o, ws)
        verified.append(S.clone())
        an = torch.empty(tree.B, dtype=torch.int32, device="cuda")
        al = torch.empty(tree.B, dtype=torch.int32, device="cuda")
        path = torch.empty((tree.B, tree.depth_max + 1), dtype=torch.int32, device="cuda")
        tgdn.accept(tree, dev["draft"], dev["target"], an, al, path)
        outs.append(o)
        prev = (tree, dev, ws, an, path)
    ptree, pdev, pws, pan, _ = prev
    tgdn.commit(ptree, dims, pan, pdev["k"], pws, S, S)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy()
    return [f(o) for o in outs], [f(v) for v in verified], f(S)


def check_decode(problems, S0, n_max=None):
    ref_o, ref_S = oracle_decode(problems, S0)
    fo, fv, fS = gpu_decode(problems, S0, fused=True, n_max=n_max)
    so, sv, sS = gpu_decode(problems, S0, fused=False, n_max=n_max)
    for s, p in enumerate(problems):
        cu = p.trees.cu_nodes
        eo = rel_fro_blocks(fo[s], ref_o[s], cu)
        print(f"step {s}: fused o={eo:.3e}")
        assert eo <= TOL_BF16, (s, eo)
        if s > 0:
            es = rel_fro_blocks(fv[s], ref_S[s - 1])
            print(f"step {s}: fused committed state={es:.3e}")
            assert es <= TOL_BF16, (s, es)
            # the fused pass commits with the same arithmetic as the separate one, in
            # another order; the state then enters the next products as bf16, where a
            # one-ulp difference can flip a rounding, so the two agree to well below the
            # tolerance but not bit for bit
            assert rel_fro_blocks(fv[s], sv[s]) <= 1e-4
        np.testing.assert_allclose(fo[s], so[s], rtol=2e-2, atol=1e-2)
    assert rel_fro_blocks(fS, ref_S[-1]) <= TOL_BF16
    return fo, fv, fS


def test_two_steps_full_size():
    """16 sequences of 64-node trees, all 32 value heads: commit of step 0 fused into step 1."""
    ps = [synth.make_problem("cfg3", step=s) for s in (0, 1)]
    check_decode(ps, ps[0].S0)


def test_three_step_decode_on_two_heads():
    ps = [head_pair_subset(synth.make_problem("cfg3", step=s), [0, 9]) for s in (0, 1, 2)]
    check_decode(ps, ps[0].S0)


def _custom(parents, seed, n_max, depth_max, all_match=False):
    cfg = synth.Config("fused", 300 + seed, B=len(parents), H_qk=2, H_v=4, dk=128, dv=128,
                       io="bf16", tree="random", s0_sigma=0.05)
    trees = synth.pack_trees([np.asarray(p, np.int32) for p in parents], n_max, depth_max)
    inputs = synth.make_node_inputs(cfg, trees.T)
    rng = np.random.default_rng(seed)
    draft = rng.integers(0, 3, trees.T).astype(np.int32)
    target = draft.copy() if all_match else np.where(
        rng.random(trees.T) < 0.8, draft, rng.integers(0, 3, trees.T)).astype(np.int32)
    return synth.Problem(cfg, trees, inputs, synth.make_state(cfg, B=trees.B), draft, target)


def test_invalid_and_empty_sequences_on_either_side():
    rng = np.random.default_rng(5)
    first = [synth.random_recursive_tree(rng, 40, 10), np.zeros(0, np.int32),
             np.array([-1, 0, -1], np.int32), synth.chain_tree(12),
             synth.random_recursive_tree(rng, 64, 20), np.array([-1, 2, 1], np.int32)]
    second = [np.zeros(0, np.int32), synth.random_recursive_tree(rng, 30, 8),
              synth.chain_tree(5), np.array([-1, 0, 7], np.int32),
              synth.random_recursive_tree(rng, 64, 12), synth.chain_tree(2)]
    p1 = _custom(first, 1, 64, 20)
    p2 = _custom(second, 2, 64, 20)
    fo, fv, fS = check_decode([p1, p2], p1.S0)
    # sequences whose first tree was empty or invalid keep their state through the commit
    for bi in (1, 2, 5):
        assert np.array_equal(fv[1][bi], p1.S0[bi])
    cu = p2.trees.cu_nodes
    assert (fo[1][cu[3]:cu[4]] == 0).all()     # invalid second tree: zero outputs


def test_deep_previous_tree_runs_two_passes():
    """A previous tree of depth 31 is above the fused kernel's path bound: commit + verify."""
    rng = np.random.default_rng(6)
    p1 = _custom([synth.chain_tree(32), synth.random_recursive_tree(rng, 50, 12)], 3, 64, 31,
                 all_match=True)
    p2 = _custom([synth.random_recursive_tree(rng, 64, 12), synth.chain_tree(20)], 4, 64, 30)
    check_decode([p1, p2], p1.S0)


def test_deep_trees_and_long_accepted_paths_fused():
    """Depth-30 chains and deep random trees on three consecutive steps with every draft
    token matching: the accepted paths (up to 31 entries) go through the fused commit's
    32-entry product, and each step's verify through the 30-deep path solve."""
    rng = np.random.default_rng(11)
    steps = []
    for s in range(3):
        parents = [synth.chain_tree(31), synth.random_recursive_tree(rng, 64, 30),
                   synth.random_recursive_tree(rng, 50, 25), synth.chain_tree(17)]
        steps.append(_custom(parents, 20 + s, 64, 30, all_match=True))
    for p in steps:
        acc = oracle.accept(p.trees.cu_nodes, p.trees.parent, p.trees.n_max, p.trees.depth_max,
                            p.draft_ids, p.target_ids)
        assert acc["accept_len"][0] == 31  # the whole chain is accepted
    check_decode(steps, steps[0].S0)


def test_trees_above_64_nodes_run_two_passes():
    ps = [head_pair_subset(synth.make_problem("cfg3", step=s), [3]) for s in (0, 1)]
    check_decode(ps, ps[0].S0, n_max=65)


def test_stack_layer_full_size_sampled():
    """One layer of the 36-layer stack at full size (32 sequences of 64-node trees, depth
    <= 12, all 32 value heads), three decode steps with the commit fused in: the launch
    configuration the benchmark times.  The oracle replays a sample of sequences on two
    query/key heads."""
    ps = [synth.make_problem("cfg5", step=s) for s in (0, 1, 2)]
    fo, fv, fS = gpu_decode(ps, ps[0].S0, fused=True)
    seqs = [0, 7, 19, 31]
    subs = [head_pair_subset(synth.select_sequences(p, seqs), [0, 11]) for p in ps]
    ref_o, ref_S = oracle_decode(subs, subs[0].S0)
    vh = subs[0].meta["v_heads"]
    for s, sub in enumerate(subs):
        rows = sub.meta["rows"]
        eo = rel_fro_blocks(fo[s][rows][:, vh], ref_o[s], sub.trees.cu_nodes)
        print(f"stack layer step {s}: sampled o={eo:.3e}")
        assert eo <= TOL_BF16, (s, eo)
        if s > 0:
            es = rel_fro_blocks(fv[s][seqs][:, vh], ref_S[s - 1])
            print(f"stack layer step {s}: sampled committed state={es:.3e}")
            assert es <= TOL_BF16, (s, es)
    assert rel_fro_blocks(fS[seqs][:, vh], ref_S[-1]) <= TOL_BF16
