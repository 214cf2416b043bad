"""GPU property sweep and edge cases against the fp64 oracle, plus invariants.

Covers random small trees (1-40 nodes, depth <= 16) for head sizes 16/64/128
and both io types, chains, stars, single nodes, empty and invalid sequences in
ragged batches, the 64-node / depth-30 limits of the tensor-core kernel, a
129-node tree, non-ancestor invariance (bitwise) and rollback-free two-step
consistency.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import (TOL_BF16, TOL_F32, assert_meta_equal, oracle_step, rel_fro_blocks,
                     run_step, upload)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


def custom(parents, H_qk, H_v, d, io, seed, n_max=None, depth_max=None, vocab=3):
    cfg = synth.Config("prop", 100 + seed, B=len(parents), H_qk=H_qk, H_v=H_v, dk=d, dv=d,
                       io=io, tree="random", s0_sigma=0.05)
    valid = [p for p in parents if len(p) and _valid(p)]
    dmax = max([int(synth.tree_depths(p).max()) for p in valid] + [0])
    trees = synth.pack_trees([np.asarray(p, np.int32) for p in parents],
                             n_max or max([len(p) for p in parents] + [1]),
                             dmax if depth_max is None else depth_max)
    inputs = synth.make_node_inputs(cfg, trees.T)
    S0 = synth.make_state(cfg, B=trees.B)
    rng = np.random.default_rng(seed)
    draft = rng.integers(0, vocab, trees.T).astype(np.int32)
    target = np.where(rng.random(trees.T) < 0.75, draft, rng.integers(0, vocab, trees.T)).astype(np.int32)
    return synth.Problem(cfg, trees, inputs, S0, draft, target)


def _valid(p):
    p = np.asarray(p)
    N = len(p)
    if ((p < -1) | (p >= N)).any() or (p == np.arange(N)).any() or (p == -1).sum() != 1:
        return False
    for i in range(N):
        j, h = i, 0
        while p[j] != -1 and h <= N:
            j, h = p[j], h + 1
        if p[j] != -1:
            return False
    return True


def run_and_check(p, tol, **kw):
    tree, dims, dev = upload(p, **kw)
    got = run_step(tree, dims, dev)
    ref = oracle_step(p)
    assert_meta_equal(got, ref)
    eo = rel_fro_blocks(got["o"], ref["o"], p.trees.cu_nodes)
    es = rel_fro_blocks(got["S"], ref["S"])
    assert eo <= tol and es <= tol, (eo, es)
    return got, ref


@pytest.mark.parametrize("seed", range(10))
def test_random_sweep(seed):
    rng = np.random.default_rng(1000 + seed)
    d = [16, 64, 128][seed % 3]
    io = "bf16" if seed % 2 == 0 else "f32"
    H_qk, H_v = [(1, 1), (2, 4), (4, 8)][seed % 3]
    B = int(rng.integers(1, 7))
    parents = []
    for _ in range(B):
        kind = rng.integers(4)
        N = int(rng.integers(1, 41))
        if kind == 0:
            parents.append(synth.chain_tree(min(N, 17)))
        elif kind == 1:
            parents.append(np.array([-1] + [0] * (N - 1), np.int32))      # star
        else:
            parents.append(synth.random_recursive_tree(rng, N, int(rng.integers(1, 17))))
    p = custom(parents, H_qk, H_v, d, io, seed)
    run_and_check(p, TOL_BF16 if io == "bf16" else TOL_F32)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_ragged_batch_with_empty_and_invalid_sequences(io):
    rng = np.random.default_rng(7)
    parents = [
        synth.random_recursive_tree(rng, 30, 8),
        np.zeros(0, np.int32),                           # empty sequence
        np.array([-1], np.int32),                        # single node
        np.array([-1, 0, 5, 1], np.int32),               # parent out of range
        np.array([-1, 0, -1, 2], np.int32),              # two roots
        np.array([-1, 2, 1, 0], np.int32),               # cycle 1 <-> 2
        synth.chain_tree(12),
        synth.random_recursive_tree(rng, 45, 10),
    ]
    p = custom(parents, 2, 4, 128, io, 3, n_max=64, depth_max=11)
    got, ref = run_and_check(p, TOL_BF16 if io == "bf16" else TOL_F32)
    assert got["status"].tolist() == [0, 0, 0, 2, 3, 4, 0, 0]
    cu = p.trees.cu_nodes
    for bi in (3, 4, 5):
        assert (got["o"][cu[bi]:cu[bi + 1]] == 0).all()
        assert np.array_equal(got["S"][bi], p.S0[bi])
    assert got["accept_node"][1] == -1 and got["accept_len"][1] == 0


def test_too_big_and_too_deep():
    parents = [synth.chain_tree(10), synth.chain_tree(5)]
    p = custom(parents, 1, 2, 64, "bf16", 4, n_max=8, depth_max=3)
    tree, dims, dev = upload(p)
    got = run_step(tree, dims, dev)
    assert got["status"].tolist() == [1, 5]
    assert (got["o"] == 0).all()
    assert np.array_equal(got["S"], p.S0)


@pytest.mark.parametrize("case", ["chain31", "chain32", "full64", "tree129"])
def test_kernel_limits(case):
    rng = np.random.default_rng(11)
    if case == "chain31":      # depth 30: the deepest tree the tensor-core kernel takes
        parents = [synth.chain_tree(31), synth.random_recursive_tree(rng, 64, 30)]
    elif case == "chain32":    # depth 31: SIMT kernel
        parents = [synth.chain_tree(32)]
    elif case == "full64":     # 64 nodes in every sequence, mixed depths
        parents = [synth.random_recursive_tree(rng, 64, int(c)) for c in (1, 4, 16, 30)]
    else:                      # 129 nodes: above the tensor-core node bound
        parents = [synth.top_m_tree(rng, 8, 16), synth.chain_tree(17)]
    p = custom(parents, 2, 4, 128, "bf16", 5)
    run_and_check(p, TOL_BF16)


def _relabel(par, new_root):
    """The same tree with its nodes renumbered so that the root gets index new_root."""
    N = len(par)
    perm = np.roll(np.arange(N), new_root)      # new index -> old index, perm[new_root] = 0
    inv = np.argsort(perm)
    return np.array([-1 if par[perm[i]] == -1 else inv[par[perm[i]]] for i in range(N)],
                    np.int32)


@pytest.mark.parametrize("case", ["random", "deep", "chain60", "star128", "ragged", "fold129",
                                  "mixed16", "mixed30", "allsmall"])
def test_trees_of_65_to_128_nodes(case):
    """The 128-node tensor-core kernel: full, deep, chain and star trees, and a ragged batch
    with empty and invalid sequences.  In a launch above 64 nodes the sequences of at most
    64 nodes go to the 64-node kernel (mixed16: its paired path solve, depth <= 16;
    mixed30: its one-row solve, depth up to 30)."""
    rng = np.random.default_rng(41)
    if case == "random":
        parents = [synth.random_recursive_tree(rng, int(n), 16) for n in (65, 90, 128, 100)]
    elif case == "deep":       # depth 30, the kernel's bound
        parents = [synth.random_recursive_tree(rng, 128, 30), synth.chain_tree(31)]
    elif case == "chain60":    # above the depth bound: SIMT kernel
        parents = [synth.chain_tree(60), synth.random_recursive_tree(rng, 90, 8)]
    elif case == "star128":
        parents = [np.array([-1] + [0] * 127, np.int32), synth.random_recursive_tree(rng, 70, 3)]
    elif case == "ragged":
        parents = [synth.random_recursive_tree(rng, 120, 12), np.zeros(0, np.int32),
                   np.array([-1, 0, 3, 2], np.int32), synth.chain_tree(5),
                   synth.random_recursive_tree(rng, 128, 20)]
    elif case == "mixed16":
        parents = [synth.chain_tree(17), synth.random_recursive_tree(rng, 100, 16),
                   np.array([-1], np.int32), synth.random_recursive_tree(rng, 64, 16),
                   synth.top_m_tree(rng, 8, 16), synth.random_recursive_tree(rng, 33, 5),
                   synth.random_recursive_tree(rng, 65, 16), np.array([-1, 0, 3, 2], np.int32)]
    elif case == "mixed30":
        parents = [synth.chain_tree(25), synth.random_recursive_tree(rng, 128, 30),
                   synth.random_recursive_tree(rng, 50, 30), synth.chain_tree(31)]
    elif case == "allsmall":   # a launch above 64 nodes whose sequences are all small
        parents = [synth.random_recursive_tree(rng, int(n), 12) for n in (64, 10, 40, 1)]
    else:   # 129 nodes: root first (folded into the state) and root in the middle (SIMT)
        t129 = synth.top_m_tree(rng, 8, 16)
        parents = [t129, _relabel(t129, 64), synth.random_recursive_tree(rng, 129, 14),
                   synth.chain_tree(17), np.array([-1, 0, 3, 2], np.int32)]
    n_max = 129 if case in ("fold129", "mixed16") else 128
    p = custom(parents, 2, 4, 128, "bf16", 12, n_max=n_max)
    got, ref = run_and_check(p, TOL_BF16)
    if case == "ragged":
        assert got["status"].tolist() == [0, 0, 4, 0, 0]
    if case == "mixed16":
        assert got["status"].tolist() == [0, 0, 0, 0, 0, 0, 0, 4]


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_non_ancestor_edits_leave_outputs_bitwise(io, n_max=None):
    rng = np.random.default_rng(21)
    par = synth.random_recursive_tree(rng, 48, 10)
    p = custom([par], 2, 4, 128, io, 6, n_max=n_max)
    tree, dims, dev = upload(p)
    base = run_step(tree, dims, dev)
    n = 47
    keep = set()
    j = n
    while j != -1:
        keep.add(j)
        j = par[j]
    other = [i for i in range(48) if i not in keep]
    i = p.inputs
    k2, v2, g2, b2 = i.k.copy(), i.v.copy(), i.g.copy(), i.b.copy()
    k2[other] = synth.round_bf16(rng.standard_normal(k2[other].shape).astype(np.float32) * 0.1)
    v2[other] = synth.round_bf16(rng.standard_normal(v2[other].shape).astype(np.float32))
    g2[other] *= 0.5
    b2[other] = 1.0 - b2[other]
    p2 = synth.Problem(p.cfg, p.trees, synth.Inputs(i.q, k2, v2, g2, b2, io), p.S0,
                       p.draft_ids, p.target_ids)
    tree2, dims2, dev2 = upload(p2)
    edit = run_step(tree2, dims2, dev2)
    assert np.array_equal(edit["o"][n], base["o"][n])


def test_two_step_rollback_free():
    """verify(T1) -> accept -> commit -> verify(T2) equals verify of T2 hung below T1's
    accepted path, started from S0 (on T2's rows)."""
    rng = np.random.default_rng(31)
    p1par = synth.random_recursive_tree(rng, 24, 6)
    p1 = custom([p1par], 2, 4, 128, "bf16", 8)
    p1.target_ids[:] = p1.draft_ids             # accept the deepest node
    tree, dims, dev = upload(p1)
    r1 = run_step(tree, dims, dev)
    n_star = int(r1["accept_node"][0])
    p2par = synth.random_recursive_tree(rng, 20, 6)
    p2 = custom([p2par], 2, 4, 128, "bf16", 9)
    p2.S0 = r1["S"].astype(np.float32)          # the committed state
    tree2, dims2, dev2 = upload(p2)
    r2 = run_step(tree2, dims2, dev2)
    path = [int(x) for x in r1["path"][0] if x >= 0]
    L = len(path)
    joined = np.array(list(range(-1, L - 1)) + [x + L if x >= 0 else L - 1 for x in p2par], np.int32)
    cat = lambda a, b: np.concatenate([a[path], b])
    i1, i2 = p1.inputs, p2.inputs
    pj = synth.Problem(p1.cfg, synth.pack_trees([joined], L + 20, 64),
                       synth.Inputs(cat(i1.q, i2.q), cat(i1.k, i2.k), cat(i1.v, i2.v),
                                    cat(i1.g, i2.g), cat(i1.b, i2.b), "bf16"),
                       p1.S0, np.zeros(L + 20, np.int32), np.zeros(L + 20, np.int32))
    ref = oracle_step(pj)
    e = rel_fro_blocks(r2["o"], ref["o"][L:], np.array([0, 20]))
    assert e <= TOL_BF16, e
    assert n_star == path[-1]


def test_non_ancestor_edits_on_the_128_node_kernel():
    test_non_ancestor_edits_leave_outputs_bitwise("bf16", n_max=100)


@pytest.mark.parametrize("io,d", [("bf16", 128), ("f32", 64)])
def test_header_maximum_sizes(io, d):
    """n_max = TGDN_MAX_NODES (256) and depth_max = TGDN_MAX_DEPTH (64): 256-node trees
    (random, a star, a 65-node chain reaching depth 64) next to a single node, through prep,
    verification, acceptance and the commit (four ancestor-mask words per node, a 65-entry
    accepted path)."""
    rng = np.random.default_rng(256)
    parents = [synth.random_recursive_tree(rng, 256, 64), synth.chain_tree(65),
               np.array([-1] + [0] * 255, np.int32), np.array([-1], np.int32),
               synth.random_recursive_tree(rng, 200, 40)]
    p = custom(parents, 1, 2, d, io, 64, n_max=256, depth_max=64)
    run_and_check(p, TOL_BF16 if io == "bf16" else TOL_F32)
