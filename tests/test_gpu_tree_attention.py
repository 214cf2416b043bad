"""tgdn_tree_attention (ancestor-masked tree attention) against the fp64 oracle.

Each node attends to its sequence's cached context and its own root path.  Checked over
grouped-query ratios 1-16, context lengths 0 .. P_max including ragged last tiles, trees
of 1-128 nodes (one or two key tiles of tree nodes), empty and invalid sequences, and
non-ancestor invariance (bitwise) on the GPU; with and without the workspace that splits
the cached context over several CTAs.  Bar: max relative Frobenius error per
(sequence, query head) block <= 2e-2 (bf16 io; P is a bf16 operand).
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, rel_fro_blocks, to_device_io

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
from tree_speculative_decoding_gated_gb300 import tgdn  # noqa: E402
from oracle import tree_attention as ta  # noqa: E402
import oracle  # noqa: E402


def make_case(parents, H_q, H_kv, P_max, prefix, n_max=None, seed=0, d=128):
    rng = np.random.default_rng(seed)
    trees = synth.pack_trees([np.asarray(p, np.int32) for p in parents],
                             n_max or max([len(p) for p in parents] + [1]), 30)
    T, B = trees.T, trees.B
    bf = lambda x: synth.round_bf16(x.astype(np.float32))
    q = bf(rng.standard_normal((T, H_q, d)))
    kt = bf(rng.standard_normal((T, H_kv, d)))
    vt = bf(rng.standard_normal((T, H_kv, d)))
    kc = bf(rng.standard_normal((B, P_max, H_kv, d)))
    vc = bf(rng.standard_normal((B, P_max, H_kv, d)))
    return dict(trees=trees, q=q, kt=kt, vt=vt, kc=kc, vc=vc,
                prefix=np.asarray(prefix, np.int32), scale=1.0 / np.sqrt(d))


def run_gpu(c, split=False):
    t = c["trees"]
    tree = tgdn.Tree.from_host(t.cu_nodes, t.parent, t.n_max, t.depth_max)
    tgdn.tree_prep(tree)
    dev = lambda x: to_device_io(x, "bf16")
    o = torch.full(c["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    P_max = c["kc"].shape[1]
    kc = dev(c["kc"]) if P_max > 0 else None
    vc = dev(c["vc"]) if P_max > 0 else None
    ws = None
    if split:
        nb = tgdn.tree_attention_workspace_bytes(tree, c["q"].shape[1], c["kt"].shape[1],
                                                 c["q"].shape[2], P_max)
        ws = torch.full((max(nb, 16),), 255, dtype=torch.uint8, device="cuda")  # stale bytes
    tgdn.tree_attention(tree, dev(c["q"]), dev(c["kt"]), dev(c["vt"]), kc, vc,
                        torch.from_numpy(c["prefix"]).cuda(), o, c["scale"], ws=ws)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), tree.status.cpu().numpy()


def run_oracle(c):
    t = c["trees"]
    st = oracle.prep(t.cu_nodes, t.parent, t.n_max, t.depth_max)["status"]
    return ta.tree_attention(t.cu_nodes, t.parent, st, c["q"], c["kt"], c["vt"], c["kc"],
                             c["vc"], np.minimum(c["prefix"], c["kc"].shape[1]), c["scale"])


def check(c):
    ref = run_oracle(c)
    for split in (False, True):
        got, status = run_gpu(c, split)
        err = rel_fro_blocks(got, ref, c["trees"].cu_nodes)
        print(f"tree attention (split={split}) rel-Frobenius {err:.3e}")
        assert err <= TOL_BF16
    return got, ref, status


def test_small_batches_split_the_context():
    """Few (sequence, head) items: the workspace lets the context be split."""
    rng = np.random.default_rng(9)
    parents = [synth.random_recursive_tree(rng, 40, 8) for _ in range(2)]
    c = make_case(parents, 8, 2, 2600, [2600, 1333], n_max=64, seed=9)
    t = c["trees"]
    tree = tgdn.Tree.from_host(t.cu_nodes, t.parent, t.n_max, t.depth_max)
    assert tgdn.tree_attention_workspace_bytes(tree, 8, 2, 128, 2600) > 0
    check(c)


@pytest.mark.parametrize("H_q,H_kv", [(16, 4), (8, 8), (16, 8), (16, 2), (16, 1)])
def test_random_trees_with_context(H_q, H_kv):
    rng = np.random.default_rng(H_q * 10 + H_kv)
    B, P_max = 6, 200
    parents = [synth.random_recursive_tree(rng, int(n), 12) for n in rng.integers(1, 65, B)]
    prefix = [0, 1, 63, 64, 130, 200]
    check(make_case(parents, H_q, H_kv, P_max, prefix, n_max=64, seed=H_q + H_kv))


def test_full_size_64_node_batch():
    """16 sequences of 64-node trees, 16 query heads over 4 key/value heads, 512 cached
    positions each (the whole batch on the GPU, checked in full)."""
    rng = np.random.default_rng(3)
    parents = [synth.random_recursive_tree(rng, 64, 16) for _ in range(16)]
    check(make_case(parents, 16, 4, 512, [512] * 16, n_max=64, seed=3))


def test_trees_up_to_128_nodes_and_no_context():
    rng = np.random.default_rng(4)
    parents = [synth.top_m_tree(rng, 8, 15), synth.random_recursive_tree(rng, 100, 20),
               synth.chain_tree(30)]
    check(make_case(parents, 16, 4, 0, [0, 0, 0], n_max=128, seed=4))


def test_empty_and_invalid_sequences():
    rng = np.random.default_rng(5)
    parents = [synth.random_recursive_tree(rng, 20, 6), np.zeros(0, np.int32),
               np.array([-1, 0, -1], np.int32), np.array([-1], np.int32),
               np.array([-1, 2, 1], np.int32)]
    c = make_case(parents, 8, 2, 96, [96, 5, 40, 0, 70], n_max=32, seed=5)
    got, ref, status = check(c)
    assert status.tolist() == [0, 0, 3, 0, 4]
    cu = c["trees"].cu_nodes
    assert (got[cu[2]:cu[3]] == 0).all() and (got[cu[4]:cu[5]] == 0).all()


def test_non_ancestor_edits_leave_outputs_bitwise():
    rng = np.random.default_rng(6)
    par = synth.random_recursive_tree(rng, 50, 10)
    c = make_case([par], 16, 4, 128, [100], n_max=64, seed=6)
    base, _ = run_gpu(c)
    n = 49
    keep, j = set(), n
    while j != -1:
        keep.add(j)
        j = par[j]
    other = [i for i in range(50) if i not in keep]
    for key in ("kt", "vt", "q"):
        c[key] = c[key].copy()
        c[key][other] = synth.round_bf16(rng.standard_normal(c[key][other].shape).astype(np.float32))
    edit, _ = run_gpu(c)
    assert np.array_equal(edit[n], base[n])


def test_unsupported_shapes_are_refused():
    c = make_case([np.array([-1, 0], np.int32)], 4, 4, 8, [8], seed=7, d=64)
    with pytest.raises(tgdn.TgdnError):
        run_gpu(c)


@pytest.mark.parametrize("scale", [0.0, -0.1, float("nan"), float("inf")])
def test_scale_must_be_positive_and_finite(scale):
    c = make_case([np.array([-1, 0], np.int32)], 4, 4, 8, [8], seed=8)
    c["scale"] = scale
    with pytest.raises(tgdn.TgdnError):
        run_gpu(c)


def test_many_context_splits_with_an_empty_context():
    """Four splits of a 4096-position context next to a sequence with no context (its
    context splits are empty and only the last one, with the tree's keys, counts)."""
    rng = np.random.default_rng(10)
    parents = [synth.random_recursive_tree(rng, 40, 8), synth.random_recursive_tree(rng, 30, 6),
               np.array([-1, 0, -1], np.int32)]
    c = make_case(parents, 8, 8, 4096, [4096, 0, 4096], n_max=64, seed=10)
    t = c["trees"]
    tree = tgdn.Tree.from_host(t.cu_nodes, t.parent, t.n_max, t.depth_max)
    assert tgdn.tree_attention_workspace_bytes(tree, 8, 8, 128, 4096) > 0
    got, ref, status = check(c)
    assert status.tolist() == [0, 0, 3]
