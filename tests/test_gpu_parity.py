"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bars: tree metadata and acceptance bit-exact; node outputs and committed
states within a max relative Frobenius error (per sequence and value head) of
2e-2 on bf16 io and 1e-4 on fp32 io.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import (TOL_BF16, TOL_F32, assert_meta_equal, head_pair_subset, oracle_step,
                     rel_fro_blocks, run_step, upload)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


def check(p, got, ref, tol, label=""):
    assert_meta_equal(got, ref)
    eo = rel_fro_blocks(got["o"], ref["o"], p.trees.cu_nodes)
    es = rel_fro_blocks(got["S"], ref["S"])
    print(f"{label} rel-Frobenius o={eo:.3e} S={es:.3e}")
    assert eo <= tol and es <= tol, (eo, es)
    return eo, es


def test_toy_fp32():
    p = synth.make_problem("toy")
    tree, dims, dev = upload(p)
    got = run_step(tree, dims, dev)
    check(p, got, oracle_step(p), TOL_F32, "toy")


@pytest.mark.parametrize("name", ["cfg2", "cfg3"])
def test_full_config(name):
    p = synth.make_problem(name)
    tree, dims, dev = upload(p)
    got = run_step(tree, dims, dev)
    check(p, got, oracle_step(p), TOL_BF16, name)


def test_cfg4_full_size_sampled():
    """B = 64 mixed chains (17 nodes) and top-8 trees (129 nodes): the whole batch runs on the
    GPU, the oracle checks every other chain/tree pair on two query/key heads."""
    p = synth.make_problem("cfg4")
    tree, dims, dev = upload(p)
    got = run_step(tree, dims, dev)
    seqs = [0, 1, 30, 31, 62, 63]
    sub = head_pair_subset(synth.select_sequences(p, seqs), [0, 15])
    ref = oracle_step(sub)
    rows = sub.meta["rows"]
    vh = sub.meta["v_heads"]
    assert np.array_equal(got["status"][seqs], ref["prep"]["status"])
    for key in ("accept_node", "accept_len", "path"):
        assert np.array_equal(got[key][seqs], ref[key]), key
    assert np.array_equal(got["depth"][rows], ref["prep"]["depth"])
    eo = rel_fro_blocks(got["o"][rows][:, vh], ref["o"], sub.trees.cu_nodes)
    es = rel_fro_blocks(got["S"][seqs][:, vh], ref["S"])
    print(f"cfg4 sampled rel-Frobenius o={eo:.3e} S={es:.3e}")
    assert eo <= TOL_BF16 and es <= TOL_BF16


def test_tc_and_simt_paths_agree():
    """cfg3 through the 64-node tensor-core kernel (n_max = 64), the 128-node tensor-core
    kernel (n_max = 65) and the SIMT kernel (n_max = 129)."""
    p = synth.make_problem("cfg3")
    ref = oracle_step(p)
    outs = []
    for n_max in (64, 65, 129):
        tree, dims, dev = upload(p, n_max=n_max)
        got = run_step(tree, dims, dev)
        eo = rel_fro_blocks(got["o"], ref["o"], p.trees.cu_nodes)
        es = rel_fro_blocks(got["S"], ref["S"])
        print(f"n_max={n_max} o={eo:.3e} S={es:.3e}")
        assert eo <= TOL_BF16 and es <= TOL_BF16
        outs.append(got)
    assert np.array_equal(outs[0]["accept_node"], outs[1]["accept_node"])


def test_commit_in_place_matches_out_of_place():
    p = synth.make_problem("cfg3")
    tree, dims, dev = upload(p)
    a = run_step(tree, dims, dev)
    b = run_step(tree, dims, dev, in_place=True)
    assert np.array_equal(a["S"], b["S"])
    assert np.array_equal(a["o"], b["o"])
