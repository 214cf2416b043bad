"""Pins of the ancestor-masked tree-attention oracle (CPU only).

Tree verification in attention layers: every draft-tree node attends to the
sequence's cached context and to its own root path (Technisches Resümee,
Problemstellung: tree verification with attention masks).  The oracle is checked
against closed forms, textbook causal attention on chains, invariances and the
grouped-query mapping.
"""
import numpy as np
import pytest

from oracle import tree_attention as ta


def rand_case(parents, H_q=4, H_kv=2, d=16, P_max=12, prefix=None, seed=0):
    rng = np.random.default_rng(seed)
    cu = np.zeros(len(parents) + 1, np.int64)
    cu[1:] = np.cumsum([len(p) for p in parents])
    par = np.concatenate(parents).astype(np.int64)
    T, B = int(cu[-1]), len(parents)
    q = rng.standard_normal((T, H_q, d))
    kt = rng.standard_normal((T, H_kv, d))
    vt = rng.standard_normal((T, H_kv, d))
    kc = rng.standard_normal((B, P_max, H_kv, d))
    vc = rng.standard_normal((B, P_max, H_kv, d))
    pl = np.array(prefix if prefix is not None else rng.integers(0, P_max + 1, B), np.int64)
    return dict(cu_nodes=cu, parent=par, status=np.zeros(B, np.int64), q=q, k_tree=kt,
                v_tree=vt, k_cache=kc, v_cache=vc, prefix_len=pl, scale=0.3)


TREE = np.array([-1, 0, 0, 1, 1, 2, 2, 3], np.int64)


def test_zero_queries_average_the_visible_values():
    c = rand_case([TREE, np.array([-1, 0, 1], np.int64)], seed=1)
    c["q"][:] = 0
    o = ta.tree_attention(**c)
    for b in range(2):
        lo, hi = c["cu_nodes"][b], c["cu_nodes"][b + 1]
        P = c["prefix_len"][b]
        for n in range(hi - lo):
            anc = [lo + s for s in ta.ancestors_or_self(c["parent"][lo:hi], n)]
            for h in range(4):
                hk = h // 2
                vis = list(c["v_cache"][b, :P, hk]) + list(c["v_tree"][anc, hk])
                np.testing.assert_allclose(o[lo + n, h], np.mean(vis, axis=0), atol=1e-13)


def test_lone_root_without_context_returns_its_value():
    c = rand_case([np.array([-1], np.int64)], prefix=[0], seed=2)
    o = ta.tree_attention(**c)
    for h in range(4):
        assert np.array_equal(o[0, h], c["v_tree"][0, h // 2])


def test_chain_is_causal_attention():
    """A chain after P cached positions is ordinary causal attention over the P + N tokens
    (a lower-triangular mask on the concatenated sequence)."""
    N, P = 6, 5
    c = rand_case([np.arange(-1, N - 1)], prefix=[P], P_max=P, seed=3)
    o = ta.tree_attention(**c)
    for hk in range(2):
        K = np.concatenate([c["k_cache"][0, :, hk], c["k_tree"][:, hk]])
        V = np.concatenate([c["v_cache"][0, :, hk], c["v_tree"][:, hk]])
        for g in range(2):
            h = hk * 2 + g
            Q = c["q"][:, h]                              # queries at positions P .. P+N-1
            logits = c["scale"] * Q @ K.T                 # [N, P + N]
            mask = np.tril(np.ones((N, P + N), bool), k=P)
            logits = np.where(mask, logits, -np.inf)
            w = np.exp(logits - logits.max(axis=1, keepdims=True))
            w /= w.sum(axis=1, keepdims=True)
            np.testing.assert_allclose(o[:, h], w @ V, atol=1e-13)


def test_dominant_key_returns_its_value():
    c = rand_case([TREE], prefix=[7], seed=4)
    n, h, j = 6, 3, 2
    hk = h // 2
    c["k_cache"][0, j, hk] = 400.0 * c["q"][n, h] / np.linalg.norm(c["q"][n, h])
    o = ta.tree_attention(**c)
    np.testing.assert_allclose(o[n, h], c["v_cache"][0, j, hk], atol=1e-12)


def test_star_two_key_closed_form():
    c = rand_case([np.array([-1, 0, 0, 0], np.int64)], prefix=[0], seed=5)
    o = ta.tree_attention(**c)
    for n in (1, 2, 3):
        for h in range(4):
            hk = h // 2
            s0 = c["scale"] * c["q"][n, h] @ c["k_tree"][0, hk]
            s1 = c["scale"] * c["q"][n, h] @ c["k_tree"][n, hk]
            want = (np.exp(s0) * c["v_tree"][0, hk] + np.exp(s1) * c["v_tree"][n, hk]) / (
                np.exp(s0) + np.exp(s1))
            np.testing.assert_allclose(o[n, h], want, atol=1e-13)


def test_non_ancestors_do_not_matter():
    c = rand_case([TREE], prefix=[4], seed=6)
    o = ta.tree_attention(**c)
    n = 7                                   # root path 0 -> 1 -> 3 -> 7
    other = [2, 4, 5, 6]
    rng = np.random.default_rng(60)
    for key in ("k_tree", "v_tree", "q"):
        c[key][other] = rng.standard_normal(c[key][other].shape)
    o2 = ta.tree_attention(**c)
    assert np.array_equal(o2[n], o[n])


def test_relabelling_permutes_outputs():
    c = rand_case([TREE], prefix=[3], seed=7)
    o = ta.tree_attention(**c)
    perm = np.array([0, 5, 2, 7, 1, 3, 6, 4])     # new index -> old index
    inv = np.argsort(perm)
    new_par = np.array([-1 if TREE[p] == -1 else inv[TREE[p]] for p in perm], np.int64)
    c2 = dict(c, parent=new_par)
    for key in ("q", "k_tree", "v_tree"):
        c2[key] = c[key][perm]
    o2 = ta.tree_attention(**c2)
    np.testing.assert_allclose(o2, o[perm], atol=1e-13)


def test_grouped_query_heads_match_repeated_kv_heads():
    c = rand_case([TREE, np.array([-1, 0], np.int64)], H_q=4, H_kv=2, seed=8)
    o = ta.tree_attention(**c)
    c2 = dict(c)
    for key in ("k_tree", "v_tree"):
        c2[key] = np.repeat(c[key], 2, axis=1)
    for key in ("k_cache", "v_cache"):
        c2[key] = np.repeat(c[key], 2, axis=2)
    o2 = ta.tree_attention(**c2)
    np.testing.assert_allclose(o2, o, atol=1e-14)


def test_invalid_sequences_get_zeros():
    c = rand_case([TREE, np.array([-1, 0], np.int64)], seed=9)
    c["status"] = np.array([0, 3])
    o = ta.tree_attention(**c)
    assert (o[8:] == 0).all() and (o[:8] != 0).any()
