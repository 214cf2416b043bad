"""Ancestor-masked tree attention — TEST INFRASTRUCTURE ONLY (CPU oracle, fp64).

"Trees from Marginals" (Technisches Resümee, Problemstellung): tree verification of
a draft tree in ordinary attention layers is done with attention masks; the
hybrid verifier's attention layers verify the same tree as its GDN layers.  Each
tree node attends to the sequence's committed context (the KV cache) and to the
tree nodes on its own root path, itself included; siblings and other branches are
masked out.  This module states that plainly, one node and one key/value head at a
time, in fp64.  Only the tests may call it.

Readings where the page is silent (also listed in the design notes):
  * the committed context of sequence b is prefix_len[b] cached positions, all
    visible to every node of b's tree;
  * logits are scale * q.k (the caller picks scale, e.g. 1/sqrt(d)); softmax over
    the visible keys; no positional encoding inside (q, k arrive rotated);
  * query head h reads key/value head h / (H_q / H_kv) (grouped-query attention);
  * a sequence whose tree is invalid gets zero outputs.

Pins (tests/test_tree_attention_oracle.py): zero queries give the mean of the
visible values, a lone root without context returns its own value, a chain equals
causal attention over context + chain, a dominant key returns its value,
two-key closed form on stars, non-ancestor and relabelling invariance, and the
grouped-query mapping against repeated key/value heads.
"""
from __future__ import annotations

import numpy as np


def ancestors_or_self(parent: np.ndarray, n: int) -> list[int]:
    """Root-path of node n (root first), by walking parents."""
    path = []
    j = int(n)
    while j != -1:
        path.append(j)
        j = int(parent[j])
    return path[::-1]


def tree_attention(cu_nodes, parent, status, q, k_tree, v_tree, k_cache, v_cache, prefix_len,
                   scale: float):
    """q [T][H_q][d]; k_tree, v_tree [T][H_kv][d]; k_cache, v_cache [B][P_max][H_kv][d];
    prefix_len [B]; status [B] (0 = valid tree).  Returns o [T][H_q][d] (fp64)."""
    q = np.asarray(q, np.float64)
    k_tree = np.asarray(k_tree, np.float64)
    v_tree = np.asarray(v_tree, np.float64)
    k_cache = np.asarray(k_cache, np.float64)
    v_cache = np.asarray(v_cache, np.float64)
    T, H_q, d = q.shape
    H_kv = k_tree.shape[1]
    G = H_q // H_kv
    o = np.zeros((T, H_q, d), np.float64)
    for b in range(len(cu_nodes) - 1):
        lo, hi = int(cu_nodes[b]), int(cu_nodes[b + 1])
        if status[b] != 0 or hi == lo:
            continue
        P = int(prefix_len[b])
        par = np.asarray(parent[lo:hi])
        for n in range(hi - lo):
            A = [lo + s for s in ancestors_or_self(par, n)]
            for hk in range(H_kv):
                keys = np.concatenate([k_cache[b, :P, hk], k_tree[A, hk]], axis=0)
                vals = np.concatenate([v_cache[b, :P, hk], v_tree[A, hk]], axis=0)
                for g in range(G):
                    h = hk * G + g
                    s = scale * (keys @ q[lo + n, h])
                    w = np.exp(s - s.max())
                    o[lo + n, h] = (w / w.sum()) @ vals
    return o
