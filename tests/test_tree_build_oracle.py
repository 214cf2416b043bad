"""Pins of the top-w best-first tree-construction oracle (CPU only).

"Trees from Marginals", Technisches Resümee, Methodik 2 "Baumerstellung": the w best
candidates are taken from the heap and expanded together.  The oracle is checked
against a hand-worked fixture, against brute force (w = 1 is plain best-first, which
keeps the best B nodes of the candidate tree), against the level order that a w
covering whole levels must give, and against per-node invariants.
"""
import math
import os

import numpy as np
import pytest

from oracle import tree_build as tb

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_build_small.txt")


def load_golden():
    table, cases, cur = {}, {}, None
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "table":
            table[int(f[1])] = (float(f[2]), float(f[3]), int(f[4]), int(f[5]))
        elif f[0] == "case":
            cur = int(f[1].split("=")[1])
            cases[cur] = {}
        else:
            cases[cur][f[0]] = [float(x) for x in f[1:]]
    n = len(table)
    logp = np.array([[table[i][0], table[i][1]] for i in range(n)], np.float32)
    tok = np.array([[table[i][2], table[i][3]] for i in range(n)], np.int32)
    return logp, tok, cases


@pytest.mark.parametrize("w", [1, 2])
def test_hand_worked_fixture(w):
    logp, tok, cases = load_golden()
    want = cases[w]
    r = tb.build_one(100, logp, tok, budget=6, w=w, depth_max=3)
    assert r["parent"].tolist() == [int(x) for x in want["parent"]]
    assert r["token"].tolist() == [int(x) for x in want["token"]]
    assert r["depth"].tolist() == [int(x) for x in want["depth"]]
    assert r["score"].tolist() == want["score"]
    assert r["rounds"] == int(want["rounds"][0])


def uniform_table(ell, budget):
    """Every node offers the same K continuations: the candidate tree no longer depends on
    the order in which nodes are taken."""
    K = len(ell)
    logp = np.tile(np.asarray(ell, np.float32), (budget, 1))
    tok = np.tile(np.arange(K, dtype=np.int32), (budget, 1))
    return logp, tok


def brute_force_scores(ell, depth_max, depth_limit):
    """Scores of every node of the K-ary candidate tree down to depth_limit, each formed by
    fp32 additions along its path (root first)."""
    ell = np.asarray(ell, np.float32)
    out = [np.float32(0.0)]
    level = [np.float32(0.0)]
    for d in range(1, min(depth_max, depth_limit) + 1):
        level = [np.float32(s + ell[r]) for s in level for r in range(len(ell))]
        out += level
    return np.array(out, np.float32)


@pytest.mark.parametrize("seed", range(6))
def test_w1_keeps_the_best_nodes(seed):
    rng = np.random.default_rng(seed)
    K = int(rng.integers(2, 4))
    budget = int(rng.integers(4, 11))
    depth_max = int(rng.integers(1, 6))
    ell = -np.sort(rng.exponential(1.0, K)).astype(np.float32)
    logp, tok = uniform_table(ell, budget)
    r = tb.build_one(0, logp, tok, budget, 1, depth_max)
    allv = np.sort(brute_force_scores(ell, depth_max, budget - 1))[::-1]
    n = min(budget, len(allv))
    assert r["n_nodes"] == n
    assert np.array_equal(np.sort(r["score"])[::-1], allv[:n])


@pytest.mark.parametrize("seed", range(4))
def test_w1_total_score_is_never_beaten(seed):
    """With the candidate tree fixed, plain best-first (w = 1) has the highest total
    score of any ancestor-closed tree of B nodes; batching w > 1 can only lose."""
    rng = np.random.default_rng(100 + seed)
    ell = -np.sort(rng.exponential(0.7, 4)).astype(np.float32)
    budget = 30
    logp, tok = uniform_table(ell, budget)
    best = tb.build_one(0, logp, tok, budget, 1, 8)["score"].astype(np.float64).sum()
    for w in (2, 3, 5, 8, 29):
        got = tb.build_one(0, logp, tok, budget, w, 8)["score"].astype(np.float64).sum()
        assert got <= best + 1e-9


def test_wide_w_gives_level_order():
    """w at least the tree size: each round takes one whole depth level (as much of it as
    the budget allows), best first."""
    rng = np.random.default_rng(7)
    K, budget = 3, 20
    logp = -rng.exponential(1.0, (budget, K)).astype(np.float32)
    tok = np.tile(np.arange(K, dtype=np.int32), (budget, 1))
    r = tb.build_one(0, logp, tok, budget, budget, 10)
    d, s = r["depth"], r["score"]
    assert np.all(np.diff(d) >= 0)
    for lev in range(1, d.max() + 1):
        assert np.all(np.diff(s[d == lev]) <= 0)
    assert (d == 1).sum() == K and (d == 2).sum() == K * K
    assert r["rounds"] == d.max()


def check_invariants(r, logp, tok, budget, w, depth_max):
    n = r["n_nodes"]
    par, dep, sc, tk = r["parent"], r["depth"], r["score"], r["token"]
    assert par[0] == -1 and dep[0] == 0 and sc[0] == 0
    seen = set()
    for i in range(1, n):
        p = par[i]
        assert 0 <= p < i
        assert dep[i] == dep[p] + 1 <= depth_max
        rank = int(np.nonzero(tok[p] == tk[i])[0][0])
        assert (p, rank) not in seen
        seen.add((p, rank))
        assert sc[i] == np.float32(sc[p] + logp[p, rank])
    assert math.ceil((n - 1) / w) <= r["rounds"] <= n - 1 or n == 1
    if n == budget and logp.shape[1] >= w:
        # the heap never holds fewer than w candidates: every round but the last is full
        assert r["rounds"] == math.ceil((budget - 1) / w)
        for r0 in range(1, n, w):                   # within a round: best first
            assert np.all(np.diff(sc[r0:min(n, r0 + w)]) <= 0)


@pytest.mark.parametrize("w,budget,K,depth_max", [(1, 40, 4, 12), (4, 64, 8, 12),
                                                   (8, 64, 8, 6), (16, 129, 8, 16),
                                                   (7, 50, 3, 30), (64, 256, 16, 30)])
def test_invariants_random_tables(w, budget, K, depth_max):
    rng = np.random.default_rng(budget * 31 + w)
    logp = -rng.exponential(1.5, (budget, K)).astype(np.float32)
    tok = np.stack([rng.permutation(1000)[:K] for _ in range(budget)]).astype(np.int32)
    r = tb.build_one(5, logp, tok, budget, w, depth_max)
    check_invariants(r, logp, tok, budget, w, depth_max)


def test_heap_runs_dry_under_the_depth_cap():
    logp, tok = uniform_table([-0.1, -0.2, -0.3], 10)
    r = tb.build_one(0, logp, tok, 10, 2, 1)
    assert r["n_nodes"] == 4 and r["rounds"] == 2
    assert r["depth"].tolist() == [0, 1, 1, 1]


def test_budget_one_is_the_root_alone():
    logp, tok = uniform_table([-0.1, -0.2], 1)
    r = tb.build_one(9, logp, tok, 1, 4, 5)
    assert r["n_nodes"] == 1 and r["rounds"] == 0 and r["token"].tolist() == [9]


def test_batch_wrapper_pads():
    logp, tok, _ = load_golden()
    out = tb.build(np.array([100, 100]), np.stack([logp, logp]), np.stack([tok, tok]), 6, 2, 3)
    assert out["n_nodes"].tolist() == [6, 6]
    out = tb.build(np.array([1]), logp[None, :, :], tok[None], 6, 2, 0)
    assert out["n_nodes"].tolist() == [1]
    assert out["parent"][0].tolist() == [-1, -1, -1, -1, -1, -1]
    assert out["token"][0].tolist() == [1, -1, -1, -1, -1, -1]
