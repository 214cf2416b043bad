"""Pins for the fp64 oracle, against things other than the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped gate, a
wrong sign, a transposed state, the wrong parent, a missing root step) fails
at least one of them:
  * hand-worked fixtures (tests/golden/) for prep, acceptance and a scalar chain;
  * closed forms: b = 0 is pure decay; d_k = d_v = 1 is a product of scalars;
  * a chain equals token-by-token GDN (the textbook recurrence);
  * the delta-rule write invariant S_n^T k_n = (1 - b) a S_p^T k_n + b v_n;
  * outputs ignore every non-ancestor node; relabelling nodes permutes outputs;
  * an independent tree solve (the masked triangular system) agrees to 1e-12;
  * committing then verifying the next tree equals one verify of the joined tree;
  * prep and accept against brute force on random valid and broken trees.
"""
import math
import os

import numpy as np
import pytest

import oracle
from tree_speculative_decoding_gated_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_cases(name):
    cases, cur = {}, None
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = cases.setdefault(vals[0], {})
            continue
        if cur is None:
            cur = cases.setdefault("", {})
        cur[key] = [float(x) if "." in x else int(x) for x in vals]
    return cases


def rand_inputs(rng, T, H_qk=1, H_v=1, dk=4, dv=3, unit=True, B=1):
    q = rng.standard_normal((T, H_qk, dk))
    k = rng.standard_normal((T, H_qk, dk))
    if unit:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H_v, dv))
    g = -np.log1p(np.exp(rng.standard_normal((T, H_v))))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, H_v))))
    S0 = 0.3 * rng.standard_normal((B, H_v, dk, dv))
    return q, k, v, g, b, S0


def one_tree(parent):
    parent = np.asarray(parent, np.int32)
    return np.array([0, len(parent)], np.int32), parent


def depth_of(parent, n):
    d = 0
    while parent[n] >= 0:
        n = parent[n]
        d += 1
    return d


def ancestors(parent, n):
    out = [n]
    while parent[n] >= 0:
        n = parent[n]
        out.append(n)
    return out


# ---------------------------------------------------------------- fixtures
@pytest.mark.parametrize("case", ["toy", "relabelled"])
def test_prep_hand_worked(case):
    c = read_cases("toy_tree_prep.txt")[case]
    cu, par = one_tree(c["parent"])
    out = oracle.prep(cu, par, n_max=7, depth_max=2)
    assert out["status"].tolist() == [0]
    assert out["depth"].tolist() == c["depth"]
    assert out["order"].tolist() == c["order"]
    assert out["pos"].tolist() == c["pos"]
    assert out["anc"][:, 0].astype(np.int64).tolist() == c["anc"]


@pytest.mark.parametrize("case", ["a", "b", "c", "d"])
def test_accept_hand_worked(case):
    c = read_cases("toy_accept.txt")[case]
    cu, par = one_tree(synth.TOY_PARENT)
    out = oracle.accept(cu, par, 7, 2, c["draft"], c["target"])
    assert out["accept_node"].tolist() == c["accept_node"]
    assert out["accept_len"].tolist() == c["accept_len"]
    assert out["path"][0].tolist() == c["path"]


def test_scalar_chain_hand_worked():
    c = read_cases("scalar_chain.txt")[""]
    cu, par = one_tree(c["parent"])
    T = len(par)
    sh = lambda x: np.asarray(x, np.float64).reshape(T, 1, 1)
    q, k, v = sh(c["q"]), sh(c["k"]), sh(c["v"])
    g = np.log(np.asarray(c["a"], np.float64)).reshape(T, 1)
    b = np.asarray(c["b"], np.float64).reshape(T, 1)
    S0 = np.asarray(c["S0"], np.float64).reshape(1, 1, 1, 1)
    o = oracle.verify(cu, par, T, T, q, k, v, g, b, S0)
    np.testing.assert_allclose(o[:, 0, 0], c["o"], rtol=0, atol=1e-15)
    for n in range(T):
        S = oracle.commit(cu, par, T, T, k, v, g, b, S0, np.array([n], np.int32))
        assert abs(S[0, 0, 0, 0] - c["S"][n]) < 1e-15


# ---------------------------------------------------------------- closed forms
def test_beta_zero_is_pure_decay():
    """b = 0: S_n = exp(G_n) S0 (the diagonal-SSM special case), so o_n = exp(G_n) S0^T q_n."""
    rng = np.random.default_rng(1)
    par = synth.random_recursive_tree(rng, 20, 6)
    cu, par = one_tree(par)
    q, k, v, g, b, S0 = rand_inputs(rng, 20, H_qk=1, H_v=2, dk=5, dv=4)
    b[:] = 0.0
    o = oracle.verify(cu, par, 20, 20, q, k, v, g, b, S0)
    for n in range(20):
        for h in range(2):
            G = sum(g[s, h] for s in ancestors(par, n))
            want = math.exp(G) * S0[0, h].T @ q[n, 0]
            np.testing.assert_allclose(o[n, h], want, rtol=1e-12, atol=1e-14)


def test_scalar_state_closed_form():
    """d_k = d_v = 1, k = +-1: S_n = sum_s (prod_{r after s} a_r (1 - b_r)) b_s k_s v_s + prod a(1-b) S0."""
    rng = np.random.default_rng(2)
    par = synth.random_recursive_tree(rng, 25, 8)
    cu, par = one_tree(par)
    T = 25
    q = rng.standard_normal((T, 1, 1))
    k = rng.choice([-1.0, 1.0], size=(T, 1, 1))
    v = rng.standard_normal((T, 1, 1))
    g = -np.log1p(np.exp(rng.standard_normal((T, 1))))
    b = rng.random((T, 1))
    S0 = rng.standard_normal((1, 1, 1, 1))
    o = oracle.verify(cu, par, T, T, q, k, v, g, b, S0)
    for n in range(T):
        path = ancestors(par, n)[::-1]               # root first
        decay = lambda nodes: np.prod([math.exp(g[r, 0]) * (1 - b[r, 0]) for r in nodes])
        S = decay(path) * S0[0, 0, 0, 0]
        for i, s in enumerate(path):
            S += decay(path[i + 1:]) * b[s, 0] * k[s, 0, 0] * v[s, 0, 0]
        assert abs(o[n, 0, 0] - S * q[n, 0, 0]) < 1e-12


def test_chain_equals_sequential_gdn():
    """A chain tree is ordinary token-by-token GDN decoding."""
    rng = np.random.default_rng(3)
    T, dk, dv = 12, 6, 5
    cu, par = one_tree(synth.chain_tree(T))
    q, k, v, g, b, S0 = rand_inputs(rng, T, H_qk=1, H_v=1, dk=dk, dv=dv)
    o = oracle.verify(cu, par, T, T, q, k, v, g, b, S0)
    S = S0[0, 0].copy()
    for t in range(T):
        kt, vt, a, bt = k[t, 0], v[t, 0], math.exp(g[t, 0]), b[t, 0]
        S = a * (np.eye(dk) - bt * np.outer(kt, kt)) @ S + bt * np.outer(kt, vt)
        np.testing.assert_allclose(o[t, 0], S.T @ q[t, 0], rtol=1e-12, atol=1e-13)
    Sc = oracle.commit(cu, par, T, T, k, v, g, b, S0, np.array([T - 1], np.int32))
    np.testing.assert_allclose(Sc[0, 0], S, rtol=1e-12, atol=1e-13)


def test_delta_rule_write_invariant():
    """With unit k: S_n^T k_n = (1 - b_n) a_n S_p^T k_n + b_n v_n; a = b = 1 stores v exactly."""
    rng = np.random.default_rng(4)
    T = 15
    cu, par = one_tree(synth.random_recursive_tree(rng, T, 5))
    q, k, v, g, b, S0 = rand_inputs(rng, T, H_qk=1, H_v=1, dk=7, dv=3)
    for n in range(1, T):
        p = par[n]
        Sn = oracle.commit(cu, par, T, T, k, v, g, b, S0, np.array([n], np.int32))[0, 0]
        Sp = oracle.commit(cu, par, T, T, k, v, g, b, S0, np.array([p], np.int32))[0, 0]
        a = math.exp(g[n, 0])
        want = (1 - b[n, 0]) * a * Sp.T @ k[n, 0] + b[n, 0] * v[n, 0]
        np.testing.assert_allclose(Sn.T @ k[n, 0], want, rtol=1e-12, atol=1e-13)
    g1, b1 = np.zeros_like(g), np.ones_like(b)
    for n in range(T):
        Sn = oracle.commit(cu, par, T, T, k, v, g1, b1, S0, np.array([n], np.int32))[0, 0]
        np.testing.assert_allclose(Sn.T @ k[n, 0], v[n, 0], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- invariances
def test_non_ancestor_edits_do_not_change_output():
    rng = np.random.default_rng(5)
    T = 30
    cu, par = one_tree(synth.random_recursive_tree(rng, T, 7))
    q, k, v, g, b, S0 = rand_inputs(rng, T, H_qk=1, H_v=2, dk=4, dv=4)
    o = oracle.verify(cu, par, T, T, q, k, v, g, b, S0)
    for n in [3, 11, 29]:
        keep = set(ancestors(par, n))
        other = [i for i in range(T) if i not in keep]
        q2, k2, v2, g2, b2 = (x.copy() for x in (q, k, v, g, b))
        for x in (q2, k2, v2):
            x[other] = rng.standard_normal(x[other].shape)
        g2[other] = -rng.random(g2[other].shape)
        b2[other] = rng.random(b2[other].shape)
        o2 = oracle.verify(cu, par, T, T, q2, k2, v2, g2, b2, S0)
        assert np.array_equal(o2[n], o[n])


def test_relabelling_permutes_outputs():
    rng = np.random.default_rng(6)
    T = 24
    cu, par = one_tree(synth.random_recursive_tree(rng, T, 6))
    q, k, v, g, b, S0 = rand_inputs(rng, T, H_qk=2, H_v=4, dk=4, dv=3)
    o = oracle.verify(cu, par, T, T, q, k, v, g, b, S0)
    perm = rng.permutation(T)            # new label of old node i is perm[i]
    inv = np.argsort(perm)
    par2 = np.array([perm[par[inv[j]]] if par[inv[j]] >= 0 else -1 for j in range(T)], np.int32)
    o2 = oracle.verify(cu, par2, T, T, q[inv], k[inv], v[inv], g[inv], b[inv], S0)
    assert np.array_equal(o2, o[inv])


# ---------------------------------------------------------------- tree solve
def tree_solve(parent, q, k, v, g, b, S0, H_qk, H_v):
    """Masked triangular-solve form, written independently: (I + X) U = diag(b)(V - diag(e^G) K S0),
    O = diag(e^G) Q S0 + Y U, with X_ns = b_n e^{G_n-G_s} k_n.k_s (s strict ancestor),
    Y_ns = e^{G_n-G_s} q_n.k_s (s ancestor or self).  Also returns every node's state."""
    T = len(parent)
    dep = [depth_of(parent, n) for n in range(T)]
    topo = sorted(range(T), key=lambda n: (dep[n], n))
    O = np.zeros((T, H_v, v.shape[-1]))
    states = {}
    for h in range(H_v):
        qh = h // (H_v // H_qk)
        Q, K, V = q[:, qh], k[:, qh], v[:, h]
        G = np.array([sum(g[s, h] for s in ancestors(parent, n)) for n in range(T)])
        R = b[:, h, None] * (V - np.exp(G)[:, None] * (K @ S0[h]))
        U = np.zeros_like(R)
        for n in topo:
            U[n] = R[n]
            for s in ancestors(parent, n)[1:]:
                U[n] -= b[n, h] * math.exp(G[n] - G[s]) * (K[n] @ K[s]) * U[s]
        for n in range(T):
            O[n, h] = math.exp(G[n]) * (Q[n] @ S0[h])
            S = math.exp(G[n]) * S0[h]
            for s in ancestors(parent, n):
                O[n, h] += math.exp(G[n] - G[s]) * (Q[n] @ K[s]) * U[s]
                S = S + math.exp(G[n] - G[s]) * np.outer(K[s], U[s])
            states[(n, h)] = S
    return O, states


@pytest.mark.parametrize("seed", [7, 8, 9])
def test_tree_solve_agrees_with_path_replay(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(2, 41))
    cu, par = one_tree(synth.random_recursive_tree(rng, T, int(rng.integers(1, 10))))
    q, k, v, g, b, S0 = rand_inputs(rng, T, H_qk=2, H_v=4, dk=6, dv=5)
    o = oracle.verify(cu, par, T, T, q, k, v, g, b, S0)
    O, states = tree_solve(par, q, k, v, g, b, S0[0], 2, 4)
    np.testing.assert_allclose(o, O, rtol=1e-12, atol=1e-12)
    n = int(rng.integers(T))
    S = oracle.commit(cu, par, T, T, k, v, g, b, S0, np.array([n], np.int32))
    for h in range(4):
        np.testing.assert_allclose(S[0, h], states[(n, h)], rtol=1e-12, atol=1e-12)


def test_commit_then_verify_equals_joined_tree():
    """Rollback-free two-step consistency: commit(accepted node of tree 1) then verify(tree 2)
    equals verifying tree 2 hung below the accepted path of tree 1, from S0."""
    rng = np.random.default_rng(10)
    T1, T2 = 18, 14
    p1 = synth.random_recursive_tree(rng, T1, 5)
    p2 = synth.random_recursive_tree(rng, T2, 5)
    q, k, v, g, b, S0 = rand_inputs(rng, T1 + T2, H_qk=1, H_v=2, dk=5, dv=4)
    cu1, par1 = one_tree(p1)
    n_star = 13
    S1 = oracle.commit(cu1, par1, T1, T1, k[:T1], v[:T1], g[:T1], b[:T1], S0,
                       np.array([n_star], np.int32))
    cu2, par2 = one_tree(p2)
    sl = slice(T1, T1 + T2)
    o2 = oracle.verify(cu2, par2, T2, T2, q[sl], k[sl], v[sl], g[sl], b[sl], S1)
    path = ancestors(p1, n_star)[::-1]
    L = len(path)
    joined = list(range(-1, L - 1)) + [int(x) + L if x >= 0 else L - 1 for x in p2]
    rows = path + list(range(T1, T1 + T2))
    cuj, parj = one_tree(joined)
    oj = oracle.verify(cuj, parj, L + T2, L + T2, q[rows], k[rows], v[rows], g[rows], b[rows], S0)
    np.testing.assert_allclose(o2, oj[L:], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- prep / accept brute force
def brute_status(parent, n_max, depth_max):
    N = len(parent)
    if N > n_max:
        return 1
    if any(p < -1 or p >= N or p == i for i, p in enumerate(parent)):
        return 2
    if N and sum(p == -1 for p in parent) != 1:
        return 3
    for i in range(N):
        seen, j = set(), i
        while parent[j] != -1:
            if j in seen:
                return 4
            seen.add(j)
            j = parent[j]
    if any(depth_of(parent, i) > depth_max for i in range(N)):
        return 5
    return 0


def random_batch(rng, B, broken=True):
    parents = []
    for _ in range(B):
        N = int(rng.integers(0, 70))
        par = synth.random_recursive_tree(rng, N, int(rng.integers(1, 20))) if N else np.zeros(0, np.int32)
        if N and broken and rng.random() < 0.5:
            kind = rng.integers(4)
            i = int(rng.integers(N))
            if kind == 0:
                par[i] = N + int(rng.integers(3))
            elif kind == 1 and N > 1:
                par[max(i, 1)] = -1
            elif kind == 2 and N > 2:
                # hang a non-root node below one of its own descendants: a cycle, one root left
                kids = [j for j in range(2, N) if par[j] >= 1]
                if kids:
                    j = kids[int(rng.integers(len(kids)))]
                    par[par[j]] = j
            else:
                par[i] = i
        if N > 1 and rng.random() < 0.5:          # scramble labels
            perm = rng.permutation(N)
            inv = np.argsort(perm)
            par = np.array([perm[par[inv[j]]] if 0 <= par[inv[j]] < N else par[inv[j]]
                            for j in range(N)], np.int32)
        parents.append(par)
    return parents


def test_prep_brute_force():
    rng = np.random.default_rng(11)
    seen = set()
    for trial in range(40):
        parents = random_batch(rng, 6)
        n_max, depth_max = 64, int(rng.integers(3, 18))
        trees = synth.pack_trees(parents, n_max, depth_max)
        out = oracle.prep(trees.cu_nodes, trees.parent, n_max, depth_max)
        for bi, par in enumerate(parents):
            lo, N = int(trees.cu_nodes[bi]), len(par)
            st = brute_status(par, n_max, depth_max)
            assert out["status"][bi] == st
            seen.add(st)
            sl = slice(lo, lo + N)
            if st != 0:
                assert (out["depth"][sl] == -1).all() and (out["anc"][sl] == 0).all()
                continue
            dep = np.array([depth_of(par, i) for i in range(N)])
            assert out["depth"][sl].tolist() == dep.tolist()
            order = out["order"][sl]
            pos = out["pos"][sl]
            assert sorted(order.tolist()) == list(range(N))
            assert (pos[order] == np.arange(N)).all()
            keys = [(dep[i], i) for i in order]
            assert keys == sorted(keys)
            for n in range(N):
                want = sum(1 << int(pos[s]) for s in ancestors(par, n))
                row = out["anc"][lo + pos[n]]
                got = sum(int(w) << (64 * j) for j, w in enumerate(row))
                assert got == want
    assert seen >= {0, 2, 3, 4, 5}


def test_accept_brute_force():
    rng = np.random.default_rng(12)
    for trial in range(30):
        parents = random_batch(rng, 5)
        n_max, depth_max = 64, 19
        trees = synth.pack_trees(parents, n_max, depth_max)
        T = trees.T
        draft = rng.integers(0, 3, T).astype(np.int32)
        target = np.where(rng.random(T) < 0.7, draft, rng.integers(0, 3, T)).astype(np.int32)
        out = oracle.accept(trees.cu_nodes, trees.parent, n_max, depth_max, draft, target)
        for bi, par in enumerate(parents):
            lo, N = int(trees.cu_nodes[bi]), len(par)
            if brute_status(par, n_max, depth_max) != 0 or N == 0:
                assert out["accept_node"][bi] == -1 and out["accept_len"][bi] == 0
                assert (out["path"][bi] == -1).all()
                continue
            # dynamic programme over a topological order, independent of path enumeration
            dep = [depth_of(par, i) for i in range(N)]
            ok = [False] * N
            for n in sorted(range(N), key=lambda i: dep[i]):
                ok[n] = par[n] == -1 or (ok[par[n]] and draft[lo + n] == target[lo + n])
            best = min((i for i in range(N) if ok[i]), key=lambda i: (-dep[i], i))
            assert out["accept_node"][bi] == best
            assert out["accept_len"][bi] == dep[best] + 1
            path = ancestors(par, best)[::-1]
            assert out["path"][bi].tolist() == path + [-1] * (depth_max + 1 - len(path))


def test_invalid_tree_outputs():
    cu = np.array([0, 3, 6], np.int32)
    par = np.array([-1, 0, 1, -1, -1, 0], np.int32)       # second sequence: two roots
    rng = np.random.default_rng(13)
    q, k, v, g, b, S0 = rand_inputs(rng, 6, dk=3, dv=2, B=2)
    o = oracle.verify(cu, par, 8, 8, q, k, v, g, b, S0)
    assert (o[3:] == 0).all() and (o[:3] != 0).any()
    S = oracle.commit(cu, par, 8, 8, k, v, g, b, S0, np.array([2, 1], np.int32))
    assert np.array_equal(S[1], S0[1])


def test_synth_is_deterministic():
    a = synth.make_problem("cfg3")
    b = synth.make_problem("cfg3")
    assert np.array_equal(a.trees.parent, b.trees.parent)
    assert np.array_equal(a.inputs.k, b.inputs.k) and np.array_equal(a.S0, b.S0)
    assert np.array_equal(a.target_ids, b.target_ids)
    assert (synth.round_bf16(a.inputs.q) == a.inputs.q).all()
    t = synth.make_trees(synth.CONFIGS["cfg4"])
    assert t.sizes().tolist() == [17, 129] * 32
    st = oracle.prep(t.cu_nodes, t.parent, t.n_max, t.depth_max)["status"]
    assert (st == 0).all()
