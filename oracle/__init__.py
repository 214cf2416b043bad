"""fp64 CPU oracle for rollback-free GDN tree verification — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package; the library's product path never does.  The
arithmetic lives in ``tgdn_oracle.cpp`` (path replay of the GDN update eq. from
"Trees from Marginals", Technisches Resümee, Methodik 3); this module only
marshals numpy arrays into it.

Two further parts of the pages' decode step have oracles of their own, written
in plain Python: ``tree_build.py`` (top-w best-first draft-tree construction,
Methodik 2) and ``tree_attention.py`` (ancestor-masked attention for the
verifier's attention layers); each is pinned by its own test module.

Pins: every function here is checked in ``tests/test_oracle.py`` against
things other than itself — closed forms (b = 0 pure decay, the scalar
d_k = d_v = 1 product form), a chain equal to token-by-token GDN, the
delta-rule write invariant, non-ancestor and relabelling invariance, an
independent tree solve, brute-force prep/accept and a hand-checked toy tree.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

I32 = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
U64 = np.ctypeslib.ndpointer(np.uint64, flags="C_CONTIGUOUS")
F64 = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
c_int = ctypes.c_int


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_prep.argtypes = [c_int, I32, I32, c_int, c_int, c_int, I32, I32, I32, U64, I32]
        L.oracle_accept.argtypes = [c_int, I32, I32, c_int, c_int, I32, I32, I32, I32, I32]
        L.oracle_verify.argtypes = [c_int, I32, I32, c_int, c_int, c_int, c_int, c_int, c_int,
                                    F64, F64, F64, F64, F64, F64, F64, c_int]
        L.oracle_commit.argtypes = [c_int, I32, I32, c_int, c_int, c_int, c_int, c_int, c_int,
                                    F64, F64, F64, F64, F64, I32, F64, c_int]
        for f in (L.oracle_prep, L.oracle_accept, L.oracle_verify, L.oracle_commit):
            f.restype = c_int
        _lib = L
    return _lib


def _i32(x):
    return np.ascontiguousarray(x, dtype=np.int32)


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def words_for(n_max: int) -> int:
    return max(1, (n_max + 63) // 64)


def prep(cu_nodes, parent, n_max: int, depth_max: int):
    """Returns dict(depth, order, pos, anc[T, words] uint64, status[B])."""
    cu, par = _i32(cu_nodes), _i32(parent)
    B, T, W = len(cu) - 1, len(par), words_for(n_max)
    out = dict(depth=np.empty(T, np.int32), order=np.empty(T, np.int32),
               pos=np.empty(T, np.int32), anc=np.zeros((T, W), np.uint64),
               status=np.empty(B, np.int32))
    rc = lib().oracle_prep(B, cu, par, n_max, depth_max, W, out["depth"], out["order"],
                           out["pos"], out["anc"], out["status"])
    if rc != 0:
        raise ValueError("oracle_prep: malformed batch description")
    return out


def accept(cu_nodes, parent, n_max: int, depth_max: int, draft_ids, target_ids):
    """Returns dict(accept_node[B], accept_len[B], path[B, depth_max + 1])."""
    cu, par = _i32(cu_nodes), _i32(parent)
    B = len(cu) - 1
    out = dict(accept_node=np.empty(B, np.int32), accept_len=np.empty(B, np.int32),
               path=np.empty((B, depth_max + 1), np.int32))
    lib().oracle_accept(B, cu, par, n_max, depth_max, _i32(draft_ids), _i32(target_ids),
                        out["accept_node"], out["accept_len"], out["path"])
    return out


def _dims(q, v, S0):
    T, H_qk, dk = q.shape
    _, H_v, dv = v.shape
    return T, H_qk, H_v, dk, dv


def verify(cu_nodes, parent, n_max, depth_max, q, k, v, g, b, S0, nthreads: int = 0,
           return_threads: bool = False):
    """Per-node outputs o[T, H_v, dv] (fp64) by replaying each node's root path."""
    cu, par = _i32(cu_nodes), _i32(parent)
    T, H_qk, H_v, dk, dv = _dims(q, v, S0)
    o = np.zeros((T, H_v, dv), np.float64)
    used = lib().oracle_verify(len(cu) - 1, cu, par, n_max, depth_max, H_qk, H_v, dk, dv,
                               _f64(q), _f64(k), _f64(v), _f64(g), _f64(b), _f64(S0), o,
                               nthreads)
    return (o, used) if return_threads else o


def commit(cu_nodes, parent, n_max, depth_max, k, v, g, b, S0, accept_node, nthreads: int = 0):
    """Committed states S[B, H_v, dk, dv] (fp64): the replayed state at each accepted node."""
    cu, par = _i32(cu_nodes), _i32(parent)
    B = len(cu) - 1
    _, H_qk, dk = k.shape
    _, H_v, dv = v.shape
    S = np.zeros((B, H_v, dk, dv), np.float64)
    lib().oracle_commit(B, cu, par, n_max, depth_max, H_qk, H_v, dk, dv, _f64(k), _f64(v),
                        _f64(g), _f64(b), _f64(S0), _i32(accept_node), S, nthreads)
    return S


def problem_prep(p):
    t = p.trees
    return prep(t.cu_nodes, t.parent, t.n_max, t.depth_max)


def problem_verify(p, nthreads: int = 0):
    t, i = p.trees, p.inputs
    return verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v, i.g, i.b, p.S0,
                  nthreads)


def problem_accept(p):
    t = p.trees
    return accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, p.draft_ids, p.target_ids)


def problem_commit(p, accept_node, nthreads: int = 0):
    t, i = p.trees, p.inputs
    return commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b, p.S0,
                  accept_node, nthreads)
