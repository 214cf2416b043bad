"""Top-w best-first draft-tree construction — TEST INFRASTRUCTURE ONLY (CPU oracle).

"Trees from Marginals" (Technisches Resümee, Methodik 2 "Baumerstellung"): the
drafter's tree is built best-first from a heap of candidate continuations, but
instead of expanding one node per step, the w best candidates are taken from the
heap together and expanded together, so a tree of B nodes takes about B / w
sequential steps.  This module states that procedure plainly with Python's
heapq, one sequence at a time.  Only the tests may call it.

Readings where the page is silent (also listed in the design notes):
  * a candidate's priority is its path log-probability: the parent's score plus
    the drafter's log-probability of the continuation, added in fp32 (the
    product of draft probabilities along the path, in log form);
  * ties go to the candidate with the smaller id = parent slot * K + rank;
  * the drafter's top-K continuations of the node in tree slot i are given as a
    table row (child_logp[i], child_token[i]); in a live system that row is
    the drafter's output for slot i, produced between two rounds;
  * the root (slot 0, score 0, depth 0) is the last committed token; every node
    taken from the heap is expanded at the end of its round unless the tree is
    already full, and children deeper than depth_max are never offered;
  * a round takes min(w, budget - size) candidates (fewer if the heap runs
    dry); `rounds` counts the rounds that took at least one candidate.

Pins (tests/test_tree_build_oracle.py): a hand-worked fixture in tests/golden/,
w = 1 equal to the brute-force best B nodes of the candidate tree (score
multiset), level order when w covers whole levels, total score of w = 1 never
below any other w, and per-node invariants.
"""
from __future__ import annotations

import heapq

import numpy as np


def build_one(root_token: int, child_logp: np.ndarray, child_token: np.ndarray, budget: int,
              w: int, depth_max: int):
    """One sequence.  child_logp/child_token: [budget][K] (row i = slot i's candidates).
    Returns dict(parent, token, score (float32), depth, n_nodes, rounds), arrays of length
    n_nodes (unpadded)."""
    child_logp = np.asarray(child_logp, np.float32)
    K = child_logp.shape[1]
    parent, token, score, depth = [-1], [int(root_token)], [np.float32(0.0)], [0]
    heap: list[tuple[np.float32, int]] = []

    def expand(i: int):
        if depth[i] + 1 > depth_max:
            return
        for r in range(K):
            s = np.float32(score[i] + child_logp[i, r])        # one fp32 addition
            heapq.heappush(heap, (np.float32(-s), i * K + r))  # best score, then smaller id

    expand(0)
    rounds = 0
    while len(parent) < budget and heap:
        take = min(w, budget - len(parent))
        new = []
        for _ in range(take):
            if not heap:
                break
            neg, cid = heapq.heappop(heap)
            i, r = divmod(cid, K)
            parent.append(i)
            token.append(int(child_token[i, r]))
            score.append(np.float32(-neg))
            depth.append(depth[i] + 1)
            new.append(len(parent) - 1)
        rounds += 1
        if len(parent) < budget:
            for n in new:
                expand(n)
    return dict(parent=np.array(parent, np.int32), token=np.array(token, np.int32),
                score=np.array(score, np.float32), depth=np.array(depth, np.int32),
                n_nodes=len(parent), rounds=rounds)


def build(root_token, child_logp, child_token, budget: int, w: int, depth_max: int):
    """A batch: root_token [B], child_logp / child_token [B][budget][K].  Returns padded
    arrays parent/token/depth [B][budget] (-1 past n_nodes), score [B][budget] (0 past
    n_nodes), n_nodes [B], rounds [B]."""
    B = len(root_token)
    out = dict(parent=np.full((B, budget), -1, np.int32), token=np.full((B, budget), -1, np.int32),
               score=np.zeros((B, budget), np.float32), depth=np.full((B, budget), -1, np.int32),
               n_nodes=np.zeros(B, np.int32), rounds=np.zeros(B, np.int32))
    for b in range(B):
        r = build_one(root_token[b], child_logp[b], child_token[b], budget, w, depth_max)
        n = r["n_nodes"]
        for key in ("parent", "token", "score", "depth"):
            out[key][b, :n] = r[key]
        out["n_nodes"][b] = n
        out["rounds"][b] = r["rounds"]
    return out
