"""Seeded synthetic inputs for rollback-free GDN tree verification.

This module is shared by the tests and the benchmark.  It
holds none of the method's arithmetic: it only draws trees, token ids and the
per-node q/k/v/gate/beta tensors plus the committed state S0, with the shapes
and distributions of the workloads studied on the pages of "Trees from
Marginals: Autoregressive drafting with factorized priors" (Technisches
Resümee, Methodik 3 and Experimentelle Ergebnisse): a Qwen3-style hybrid model
with H_qk = 16 query/key heads, H_v = 32 value heads and d_k = d_v = 128.

Recipe (all draws from numpy PCG64 through SeedSequence, so any
(config, step, layer) slice can be regenerated on its own):
  * q, k ~ N(0, 1), L2-normalised over d_k, then rounded to bf16 (bf16 configs);
  * v ~ N(0, 1), rounded to bf16 (bf16 configs);
  * g = -softplus(N(0, 1)) is the log-gate (a = exp(g) in (0, 1));
  * b = sigmoid(N(0, 1)) is the write strength;
  * S0 ~ N(0, sigma) with sigma = 0.1 (toy) or 0.02 (model shapes);
  * draft ids uniform over the vocabulary (distinct within a depth for top-M
    trees); the verifier id equals the draft id with probability 0.7, else it
    is another uniform id.  The toy draws both uniformly from [0, 8).

Seeds: topology 20260709 + c, tensors 20260709 + c + 1000, ids
20260709 + c + 2000, where c is the config number (toy = 1 ... stack = 5),
each extended by the (step, layer) key.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np

BASE_SEED = 20260709
VOCAB = 151_936


# --------------------------------------------------------------------------
# workload presets
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Config:
    name: str
    number: int
    B: int
    H_qk: int
    H_v: int
    dk: int
    dv: int
    io: str                  # "bf16" or "f32"
    tree: str                # "toy", "topm", "random", "mixed"
    n_nodes: int = 0         # nodes per tree for "random" (root included)
    depth_cap: int = 16
    M: int = 0               # width of top-M trees
    depth: int = 0           # depth of top-M trees / chains
    s0_sigma: float = 0.02
    vocab: int = VOCAB
    p_match: float = 0.7
    layers: int = 1
    steps: int = 1

    @property
    def n_max(self) -> int:
        if self.tree == "toy":
            return 7
        if self.tree == "topm":
            return 1 + self.M * self.depth
        if self.tree == "random":
            return self.n_nodes
        if self.tree == "mixed":
            return max(1 + self.depth, 1 + self.M * self.depth)
        raise ValueError(self.tree)

    @property
    def depth_max(self) -> int:
        if self.tree == "toy":
            return 2
        if self.tree in ("topm", "mixed"):
            return self.depth
        return self.depth_cap


CONFIGS = {
    # complete binary tree of 7 nodes, one 16x16 head, fp32 path
    "toy": Config("toy", 1, B=1, H_qk=1, H_v=1, dk=16, dv=16, io="f32",
                  tree="toy", s0_sigma=0.1, vocab=8),
    # one layer, one sequence: top-4 tree of depth 8 (32 nodes + root)
    "cfg2": Config("cfg2", 2, B=1, H_qk=16, H_v=32, dk=128, dv=128, io="bf16",
                   tree="topm", M=4, depth=8),
    # one layer, 16 sequences of 64-node random recursive trees, depth <= 16
    "cfg3": Config("cfg3", 3, B=16, H_qk=16, H_v=32, dk=128, dv=128, io="bf16",
                   tree="random", n_nodes=64, depth_cap=16),
    # one layer, 64 sequences alternating a 16-token chain (17 nodes with the
    # root) and a top-8 tree of depth 16 (129 nodes with the root)
    "cfg4": Config("cfg4", 4, B=64, H_qk=16, H_v=32, dk=128, dv=128, io="bf16",
                   tree="mixed", M=8, depth=16),
    # 36-layer stack, 32 sequences of 64-node random trees, depth <= 12, 50 steps
    "cfg5": Config("cfg5", 5, B=32, H_qk=16, H_v=32, dk=128, dv=128, io="bf16",
                   tree="random", n_nodes=64, depth_cap=12, layers=36, steps=50),
}


def rng_for(cfg: Config, stream: int, *key: int) -> np.random.Generator:
    """Counter-style generator: one independent PCG64 per (config, stream, key)."""
    seed = BASE_SEED + cfg.number + stream
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


TOPOLOGY, TENSORS, IDS = 0, 1000, 2000


# --------------------------------------------------------------------------
# trees (parent arrays: local index of the parent, -1 for the root)
# --------------------------------------------------------------------------
def chain_tree(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def random_recursive_tree(rng: np.random.Generator, n: int, depth_cap: int) -> np.ndarray:
    """Node i picks its parent uniformly among earlier nodes of depth < depth_cap."""
    parent = np.full(n, -1, np.int32)
    depth = np.zeros(n, np.int32)
    for i in range(1, n):
        cand = np.nonzero(depth[:i] < depth_cap)[0]
        p = int(cand[rng.integers(len(cand))])
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def top_m_tree(rng: np.random.Generator, M: int, depth: int) -> np.ndarray:
    """Root, then M nodes per depth, each child of a uniformly drawn node one level up."""
    parent = [-1]
    prev = [0]
    for _ in range(depth):
        cur = []
        for _ in range(M):
            parent.append(int(prev[rng.integers(len(prev))]))
            cur.append(len(parent) - 1)
        prev = cur
    return np.asarray(parent, np.int32)


TOY_PARENT = np.array([-1, 0, 0, 1, 1, 2, 2], np.int32)


def tree_depths(parent: np.ndarray) -> np.ndarray:
    """Depth by walking parents (used only to shape generated ids)."""
    d = np.zeros(len(parent), np.int32)
    for i in range(len(parent)):
        j, h = i, 0
        while parent[j] >= 0:
            j = parent[j]
            h += 1
        d[i] = h
    return d


@dataclass
class Trees:
    cu_nodes: np.ndarray     # int32 [B+1]
    parent: np.ndarray       # int32 [T], local parent index, -1 = root
    n_max: int
    depth_max: int

    @property
    def B(self) -> int:
        return len(self.cu_nodes) - 1

    @property
    def T(self) -> int:
        return int(self.cu_nodes[-1])

    def sizes(self) -> np.ndarray:
        return np.diff(self.cu_nodes)


def pack_trees(parents: list[np.ndarray], n_max: int, depth_max: int) -> Trees:
    cu = np.zeros(len(parents) + 1, np.int32)
    cu[1:] = np.cumsum([len(p) for p in parents])
    par = np.concatenate(parents).astype(np.int32) if parents else np.zeros(0, np.int32)
    return Trees(cu, par, n_max, depth_max)


def make_trees(cfg: Config, step: int = 0) -> Trees:
    rng = rng_for(cfg, TOPOLOGY, step)
    if cfg.tree == "toy":
        parents = [TOY_PARENT.copy() for _ in range(cfg.B)]
    elif cfg.tree == "topm":
        parents = [top_m_tree(rng, cfg.M, cfg.depth) for _ in range(cfg.B)]
    elif cfg.tree == "random":
        parents = [random_recursive_tree(rng, cfg.n_nodes, cfg.depth_cap) for _ in range(cfg.B)]
    elif cfg.tree == "mixed":
        parents = [chain_tree(cfg.depth + 1) if i % 2 == 0 else top_m_tree(rng, cfg.M, cfg.depth)
                   for i in range(cfg.B)]
    else:
        raise ValueError(cfg.tree)
    return pack_trees(parents, cfg.n_max, cfg.depth_max)


# --------------------------------------------------------------------------
# token ids
# --------------------------------------------------------------------------
def make_ids(cfg: Config, trees: Trees, step: int = 0) -> tuple[np.ndarray, np.ndarray]:
    rng = rng_for(cfg, IDS, step)
    T = trees.T
    if cfg.tree == "toy":
        draft = rng.integers(0, cfg.vocab, T).astype(np.int32)
        target = rng.integers(0, cfg.vocab, T).astype(np.int32)
        return draft, target
    draft = np.empty(T, np.int32)
    for bi in range(trees.B):
        lo, hi = int(trees.cu_nodes[bi]), int(trees.cu_nodes[bi + 1])
        par = trees.parent[lo:hi]
        dep = tree_depths(par)
        for d in range(int(dep.max()) + 1 if hi > lo else 0):
            idx = np.nonzero(dep == d)[0]
            # distinct draft tokens within a depth (so siblings never repeat a token)
            draft[lo + idx] = rng.choice(cfg.vocab, size=len(idx), replace=False)
    match = rng.random(T) < cfg.p_match
    other = rng.integers(0, cfg.vocab - 1, T).astype(np.int64)
    other = np.where(other >= draft, other + 1, other)
    target = np.where(match, draft, other).astype(np.int32)
    return draft, target


# --------------------------------------------------------------------------
# GDN tensors
# --------------------------------------------------------------------------
def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = (u + (((u >> 16) & 1) + 0x7FFF)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of bf16-exact float32 values, as int16 (for device upload)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16).view(np.int16)


def _unit_rows(rng, shape) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)


def _softplus(x):
    return np.logaddexp(np.float32(0), x).astype(np.float32)


def _sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


@dataclass
class Inputs:
    q: np.ndarray            # float32 [T, H_qk, dk]  (bf16-exact on bf16 configs)
    k: np.ndarray            # float32 [T, H_qk, dk]
    v: np.ndarray            # float32 [T, H_v, dv]
    g: np.ndarray            # float32 [T, H_v], log-gate <= 0
    b: np.ndarray            # float32 [T, H_v], in (0, 1)
    io: str


def make_node_inputs(cfg: Config, T: int, step: int = 0, layer: int = 0) -> Inputs:
    rng = rng_for(cfg, TENSORS, step, layer)
    q = _unit_rows(rng, (T, cfg.H_qk, cfg.dk))
    k = _unit_rows(rng, (T, cfg.H_qk, cfg.dk))
    v = rng.standard_normal((T, cfg.H_v, cfg.dv), dtype=np.float32)
    g = -_softplus(rng.standard_normal((T, cfg.H_v), dtype=np.float32))
    b = _sigmoid(rng.standard_normal((T, cfg.H_v), dtype=np.float32))
    if cfg.io == "bf16":
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    return Inputs(q, k, v, g, b, cfg.io)


def make_state(cfg: Config, B: int | None = None, layer: int = 0) -> np.ndarray:
    rng = rng_for(cfg, TENSORS, 1_000_000, layer)
    B = cfg.B if B is None else B
    return (cfg.s0_sigma * rng.standard_normal((B, cfg.H_v, cfg.dk, cfg.dv), dtype=np.float32)
            ).astype(np.float32)


@dataclass
class Problem:
    cfg: Config
    trees: Trees
    inputs: Inputs
    S0: np.ndarray
    draft_ids: np.ndarray
    target_ids: np.ndarray
    meta: dict = field(default_factory=dict)


def make_problem(name: str, step: int = 0, layer: int = 0) -> Problem:
    cfg = CONFIGS[name]
    trees = make_trees(cfg, step)
    inputs = make_node_inputs(cfg, trees.T, step, layer)
    S0 = make_state(cfg, layer=layer)
    draft, target = make_ids(cfg, trees, step)
    return Problem(cfg, trees, inputs, S0, draft, target)


def select_sequences(p: Problem, seqs) -> Problem:
    """Sub-batch of whole sequences (sequences are independent on this path)."""
    seqs = list(seqs)
    cu = p.trees.cu_nodes
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]) if seqs else np.zeros(0, int)
    parents = [p.trees.parent[cu[s]:cu[s + 1]] for s in seqs]
    trees = pack_trees(parents, p.trees.n_max, p.trees.depth_max)
    i = p.inputs
    inputs = Inputs(i.q[rows], i.k[rows], i.v[rows], i.g[rows], i.b[rows], i.io)
    return Problem(p.cfg, trees, inputs, p.S0[seqs], p.draft_ids[rows], p.target_ids[rows],
                   dict(p.meta, seqs=seqs, rows=rows))


# --------------------------------------------------------------------------
# device-side draws for benchmark-scale inputs (same recipe, torch's RNG)
# --------------------------------------------------------------------------
def make_node_inputs_device(cfg: Config, T: int, gen, device):
    """q, k, v as bf16 and g, b as fp32, drawn on the device with a seeded torch.Generator."""
    import torch
    def unit(shape):
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        return x / x.norm(dim=-1, keepdim=True)
    q = unit((T, cfg.H_qk, cfg.dk)).to(torch.bfloat16)
    k = unit((T, cfg.H_qk, cfg.dk)).to(torch.bfloat16)
    v = torch.randn((T, cfg.H_v, cfg.dv), generator=gen, device=device).to(torch.bfloat16)
    g = -torch.nn.functional.softplus(torch.randn((T, cfg.H_v), generator=gen, device=device))
    b = torch.sigmoid(torch.randn((T, cfg.H_v), generator=gen, device=device))
    return q, k, v, g.contiguous(), b.contiguous()


def make_state_device(cfg: Config, B: int, gen, device):
    import torch
    return cfg.s0_sigma * torch.randn((B, cfg.H_v, cfg.dk, cfg.dv), generator=gen, device=device)


# --------------------------------------------------------------------------
# drafter tables for top-w best-first tree construction
# --------------------------------------------------------------------------
def make_build_tables(B: int, budget: int, K: int, seed: int = 0, tie_step: float = 0.0):
    """Seeded stand-in for the drafter's top-K continuations of every tree slot.

    Per (sequence, slot): K + 1 logits ~ N(0, 2) (the last one standing for the rest of
    the vocabulary), log-softmax, the K candidate log-probabilities sorted descending;
    K distinct token ids from the vocabulary.  tie_step > 0 rounds the log-probabilities
    to multiples of tie_step (many exact ties).  Returns root_token [B], child_logp
    [B][budget][K] float32, child_token [B][budget][K] int32."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([BASE_SEED, 3000, seed])))
    logits = 2.0 * rng.standard_normal((B, budget, K + 1))
    m = logits.max(axis=-1, keepdims=True)
    lse = m + np.log(np.exp(logits - m).sum(axis=-1, keepdims=True))
    logp = -np.sort(-(logits[..., :K] - lse), axis=-1)
    if tie_step > 0:
        logp = np.minimum(np.round(logp / tie_step) * tie_step, -tie_step)
    tok = np.empty((B, budget, K), np.int32)
    for b in range(B):
        for i in range(budget):
            tok[b, i] = rng.choice(VOCAB, K, replace=False)
    root = rng.integers(0, VOCAB, B).astype(np.int32)
    return root, logp.astype(np.float32), tok
