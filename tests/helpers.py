"""Shared test utilities: upload seeded problems, run one step through the C ABI, error norms."""
from __future__ import annotations

import numpy as np

from tree_speculative_decoding_gated_gb300 import synth

# Tolerances (max over (sequence, v-head) blocks of the relative Frobenius error).
TOL_BF16 = 2e-2
TOL_F32 = 1e-4


def rel_fro_blocks(got, ref, cu_nodes=None):
    """Max relative Frobenius error over (sequence, head) blocks.

    got/ref: [T, H, d] node outputs (blocks = rows of one sequence, one head) when
    cu_nodes is given, else [B, H, dk, dv] states (blocks = one state matrix)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    worst = 0.0
    if cu_nodes is None:
        for bi in range(ref.shape[0]):
            for h in range(ref.shape[1]):
                d = np.linalg.norm(got[bi, h] - ref[bi, h])
                worst = max(worst, d / max(np.linalg.norm(ref[bi, h]), 1e-30))
        return worst
    for bi in range(len(cu_nodes) - 1):
        lo, hi = int(cu_nodes[bi]), int(cu_nodes[bi + 1])
        if hi == lo:
            continue
        for h in range(ref.shape[1]):
            d = np.linalg.norm(got[lo:hi, h] - ref[lo:hi, h])
            worst = max(worst, d / max(np.linalg.norm(ref[lo:hi, h]), 1e-30))
    return worst


def to_device_io(x: np.ndarray, io: str, device="cuda"):
    import torch
    if io == "bf16":
        return torch.from_numpy(synth.bf16_bits(x)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


def upload(p: synth.Problem, device="cuda", n_max=None, depth_max=None):
    import torch
    from tree_speculative_decoding_gated_gb300 import tgdn
    cfg = p.cfg
    tree = tgdn.Tree.from_host(p.trees.cu_nodes, p.trees.parent,
                               n_max or p.trees.n_max, depth_max if depth_max is not None
                               else p.trees.depth_max, device)
    i = p.inputs
    # head counts from the tensors themselves (a head subset keeps the workload's cfg)
    dims = tgdn.Dims(i.q.shape[1], i.v.shape[1], cfg.dk, cfg.dv,
                     tgdn.BF16 if cfg.io == "bf16" else tgdn.F32)
    f32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)
    dev = dict(q=to_device_io(i.q, cfg.io, device), k=to_device_io(i.k, cfg.io, device),
               v=to_device_io(i.v, cfg.io, device), g=f32(i.g), b=f32(i.b), S0=f32(p.S0),
               draft=torch.from_numpy(p.draft_ids.astype(np.int32)).to(device),
               target=torch.from_numpy(p.target_ids.astype(np.int32)).to(device))
    return tree, dims, dev


def run_step(tree, dims, dev, in_place=False):
    """prep -> verify -> accept -> commit through the C ABI; returns host numpy results."""
    import torch
    from tree_speculative_decoding_gated_gb300 import tgdn
    T, B = tree.T, tree.B
    tgdn.tree_prep(tree)
    ws = tgdn.alloc_workspace(tree, dims)
    o = torch.full((T, dims.H_v, dims.d_v), float("nan"), dtype=dims.torch_dtype, device="cuda")
    tgdn.verify(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], dev["S0"], o, ws)
    an = torch.empty(B, dtype=torch.int32, device="cuda")
    al = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.empty((B, tree.depth_max + 1), dtype=torch.int32, device="cuda")
    tgdn.accept(tree, dev["draft"], dev["target"], an, al, path)
    if in_place:
        S = dev["S0"].clone()
        tgdn.commit(tree, dims, an, dev["k"], ws, S, S)
    else:
        S = torch.full_like(dev["S0"], float("nan"))
        tgdn.commit(tree, dims, an, dev["k"], ws, dev["S0"], S)
    torch.cuda.synchronize()
    c = lambda t: t.cpu().float().numpy() if t.is_floating_point() else t.cpu().numpy()
    return dict(o=c(o), S=c(S), accept_node=c(an), accept_len=c(al), path=c(path),
                depth=c(tree.depth), order=c(tree.order), pos=c(tree.pos),
                anc=tree.anc.cpu().numpy().view(np.uint64), status=c(tree.status), ws=ws)


def oracle_step(p: synth.Problem, nthreads=0):
    import oracle
    t, i = p.trees, p.inputs
    prep = oracle.prep(t.cu_nodes, t.parent, t.n_max, t.depth_max)
    acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, p.draft_ids, p.target_ids)
    o = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v, i.g, i.b, p.S0,
                      nthreads)
    S = oracle.commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b, p.S0,
                      acc["accept_node"], nthreads)
    return dict(prep=prep, **acc, o=o, S=S)


def assert_meta_equal(got, ref):
    for key in ("status", "depth", "order", "pos"):
        assert np.array_equal(got[key], ref["prep"][key]), key
    assert np.array_equal(got["anc"], ref["prep"]["anc"]), "anc"
    for key in ("accept_node", "accept_len", "path"):
        assert np.array_equal(got[key], ref[key]), key


def head_pair_subset(p: synth.Problem, qk_heads) -> synth.Problem:
    """Keeps the given query/key heads and the value heads that read them (GQA kept intact)."""
    cfg = p.cfg
    grp = cfg.H_v // cfg.H_qk
    vh = [qh * grp + j for qh in qk_heads for j in range(grp)]
    i = p.inputs
    inputs = synth.Inputs(i.q[:, qk_heads], i.k[:, qk_heads], i.v[:, vh], i.g[:, vh], i.b[:, vh],
                          i.io)
    return synth.Problem(p.cfg, p.trees, inputs, p.S0[:, vh], p.draft_ids, p.target_ids,
                         dict(p.meta, v_heads=vh))
