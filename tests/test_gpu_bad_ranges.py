"""Sequences whose row range (cu_nodes) leaves [0, T) are reported, never touched.

tgdn_tree_prep gives a sequence with cu_nodes[b] < 0, cu_nodes[b+1] < cu_nodes[b] or
cu_nodes[b+1] > T the status TGDN_SEQ_BAD_RANGE, and no call reads or writes a row of
it.  Every [T]-leading array here is a view into a larger buffer with canary rows on
both sides (more than any offset the bad ranges reach), so a stray access would land in
the canaries, inside the allocation, instead of faulting; the canaries are checked
after every call.  The valid sequences of the same batch must still match the fp64
oracle run on them alone.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, TOL_F32, rel_fro_blocks

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
from tree_speculative_decoding_gated_gb300 import tgdn  # noqa: E402
import oracle  # noqa: E402

GUARD = 32          # canary rows before and after every [T]-leading array
CANARY_I32 = -77777
CANARY_F32 = 12345.5


class Guarded:
    """A [T, ...] view inside a [GUARD + T + GUARD, ...] buffer filled with a canary."""

    def __init__(self, T, tail, dtype, canary, init=None):
        self.T = T
        self.full = torch.full((GUARD + T + GUARD, *tail), canary, dtype=dtype, device="cuda")
        self.view = self.full[GUARD:GUARD + T]
        if init is not None:
            self.view.copy_(init)
        self.canary = canary

    def guards_intact(self):
        c = torch.full((), self.canary, dtype=self.full.dtype, device="cuda")
        f = self.full
        return bool((f[:GUARD] == c).all()) and bool((f[GUARD + self.T:] == c).all())


def bad_batch(n_max):
    """Six sequences over T = 10 rows: two valid trees (rows 0-4 and 5-9) and four
    bad ranges (decreasing, past T, decreasing from past T, negative start)."""
    cu = np.array([0, 5, 3, 12, -2, 5, 10], np.int32)
    p0 = np.array([-1, 0, 0, 1, 2], np.int32)
    p1 = np.array([-1, 0, 1, 1, 0], np.int32)
    parent = np.concatenate([p0, p1])
    return cu, parent, [0, 5], (p0, p1)


def run_case(io, dk, n_max):
    cu, parent, good, (p0, p1) = bad_batch(n_max)
    T, B = 10, len(cu) - 1
    H_qk, H_v = 2, 4
    cfg = synth.Config("badrange", 41, B=2, H_qk=H_qk, H_v=H_v, dk=dk, dv=dk, io=io,
                       tree="random", s0_sigma=0.05)
    sub_trees = synth.pack_trees([p0, p1], n_max, 8)
    inp = synth.make_node_inputs(cfg, T)
    S0_good = synth.make_state(cfg, B=2)
    dt = torch.bfloat16 if io == "bf16" else torch.float32
    tobf = lambda x: (torch.from_numpy(synth.bf16_bits(x)).view(torch.bfloat16) if io == "bf16"
                      else torch.from_numpy(np.ascontiguousarray(x, np.float32))).cuda()
    f32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    rows = {}
    rows["parent"] = Guarded(T, (), torch.int32, CANARY_I32, torch.from_numpy(parent).cuda())
    rows["q"] = Guarded(T, (H_qk, dk), dt, CANARY_F32, tobf(inp.q))
    rows["k"] = Guarded(T, (H_qk, dk), dt, CANARY_F32, tobf(inp.k))
    rows["v"] = Guarded(T, (H_v, dk), dt, CANARY_F32, tobf(inp.v))
    rows["g"] = Guarded(T, (H_v,), torch.float32, CANARY_F32, f32(inp.g))
    rows["b"] = Guarded(T, (H_v,), torch.float32, CANARY_F32, f32(inp.b))
    rows["o"] = Guarded(T, (H_v, dk), dt, CANARY_F32)
    rng = np.random.default_rng(3)
    draft = rng.integers(0, 3, T).astype(np.int32)
    target = np.where(rng.random(T) < 0.8, draft, rng.integers(0, 3, T)).astype(np.int32)
    rows["draft"] = Guarded(T, (), torch.int32, CANARY_I32, torch.from_numpy(draft).cuda())
    rows["target"] = Guarded(T, (), torch.int32, CANARY_I32, torch.from_numpy(target).cuda())
    tree = tgdn.Tree(torch.from_numpy(cu).cuda(), rows["parent"].view, n_max, 8, T=T)
    words = tree.words
    meta = {n: Guarded(T, (), torch.int32, CANARY_I32) for n in ("depth", "order", "pos")}
    meta["anc"] = Guarded(T, (words,), torch.int64, CANARY_I32)
    tree.depth, tree.order, tree.pos, tree.anc = (meta[n].view for n in
                                                  ("depth", "order", "pos", "anc"))
    # the state: one block per sequence, the two valid ones hold the oracle's S0
    S0 = torch.full((B, H_v, dk, dk), 0.25, dtype=torch.float32, device="cuda")
    S0[0], S0[5] = f32(S0_good[0]), f32(S0_good[1])
    dims = tgdn.Dims(H_qk, H_v, dk, dk, tgdn.BF16 if io == "bf16" else tgdn.F32)
    # workspace with canary bytes on both sides (256-byte aligned view)
    wsn = tgdn.verify_workspace_bytes(tree, dims)
    pad = 256 * ((GUARD * H_v * dk * 4 + 255) // 256)
    ws_full = torch.full((pad + wsn + pad,), 0x5A, dtype=torch.uint8, device="cuda")
    ws = ws_full[pad:pad + wsn]

    def all_guards():
        bad = [n for n, g in list(rows.items()) + list(meta.items()) if not g.guards_intact()]
        if not bool((ws_full[:pad] == 0x5A).all()) or not bool((ws_full[pad + wsn:] == 0x5A).all()):
            bad.append("ws")
        return bad

    tgdn.tree_prep(tree)
    torch.cuda.synchronize()
    st = tree.status.cpu().numpy()
    assert st.tolist() == [0, 7, 7, 7, 7, 0], st
    assert all_guards() == []
    tgdn.verify(tree, dims, rows["q"].view, rows["k"].view, rows["v"].view, rows["g"].view,
                rows["b"].view, S0, rows["o"].view, ws)
    an = torch.full((B,), 99, dtype=torch.int32, device="cuda")
    al = torch.full((B,), 99, dtype=torch.int32, device="cuda")
    path = torch.full((B, 9), 99, dtype=torch.int32, device="cuda")
    tgdn.accept(tree, rows["draft"].view, rows["target"].view, an, al, path)
    S = S0.clone()
    tgdn.commit(tree, dims, an, rows["k"].view, ws, S, S)
    o_rec = Guarded(T, (H_v, dk), dt, CANARY_F32)
    tgdn.verify_recurrent(tree, dims, rows["q"].view, rows["k"].view, rows["v"].view,
                          rows["g"].view, rows["b"].view, S0, o_rec.view)
    torch.cuda.synchronize()
    assert all_guards() == [] and o_rec.guards_intact()
    # bad sequences: no acceptance, state kept
    anh = an.cpu().numpy()
    assert (anh[1:5] == -1).all() and (al.cpu().numpy()[1:5] == 0).all()
    Sh = S.cpu().numpy()
    assert (Sh[1:5] == 0.25).all()
    # the valid sequences against the oracle run on them alone
    sub = synth.Problem(cfg, sub_trees, inp, S0_good, draft, target)
    t, i = sub.trees, sub.inputs
    ref_o = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v, i.g, i.b,
                          sub.S0)
    acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, draft, target)
    ref_S = oracle.commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b,
                          sub.S0, acc["accept_node"])
    tol = TOL_BF16 if io == "bf16" else TOL_F32
    for got in (rows["o"].view, o_rec.view):
        assert rel_fro_blocks(got.float().cpu().numpy(), ref_o, t.cu_nodes) <= tol
    assert np.array_equal(anh[[0, 5]], acc["accept_node"])
    assert rel_fro_blocks(Sh[[0, 5]], ref_S) <= tol
    # the same batch again with its commit folded into the verification
    ws2_full = torch.full((pad + wsn + pad,), 0x5A, dtype=torch.uint8, device="cuda")
    ws2 = ws2_full[pad:pad + wsn]
    S2 = S0.clone()
    o2 = Guarded(T, (H_v, dk), dt, CANARY_F32)
    tgdn.verify_fused(tree, dims, rows["q"].view, rows["k"].view, rows["v"].view,
                      rows["g"].view, rows["b"].view, S2, o2.view, ws2, tree, an, path,
                      rows["k"].view, ws)
    torch.cuda.synchronize()
    assert all_guards() == [] and o2.guards_intact()
    assert bool((ws2_full[:pad] == 0x5A).all()) and bool((ws2_full[pad + wsn:] == 0x5A).all())
    S2h = S2.cpu().numpy()
    assert (S2h[1:5] == 0.25).all()
    assert rel_fro_blocks(S2h[[0, 5]], ref_S) <= tol
    return tree, rows, meta, dims, all_guards


@pytest.mark.parametrize("io,dk,n_max", [("bf16", 128, 64), ("bf16", 128, 100),
                                         ("f32", 16, 64)])
def test_bad_ranges_are_untouched(io, dk, n_max):
    """Tensor-core kernels (<= 64 and <= 129 nodes) and the SIMT kernel."""
    run_case(io, dk, n_max)


def test_bad_ranges_in_tree_attention():
    tree, rows, meta, dims, all_guards = run_case("bf16", 128, 64)
    T, B = tree.T, tree.B
    H_q, H_kv, d, P = 4, 2, 128, 64
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    rnd = lambda *s: torch.randn(s, generator=gen, device="cuda").to(torch.bfloat16)
    q = Guarded(T, (H_q, d), torch.bfloat16, CANARY_F32, rnd(T, H_q, d))
    kt = Guarded(T, (H_kv, d), torch.bfloat16, CANARY_F32, rnd(T, H_kv, d))
    vt = Guarded(T, (H_kv, d), torch.bfloat16, CANARY_F32, rnd(T, H_kv, d))
    o = Guarded(T, (H_q, d), torch.bfloat16, CANARY_F32)
    kc, vc = rnd(B, P, H_kv, d), rnd(B, P, H_kv, d)
    pl = torch.full((B,), P, dtype=torch.int32, device="cuda")
    tgdn.tree_attention(tree, q.view, kt.view, vt.view, kc, vc, pl, o.view, d ** -0.5)
    torch.cuda.synchronize()
    assert all_guards() == []
    assert q.guards_intact() and kt.guards_intact() and vt.guards_intact() and o.guards_intact()
    assert torch.isfinite(o.view.float()).all()
