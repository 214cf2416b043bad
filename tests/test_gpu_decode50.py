"""The 36-layer stack workload over its whole horizon: 50 decode steps.

For three layers of the stack (0, 17, 35), a full one-layer batch (32 sequences of
64-node random trees, depth <= 12, H_qk = 16, H_v = 32, d = 128, bf16) runs 50
steps of the benchmark's step -- tree prep, the verification with the previous
step's commit folded in (tgdn_verify_fused, the launch configuration bench.py
times), greedy acceptance -- and a final tgdn_commit.  Every step starts from the
state the previous steps committed ("Trees from Marginals", Methodik 3, last
bullet: the deferred, rollback-free commit), so any drift compounds over the
horizon.  The fp64 oracle replays the same decode on a sample of 4 sequences x 2
query/key heads (4 value heads): outputs, acceptance and the committed state are
compared at every step.  Node inputs are drawn on the device by the shared seeded
generator and the sampled rows are copied back for the oracle.
"""
import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, rel_fro_blocks

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
from tree_speculative_decoding_gated_gb300 import tgdn  # noqa: E402
import oracle  # noqa: E402

LAYERS = (0, 17, 35)
STEPS = 50
SEQS = [0, 1, 2, 3]
QK_HEADS = [0, 11]


def _rows(cu, seqs):
    return np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])


@pytest.mark.parametrize("layer", LAYERS)
def test_stack_decode_fifty_steps(layer):
    cfg = synth.CONFIGS["cfg5"]
    assert cfg.steps == STEPS and cfg.B == 32
    dims = tgdn.Dims(cfg.H_qk, cfg.H_v, cfg.dk, cfg.dv, tgdn.BF16)
    grp = cfg.H_v // cfg.H_qk
    vh = [qh * grp + j for qh in QK_HEADS for j in range(grp)]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(synth.BASE_SEED + cfg.number + 1000 + 97 * layer)
    S = synth.make_state_device(cfg, cfg.B, gen, "cuda")
    S_ref = S[SEQS][:, vh].double().cpu().numpy()
    prev = None
    worst_o = worst_s = 0.0
    for step in range(STEPS):
        trees = synth.make_trees(cfg, step)
        draft, target = synth.make_ids(cfg, trees, step)
        tree = tgdn.Tree.from_host(trees.cu_nodes, trees.parent, trees.n_max, trees.depth_max,
                                   "cuda")
        q, k, v, g, b = synth.make_node_inputs_device(cfg, trees.T, gen, "cuda")
        tgdn.tree_prep(tree)
        ws = tgdn.alloc_workspace(tree, dims)
        o = torch.full((trees.T, cfg.H_v, cfg.dv), float("nan"), dtype=torch.bfloat16,
                       device="cuda")
        if prev is None:
            tgdn.verify(tree, dims, q, k, v, g, b, S, o, ws)
        else:
            ptree, pan, ppath, pk, pws = prev
            tgdn.verify_fused(tree, dims, q, k, v, g, b, S, o, ws, ptree, pan, ppath, pk, pws)
        an = torch.empty(cfg.B, dtype=torch.int32, device="cuda")
        al = torch.empty_like(an)
        path = torch.empty((cfg.B, trees.depth_max + 1), dtype=torch.int32, device="cuda")
        tgdn.accept(tree, torch.from_numpy(draft).cuda(), torch.from_numpy(target).cuda(), an,
                    al, path)
        torch.cuda.synchronize()
        # the oracle on the sample: the same exact inputs, from the state it committed
        rows = _rows(trees.cu_nodes, SEQS)
        sub = synth.pack_trees([trees.parent[trees.cu_nodes[s]:trees.cu_nodes[s + 1]]
                                for s in SEQS], trees.n_max, trees.depth_max)
        f = lambda x: x.float().cpu().numpy().astype(np.float64)
        qs, ks = f(q[rows][:, QK_HEADS]), f(k[rows][:, QK_HEADS])
        vs, gs, bs = f(v[rows][:, vh]), f(g[rows][:, vh]), f(b[rows][:, vh])
        ref_o = oracle.verify(sub.cu_nodes, sub.parent, sub.n_max, sub.depth_max, qs, ks, vs,
                              gs, bs, S_ref)
        acc = oracle.accept(sub.cu_nodes, sub.parent, sub.n_max, sub.depth_max, draft[rows],
                            target[rows])
        eo = rel_fro_blocks(f(o[rows][:, vh]), ref_o, sub.cu_nodes)
        worst_o = max(worst_o, eo)
        assert eo <= TOL_BF16, (layer, step, eo)
        assert np.array_equal(an.cpu().numpy()[SEQS], acc["accept_node"]), (layer, step)
        if step > 0:  # the state this step verified from: the commit of step - 1
            es = rel_fro_blocks(S[SEQS][:, vh].double().cpu().numpy(), S_ref)
            worst_s = max(worst_s, es)
            assert es <= TOL_BF16, (layer, step, es)
        S_ref = oracle.commit(sub.cu_nodes, sub.parent, sub.n_max, sub.depth_max, ks, vs, gs,
                              bs, S_ref, acc["accept_node"])
        prev = (tree, an, path, k, ws)
    ptree, pan, _, pk, pws = prev
    tgdn.commit(ptree, dims, pan, pk, pws, S, S)
    torch.cuda.synchronize()
    es = rel_fro_blocks(S[SEQS][:, vh].double().cpu().numpy(), S_ref)
    worst_s = max(worst_s, es)
    print(f"layer {layer}: {STEPS} steps, worst output error {worst_o:.3e}, "
          f"worst committed-state error {worst_s:.3e}")
    assert es <= TOL_BF16
