"""A bounded device wait that runs out: TGDN_SEQ_TIMEOUT, no fault, no hang.

Every wait of the tensor-core verification kernel gives up after a limit, marks
the sequences of every work item its CTA owns TGDN_SEQ_TIMEOUT, waits for its own
copies and products to finish, frees its tensor memory and returns.  A test hook
(tgdn_debug_set_wait_hooks) shortens the limit to 1 ms and makes the producer
warps withhold the first tensor-core product of one work item, so the consumer's
wait for it expires -- a flag that nothing sets, not a fault.  The test checks the statuses,
that every other sequence still matches the fp64 oracle, that the launch returns
promptly, and that the context stays usable for a normal verification afterwards.
"""
import time

import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth
from helpers import TOL_BF16, oracle_step, rel_fro_blocks, upload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)
from tree_speculative_decoding_gated_gb300 import tgdn  # noqa: E402


def test_withheld_hand_over_times_out_and_the_rest_is_verified():
    p = synth.make_problem("cfg3")               # 16 sequences x 32 value heads = 512 items
    tree, dims, dev = upload(p)
    B, H_v = tree.B, dims.H_v
    items = B * H_v
    grid = min(items, torch.cuda.get_device_properties(0).multi_processor_count)
    hold = grid                                   # CTA 0's second item (items are dealt
    cta0 = list(range(0, items, grid))            # round robin: CTA 0 owns 0, grid, 2 grid...)
    hit = sorted({it // H_v for it in cta0})
    ref = oracle_step(p)
    shape = (tree.T, H_v, dims.d_v)
    try:
        tgdn.debug_set_wait_hooks(1_000_000, hold)
        tgdn.tree_prep(tree)
        ws = tgdn.alloc_workspace(tree, dims)
        o = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        t0 = time.time()
        tgdn.verify(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], dev["S0"], o,
                    ws)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        tgdn.debug_set_wait_hooks()
    status = tree.status.cpu().numpy()
    assert elapsed < 1.0, elapsed                 # a 1 ms limit, not the 2 s default
    assert [b for b in range(B) if status[b] == tgdn.SEQ_TIMEOUT] == hit, (status, hit)
    assert (status[[b for b in range(B) if b not in hit]] == tgdn.SEQ_OK).all()
    # every other sequence was verified as usual
    keep = [b for b in range(B) if b not in hit]
    got = o.float().cpu().numpy()
    cu = p.trees.cu_nodes
    for b in keep:
        lo, hi = cu[b], cu[b + 1]
        err = rel_fro_blocks(got[lo:hi], ref["o"][lo:hi], np.array([0, hi - lo]))
        assert err <= TOL_BF16, (b, err)
    # the context is still usable: the same batch verifies normally now
    tgdn.tree_prep(tree)
    o2 = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    tgdn.verify(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], dev["S0"], o2, ws)
    torch.cuda.synchronize()
    assert (tree.status.cpu().numpy() == tgdn.SEQ_OK).all()
    assert rel_fro_blocks(o2.float().cpu().numpy(), ref["o"], cu) <= TOL_BF16


def test_wait_hook_arguments_are_checked():
    with pytest.raises(tgdn.TgdnError):
        tgdn.debug_set_wait_hooks(3_000_000_000, -1)
    with pytest.raises(tgdn.TgdnError):
        tgdn.debug_set_wait_hooks(0, -2)
    tgdn.debug_set_wait_hooks()
