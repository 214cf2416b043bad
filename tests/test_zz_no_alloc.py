"""tgdn_verify_noalloc: verification for callers that cannot allocate device memory.

Some users of this library cannot call cudaMalloc themselves -- for example a plugin
inside a serving engine that has reserved all device memory for its own pools and hands
its extensions only input and output buffers, or a latency-critical path that must not
take cudaMalloc's implicit device synchronisation.  For them the library keeps the
verification factors in its own fixed-size device array instead of a caller workspace.

The entry point runs the same kernels as tgdn_verify and differs only in where the
factors live, so its outputs must equal tgdn_verify's bit for bit, on two calls in a
row, even when an earlier, larger call has left other values in the array (a read of
a stale row would show).  One comparison with the fp64 oracle checks the values
themselves.  This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import synth, tgdn
from helpers import TOL_BF16, TOL_F32, oracle_step, rel_fro_blocks, upload


def test_noalloc_rejects_sizes_above_its_array():
    """A batch whose factors exceed the array is refused before any launch (host check)."""
    FAKE = 0x10000
    T = 2048                                  # 32 sequences x 64 nodes, 32 heads x 128
    t = tgdn.CTree(32, T, 64, 12, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    d = tgdn.CDims(16, 32, 128, 128, tgdn.BF16)
    assert tgdn.lib().tgdn_verify_workspace_bytes(ctypes.byref(t), ctypes.byref(d)) > \
        tgdn.NOALLOC_SCRATCH_BYTES
    rc = tgdn.lib().tgdn_verify_noalloc(ctypes.byref(t), ctypes.byref(d),
                                        *([FAKE] * 7), None)
    assert rc == tgdn.ETOOBIG


def _bits(t):
    """The raw bits of an output tensor, for exact comparison."""
    torch = pytest.importorskip("torch")
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)).cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("name,tol", [("cfg3", TOL_BF16), ("toy", TOL_F32)])
def test_noalloc_matches_workspace_verify_on_two_calls(name, tol):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    # an earlier, larger call leaves its own factors in the array
    big = synth.make_problem("cfg3", step=7)
    btree, bdims, bdev = upload(big)
    tgdn.tree_prep(btree)
    bo = torch.empty((btree.T, bdims.H_v, bdims.d_v), dtype=bdims.torch_dtype, device="cuda")
    tgdn.verify_noalloc(btree, bdims, bdev["q"], bdev["k"], bdev["v"], bdev["g"], bdev["b"],
                        bdev["S0"], bo)
    # the case under test, smaller than the earlier call
    p = synth.make_problem(name)
    if name == "cfg3":
        p = synth.select_sequences(p, range(5))
    tree, dims, dev = upload(p)
    assert tgdn.verify_workspace_bytes(tree, dims) < tgdn.verify_workspace_bytes(btree, bdims)
    tgdn.tree_prep(tree)
    ws = tgdn.alloc_workspace(tree, dims)
    shape = (tree.T, dims.H_v, dims.d_v)
    o_ref = torch.full(shape, float("nan"), dtype=dims.torch_dtype, device="cuda")
    tgdn.verify(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], dev["S0"], o_ref,
                ws)
    ref_bits = _bits(o_ref)
    for call in range(2):
        o = torch.full(shape, float("nan"), dtype=dims.torch_dtype, device="cuda")
        tgdn.verify_noalloc(tree, dims, dev["q"], dev["k"], dev["v"], dev["g"], dev["b"],
                            dev["S0"], o)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(o), ref_bits), call
    ref = oracle_step(p)
    err = rel_fro_blocks(o.float().cpu().numpy(), ref["o"], p.trees.cu_nodes)
    assert err <= tol, err
