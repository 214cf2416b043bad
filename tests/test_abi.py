"""CPU-only checks of the C ABI: the library loads, exports every declared call, and its
host-side argument checks reject bad input before any launch (no GPU work here)."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

from tree_speculative_decoding_gated_gb300 import tgdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from tree_speculative_decoding_gated_gb300 import build
    build.build()
    return tgdn.lib()


FAKE = 0x10000  # a non-null address; never dereferenced on the host


def ctree(B=2, T=10, n_max=8, depth_max=4, words=None):
    w = (n_max + 63) // 64 if words is None else words
    return tgdn.CTree(B, T, n_max, depth_max, w, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)


def cdims(H_qk=2, H_v=4, dk=128, dv=128, io=tgdn.BF16):
    return tgdn.CDims(H_qk, H_v, dk, dv, io)


def test_exports_every_declared_function(L):
    names = tgdn.header_functions()
    assert set(names) >= {"tgdn_tree_prep", "tgdn_verify_workspace_bytes", "tgdn_verify",
                          "tgdn_accept", "tgdn_commit", "tgdn_status_string", "tgdn_version"}
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", tgdn.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_header_is_plain_c():
    """The header compiles as C99 with no CUDA or torch headers on the include path."""
    src = "#include \"tgdn.h\"\nint main(void){ return tgdn_version() < 0; }\n"
    r = subprocess.run(["gcc", "-std=c99", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        "-x", "c", "-"], input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings_and_version(L):
    assert tgdn.status_string(0) == "ok"
    assert "invalid" in tgdn.status_string(-1)
    assert L.tgdn_version() >= 100


def test_struct_layout_matches_c():
    assert ctypes.sizeof(tgdn.CTree) == 5 * 4 + 4 + 7 * 8
    assert tgdn.CTree.cu_nodes.offset == 24
    assert ctypes.sizeof(tgdn.CDims) == 20


def call_prep(L, t):
    return L.tgdn_tree_prep(ctypes.byref(t), None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), tgdn.EINVAL), (dict(T=-1), tgdn.EINVAL), (dict(n_max=0), tgdn.EINVAL),
    (dict(n_max=257), tgdn.ETOOBIG), (dict(depth_max=65), tgdn.ETOOBIG),
    (dict(depth_max=-1), tgdn.EINVAL), (dict(words=2), tgdn.EINVAL),
])
def test_prep_rejects(L, kw, code):
    assert call_prep(L, ctree(**kw)) == code


def test_null_pointers_rejected(L):
    t = ctree()
    t.parent = None
    assert call_prep(L, t) == tgdn.EINVAL
    assert L.tgdn_tree_prep(None, None) == tgdn.EINVAL
    t = ctree()
    d = cdims()
    args = [FAKE] * 8
    args[0] = None   # q
    assert L.tgdn_verify(ctypes.byref(t), ctypes.byref(d), *args, None) == tgdn.EINVAL
    assert L.tgdn_accept(ctypes.byref(t), None, FAKE, FAKE, FAKE, FAKE, None) == tgdn.EINVAL
    assert L.tgdn_commit(ctypes.byref(t), ctypes.byref(d), None, FAKE, FAKE, FAKE, FAKE + 10**9,
                         None) == tgdn.EINVAL


@pytest.mark.parametrize("kw,code", [
    (dict(H_qk=3, H_v=4), tgdn.EINVAL), (dict(H_qk=0), tgdn.EINVAL), (dict(dk=0), tgdn.EINVAL),
    (dict(dk=129), tgdn.ETOOBIG), (dict(dv=256), tgdn.ETOOBIG), (dict(io=7), tgdn.EINVAL),
])
def test_dims_rejected(L, kw, code):
    t, d = ctree(), cdims(**kw)
    assert L.tgdn_verify(ctypes.byref(t), ctypes.byref(d), *([FAKE] * 8), None) == code
    assert L.tgdn_verify_workspace_bytes(ctypes.byref(t), ctypes.byref(d)) == 0


def test_workspace_misaligned_rejected(L):
    t, d = ctree(), cdims()
    args = [FAKE] * 8
    args[7] = FAKE + 16
    assert L.tgdn_verify(ctypes.byref(t), ctypes.byref(d), *args, None) == tgdn.EINVAL


def test_commit_overlap_rejected(L):
    t, d = ctree(), cdims()
    assert L.tgdn_commit(ctypes.byref(t), ctypes.byref(d), FAKE, FAKE, FAKE, FAKE,
                         FAKE + 4096, None) == tgdn.EINVAL


def test_workspace_bytes(L):
    t, d = ctree(B=3, T=100), cdims(H_qk=16, H_v=32)
    u = 100 * 32 * 128 * 4
    want = (u + 255) // 256 * 256 + 100 * 32 * 4
    assert L.tgdn_verify_workspace_bytes(ctypes.byref(t), ctypes.byref(d)) == want


def test_empty_batch_is_a_no_op(L):
    t = tgdn.CTree(0, 0, 8, 4, 1, None, None, None, None, None, None, None)
    d = cdims()
    assert L.tgdn_tree_prep(ctypes.byref(t), None) == 0
    assert L.tgdn_verify(ctypes.byref(t), ctypes.byref(d), *([None] * 7), FAKE, None) == 0
    assert L.tgdn_accept(ctypes.byref(t), None, None, None, None, None, None) == 0
    assert L.tgdn_commit(ctypes.byref(t), ctypes.byref(d), None, None, None, None, None, None) == 0


def test_binding_refuses_host_tensors():
    torch = pytest.importorskip("torch")
    cu = torch.tensor([0, 3], dtype=torch.int32)
    par = torch.tensor([-1, 0, 0], dtype=torch.int32)
    tree = tgdn.Tree(cu, par, 4, 2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        tgdn.tree_prep(tree)


def test_product_path_does_not_reach_the_oracle():
    """The package and the C ABI never import, link or open the oracle."""
    pkg = os.path.join(ROOT, "tree_speculative_decoding_gated_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f
    assert "oracle" not in open(os.path.join(ROOT, "include", "tgdn.h")).read().lower()


def test_verify_fused_rejects_bad_arguments(L):
    """Host checks of tgdn_verify_fused: batch sizes must match, the two workspaces must not
    overlap and both must be 256-byte aligned (nothing is launched)."""
    d = cdims()
    t, pt = ctree(B=2, T=10), ctree(B=2, T=10)
    f = L.tgdn_verify_fused
    ws, pws = FAKE * 16, FAKE * 64

    def call(t, pt, ws, pws):
        return f(ctypes.byref(t), ctypes.byref(d), *([FAKE] * 7), ws, ctypes.byref(pt),
                 FAKE, FAKE, FAKE, pws, None)

    assert call(t, ctree(B=3, T=10), ws, pws) == tgdn.EINVAL      # different batch
    assert call(t, pt, ws, ws) == tgdn.EINVAL                       # same workspace
    assert call(t, pt, ws, ws + 256) == tgdn.EINVAL                 # overlapping workspaces
    assert call(t, pt, ws + 16, pws) == tgdn.EINVAL                 # misaligned
    assert call(t, pt, ws, pws + 16) == tgdn.EINVAL
    assert f(ctypes.byref(t), ctypes.byref(d), *([FAKE] * 7), ws, None, FAKE, FAKE, FAKE, pws,
             None) == tgdn.EINVAL                                   # no previous tree
    assert f(ctypes.byref(t), ctypes.byref(d), *([FAKE] * 7), ws, ctypes.byref(pt), None,
             FAKE, FAKE, pws, None) == tgdn.EINVAL                  # no accepted nodes


def test_tree_attention_rejects_bad_arguments(L):
    """Host checks of tgdn_tree_attention: head counts, context length, the softmax scale
    (positive and finite), the supported shapes and 16-byte alignment are checked before
    anything is launched."""
    t = ctree(B=2, T=10, n_max=8)
    f = L.tgdn_tree_attention

    def call(tree=t, H_q=8, H_kv=2, d=128, P_max=16, scale=0.088, q=FAKE):
        return f(ctypes.byref(tree), H_q, H_kv, d, q, FAKE, FAKE, FAKE, FAKE, FAKE, P_max,
                 scale, FAKE, None, 0, None)

    assert call(H_q=0) == tgdn.EINVAL
    assert call(H_kv=3) == tgdn.EINVAL                  # 8 query heads over 3 kv heads
    assert call(P_max=-1) == tgdn.EINVAL
    for bad in (0.0, -0.5, float("nan"), float("inf"), -float("inf")):
        assert call(scale=bad) == tgdn.EINVAL, bad
    assert call(d=64) == tgdn.EUNSUPPORTED              # head size other than 128
    assert call(H_q=32, H_kv=1) == tgdn.EUNSUPPORTED    # 32 query heads per kv head
    assert call(tree=ctree(B=2, T=300, n_max=129)) == tgdn.EUNSUPPORTED
    assert call(q=FAKE + 2) == tgdn.EINVAL              # misaligned query rows


def test_tree_build_rejects_bad_arguments(L):
    """Host checks of tgdn_tree_build: sizes must be positive and within the library's
    bounds, and no pointer may be null (nothing is launched)."""
    f = L.tgdn_tree_build

    def call(B=2, budget=16, K=4, w=2, depth_max=8, root=FAKE):
        return f(B, budget, K, w, depth_max, root, *([FAKE] * 8), None)

    assert call(budget=0) == tgdn.EINVAL
    assert call(K=0) == tgdn.EINVAL
    assert call(w=0) == tgdn.EINVAL
    assert call(depth_max=-1) == tgdn.EINVAL
    assert call(B=-1) == tgdn.EINVAL
    assert call(budget=1 << 20) == tgdn.ETOOBIG
    assert call(root=None) == tgdn.EINVAL
    assert call(B=0, root=None) == tgdn.OK               # an empty batch is a no-op
