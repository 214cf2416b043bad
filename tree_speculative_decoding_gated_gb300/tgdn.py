"""Thin Python binding of libtgdn.so (include/tgdn.h) — argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module only
checks that the torch tensors it is handed live on the GPU with the dtype,
layout and size the C ABI expects (a host pointer handed to a kernel would
fault the device), packs the C structs and raises on a non-zero status.  There
is no fallback: if the library has not been built this module fails to load.

Names follow the C ABI: tree_prep, verify_workspace_bytes, verify, accept,
commit.  All calls are asynchronous on the given stream (default: torch's
current stream).
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtgdn.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "tgdn.h")

OK, EINVAL, ETOOBIG, ECUDA, EUNSUPPORTED = 0, -1, -3, -4, -5
SEQ_OK, SEQ_TOO_BIG, SEQ_BAD_PARENT, SEQ_ROOTS, SEQ_CYCLE, SEQ_TOO_DEEP, SEQ_TIMEOUT = range(7)
F32, BF16 = 0, 1
MAX_NODES, MAX_DEPTH, MAX_HEAD_DIM = 256, 64, 128
NOALLOC_SCRATCH_BYTES = 20 * 1024 * 1024


class TgdnError(RuntimeError):
    def __init__(self, code: int, call: str):
        self.code = code
        super().__init__(f"{call}: {status_string(code)} ({code})")


class CTree(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("n_max", ctypes.c_int32),
                ("depth_max", ctypes.c_int32), ("words", ctypes.c_int32),
                ("cu_nodes", ctypes.c_void_p), ("parent", ctypes.c_void_p),
                ("depth", ctypes.c_void_p), ("order", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("anc", ctypes.c_void_p), ("status", ctypes.c_void_p)]


class CDims(ctypes.Structure):
    _fields_ = [("H_qk", ctypes.c_int32), ("H_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("io", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libtgdn.so; raises if it has not been built (there is no other path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        P = ctypes.POINTER
        L.tgdn_tree_prep.argtypes = [P(CTree), st]
        L.tgdn_verify_workspace_bytes.argtypes = [P(CTree), P(CDims)]
        L.tgdn_verify_workspace_bytes.restype = ctypes.c_size_t
        L.tgdn_verify.argtypes = [P(CTree), P(CDims), vp, vp, vp, vp, vp, vp, vp, vp, st]
        L.tgdn_accept.argtypes = [P(CTree), vp, vp, vp, vp, vp, st]
        L.tgdn_commit.argtypes = [P(CTree), P(CDims), vp, vp, vp, vp, vp, st]
        L.tgdn_verify_recurrent.argtypes = [P(CTree), P(CDims), vp, vp, vp, vp, vp, vp, vp, st]
        L.tgdn_verify_recurrent.restype = ctypes.c_int
        L.tgdn_verify_noalloc.argtypes = [P(CTree), P(CDims), vp, vp, vp, vp, vp, vp, vp, st]
        L.tgdn_verify_noalloc.restype = ctypes.c_int
        L.tgdn_verify_fused.argtypes = [P(CTree), P(CDims), vp, vp, vp, vp, vp, vp, vp, vp,
                                        P(CTree), vp, vp, vp, vp, st]
        L.tgdn_verify_fused.restype = ctypes.c_int
        L.tgdn_tree_build.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                      vp, st]
        L.tgdn_tree_build.restype = ctypes.c_int
        L.tgdn_tree_attention.argtypes = [P(CTree), i32, i32, i32, vp, vp, vp, vp, vp, vp, i32,
                                          ctypes.c_float, vp, vp, ctypes.c_size_t, st]
        L.tgdn_tree_attention.restype = ctypes.c_int
        L.tgdn_tree_attention_workspace_bytes.argtypes = [P(CTree), i32, i32, i32, i32]
        L.tgdn_tree_attention_workspace_bytes.restype = ctypes.c_size_t
        L.tgdn_debug_set_wait_hooks.argtypes = [ctypes.c_uint64, ctypes.c_int32]
        L.tgdn_debug_set_wait_hooks.restype = ctypes.c_int
        L.tgdn_status_string.argtypes = [i32]
        L.tgdn_status_string.restype = ctypes.c_char_p
        L.tgdn_version.argtypes = []
        for f in (L.tgdn_tree_prep, L.tgdn_verify, L.tgdn_accept, L.tgdn_commit, L.tgdn_version):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/tgdn.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(tgdn_\w+)\s*\(", text, re.M)))


def status_string(code: int) -> str:
    return lib().tgdn_status_string(int(code)).decode()


def _check(rc: int, call: str):
    if rc != OK:
        raise TgdnError(rc, call)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, dtype, numel: int, name: str) -> int:
    """Device pointer of a contiguous CUDA tensor holding at least `numel` elements."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (the library takes device pointers)")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, need {numel}")
    return t.data_ptr() if numel > 0 else (t.data_ptr() or None)


@dataclass
class Dims:
    H_qk: int
    H_v: int
    d_k: int
    d_v: int
    io: int = BF16

    def c(self) -> CDims:
        return CDims(self.H_qk, self.H_v, self.d_k, self.d_v, self.io)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.io == BF16 else torch.float32


class Tree:
    """A batch of draft trees on the device plus the metadata tree_prep writes."""

    def __init__(self, cu_nodes: torch.Tensor, parent: torch.Tensor, n_max: int,
                 depth_max: int, T: int | None = None):
        self.B = int(cu_nodes.numel()) - 1
        self.T = int(parent.numel()) if T is None else int(T)
        self.n_max, self.depth_max = int(n_max), int(depth_max)
        self.words = max(1, (self.n_max + 63) // 64)
        dev = cu_nodes.device
        self.cu_nodes, self.parent = cu_nodes, parent
        self.depth = torch.empty(self.T, dtype=torch.int32, device=dev)
        self.order = torch.empty(self.T, dtype=torch.int32, device=dev)
        self.pos = torch.empty(self.T, dtype=torch.int32, device=dev)
        self.anc = torch.empty((self.T, self.words), dtype=torch.int64, device=dev)
        self.status = torch.empty(max(self.B, 0), dtype=torch.int32, device=dev)

    @classmethod
    def from_host(cls, cu_nodes, parent, n_max: int, depth_max: int, device="cuda"):
        cu = torch.as_tensor(cu_nodes, dtype=torch.int32).to(device)
        par = torch.as_tensor(parent, dtype=torch.int32).to(device)
        return cls(cu, par, n_max, depth_max)

    def c(self) -> CTree:
        B, T = self.B, self.T
        return CTree(B, T, self.n_max, self.depth_max, self.words,
                     _dev(self.cu_nodes, torch.int32, B + 1, "cu_nodes"),
                     _dev(self.parent, torch.int32, T, "parent"),
                     _dev(self.depth, torch.int32, T, "depth"),
                     _dev(self.order, torch.int32, T, "order"),
                     _dev(self.pos, torch.int32, T, "pos"),
                     _dev(self.anc, torch.int64, T * self.words, "anc"),
                     _dev(self.status, torch.int32, B, "status"))


def tree_prep(tree: Tree, stream=None) -> None:
    ct = tree.c()
    _check(lib().tgdn_tree_prep(ctypes.byref(ct), _stream(stream)), "tgdn_tree_prep")


def verify_workspace_bytes(tree: Tree, dims: Dims) -> int:
    ct, cd = tree.c(), dims.c()
    return int(lib().tgdn_verify_workspace_bytes(ctypes.byref(ct), ctypes.byref(cd)))


def alloc_workspace(tree: Tree, dims: Dims, device="cuda") -> torch.Tensor:
    n = verify_workspace_bytes(tree, dims)
    if n == 0 and tree.T > 0:
        raise TgdnError(EINVAL, "tgdn_verify_workspace_bytes")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def verify(tree: Tree, dims: Dims, q, k, v, g, b, S0, o, ws, stream=None) -> None:
    T, B = tree.T, tree.B
    io = dims.torch_dtype
    ct, cd = tree.c(), dims.c()
    args = (_dev(q, io, T * dims.H_qk * dims.d_k, "q"), _dev(k, io, T * dims.H_qk * dims.d_k, "k"),
            _dev(v, io, T * dims.H_v * dims.d_v, "v"), _dev(g, torch.float32, T * dims.H_v, "g"),
            _dev(b, torch.float32, T * dims.H_v, "b"),
            _dev(S0, torch.float32, B * dims.H_v * dims.d_k * dims.d_v, "S0"),
            _dev(o, io, T * dims.H_v * dims.d_v, "o"),
            _dev(ws, torch.uint8, verify_workspace_bytes(tree, dims), "ws"))
    _check(lib().tgdn_verify(ctypes.byref(ct), ctypes.byref(cd), *args, _stream(stream)),
           "tgdn_verify")


def verify_fused(tree: Tree, dims: Dims, q, k, v, g, b, S, o, ws, prev_tree: Tree,
                 prev_accept_node, prev_path, prev_k, prev_ws, stream=None) -> None:
    """tgdn_verify_fused: commit the previous step's accepted node into S (in place),
    then verify this step's tree from the committed state."""
    T, B = tree.T, tree.B
    io = dims.torch_dtype
    ct, cd, pt = tree.c(), dims.c(), prev_tree.c()
    args = (_dev(q, io, T * dims.H_qk * dims.d_k, "q"), _dev(k, io, T * dims.H_qk * dims.d_k, "k"),
            _dev(v, io, T * dims.H_v * dims.d_v, "v"), _dev(g, torch.float32, T * dims.H_v, "g"),
            _dev(b, torch.float32, T * dims.H_v, "b"),
            _dev(S, torch.float32, B * dims.H_v * dims.d_k * dims.d_v, "S"),
            _dev(o, io, T * dims.H_v * dims.d_v, "o"),
            _dev(ws, torch.uint8, verify_workspace_bytes(tree, dims), "ws"))
    prev = (_dev(prev_accept_node, torch.int32, prev_tree.B, "prev_accept_node"),
            _dev(prev_path, torch.int32, prev_tree.B * (prev_tree.depth_max + 1), "prev_path"),
            _dev(prev_k, io, prev_tree.T * dims.H_qk * dims.d_k, "prev_k"),
            _dev(prev_ws, torch.uint8, verify_workspace_bytes(prev_tree, dims), "prev_ws"))
    _check(lib().tgdn_verify_fused(ctypes.byref(ct), ctypes.byref(cd), *args, ctypes.byref(pt),
                                   *prev, _stream(stream)), "tgdn_verify_fused")


def verify_recurrent(tree: Tree, dims: Dims, q, k, v, g, b, S0, o, stream=None) -> None:
    """tgdn_verify_recurrent: the per-branch recurrent baseline (same outputs as verify)."""
    T, B = tree.T, tree.B
    io = dims.torch_dtype
    ct, cd = tree.c(), dims.c()
    args = (_dev(q, io, T * dims.H_qk * dims.d_k, "q"), _dev(k, io, T * dims.H_qk * dims.d_k, "k"),
            _dev(v, io, T * dims.H_v * dims.d_v, "v"), _dev(g, torch.float32, T * dims.H_v, "g"),
            _dev(b, torch.float32, T * dims.H_v, "b"),
            _dev(S0, torch.float32, B * dims.H_v * dims.d_k * dims.d_v, "S0"),
            _dev(o, io, T * dims.H_v * dims.d_v, "o"))
    _check(lib().tgdn_verify_recurrent(ctypes.byref(ct), ctypes.byref(cd), *args,
                                       _stream(stream)), "tgdn_verify_recurrent")


BUILD_MAX_K = 16


def tree_build(root_token, child_logp, child_token, budget: int, w: int, depth_max: int,
               out=None, stream=None) -> dict:
    """tgdn_tree_build: top-w best-first draft trees for a batch of sequences.
    root_token [B] int32, child_logp [B][budget][K] fp32, child_token [B][budget][K] int32.
    Returns (or fills `out` with) parent/token/depth [B][budget] int32, score [B][budget]
    fp32, n_nodes [B] and rounds [B] int32, all on the device."""
    B = root_token.shape[0]
    K = child_logp.shape[-1] if child_logp.dim() == 3 else 0
    dev = root_token.device
    if out is None:
        out = dict(parent=torch.empty((B, budget), dtype=torch.int32, device=dev),
                   token=torch.empty((B, budget), dtype=torch.int32, device=dev),
                   score=torch.empty((B, budget), dtype=torch.float32, device=dev),
                   depth=torch.empty((B, budget), dtype=torch.int32, device=dev),
                   n_nodes=torch.empty(B, dtype=torch.int32, device=dev),
                   rounds=torch.empty(B, dtype=torch.int32, device=dev))
    nt = B * budget * K
    args = (_dev(root_token, torch.int32, B, "root_token"),
            _dev(child_logp, torch.float32, nt, "child_logp"),
            _dev(child_token, torch.int32, nt, "child_token"),
            _dev(out["parent"], torch.int32, B * budget, "parent"),
            _dev(out["token"], torch.int32, B * budget, "token"),
            _dev(out["score"], torch.float32, B * budget, "score"),
            _dev(out["depth"], torch.int32, B * budget, "depth"),
            _dev(out["n_nodes"], torch.int32, B, "n_nodes"),
            _dev(out["rounds"], torch.int32, B, "rounds"))
    _check(lib().tgdn_tree_build(B, budget, K, w, depth_max, *args, _stream(stream)),
           "tgdn_tree_build")
    return out


def tree_attention_workspace_bytes(tree: Tree, H_q: int, H_kv: int, d: int, P_max: int) -> int:
    return int(lib().tgdn_tree_attention_workspace_bytes(ctypes.byref(tree.c()), H_q, H_kv, d,
                                                         P_max))


def tree_attention(tree: Tree, q, k_tree, v_tree, k_cache, v_cache, prefix_len, o,
                   scale: float, ws=None, stream=None) -> None:
    """tgdn_tree_attention: each node attends to its sequence's cached context and its
    own root path.  q/o [T][H_q][d], k_tree/v_tree [T][H_kv][d], k_cache/v_cache
    [B][P_max][H_kv][d] (bf16), prefix_len [B] int32; scale positive and finite (the
    logits are scale * q.k).  ws: optional uint8 workspace of
    tree_attention_workspace_bytes() bytes (splits the cached context over more CTAs)."""
    T, B = tree.T, tree.B
    H_q, d = q.shape[1], q.shape[2]
    H_kv = k_tree.shape[1]
    P_max = k_cache.shape[1] if k_cache is not None else 0
    bf = torch.bfloat16
    ncache = B * P_max * H_kv * d
    args = (_dev(q, bf, T * H_q * d, "q"), _dev(k_tree, bf, T * H_kv * d, "k_tree"),
            _dev(v_tree, bf, T * H_kv * d, "v_tree"),
            _dev(k_cache, bf, ncache, "k_cache") if P_max > 0 else None,
            _dev(v_cache, bf, ncache, "v_cache") if P_max > 0 else None,
            _dev(prefix_len, torch.int32, B, "prefix_len"))
    wsp, wsn = None, 0
    if ws is not None:
        wsn = ws.numel() * ws.element_size()
        wsp = _dev(ws, ws.dtype, ws.numel(), "ws") if wsn > 0 else None
    _check(lib().tgdn_tree_attention(ctypes.byref(tree.c()), H_q, H_kv, d, *args, P_max,
                                     float(scale), _dev(o, bf, T * H_q * d, "o"), wsp, wsn,
                                     _stream(stream)), "tgdn_tree_attention")


def accept(tree: Tree, draft_ids, target_ids, accept_node, accept_len, path, stream=None) -> None:
    T, B = tree.T, tree.B
    ct = tree.c()
    args = (_dev(draft_ids, torch.int32, T, "draft_ids"),
            _dev(target_ids, torch.int32, T, "target_ids"),
            _dev(accept_node, torch.int32, B, "accept_node"),
            _dev(accept_len, torch.int32, B, "accept_len"),
            _dev(path, torch.int32, B * (tree.depth_max + 1), "path"))
    _check(lib().tgdn_accept(ctypes.byref(ct), *args, _stream(stream)), "tgdn_accept")


def commit(tree: Tree, dims: Dims, accept_node, k, ws, S_in, S_out, stream=None) -> None:
    T, B = tree.T, tree.B
    ct, cd = tree.c(), dims.c()
    ns = B * dims.H_v * dims.d_k * dims.d_v
    args = (_dev(accept_node, torch.int32, B, "accept_node"),
            _dev(k, dims.torch_dtype, T * dims.H_qk * dims.d_k, "k"),
            _dev(ws, torch.uint8, verify_workspace_bytes(tree, dims), "ws"),
            _dev(S_in, torch.float32, ns, "S_in"), _dev(S_out, torch.float32, ns, "S_out"))
    _check(lib().tgdn_commit(ctypes.byref(ct), ctypes.byref(cd), *args, _stream(stream)),
           "tgdn_commit")


def verify_noalloc(tree: Tree, dims: Dims, q, k, v, g, b, S0, o, stream=None) -> None:
    """tgdn_verify_noalloc: verification for callers that cannot allocate device memory.

    Same outputs as verify(); the factors stay in a library-owned device array of
    NOALLOC_SCRATCH_BYTES (so they cannot be committed from).  Calls on one device share
    that array: keep them ordered on one stream."""
    T, B = tree.T, tree.B
    io = dims.torch_dtype
    ct, cd = tree.c(), dims.c()
    args = (_dev(q, io, T * dims.H_qk * dims.d_k, "q"), _dev(k, io, T * dims.H_qk * dims.d_k, "k"),
            _dev(v, io, T * dims.H_v * dims.d_v, "v"), _dev(g, torch.float32, T * dims.H_v, "g"),
            _dev(b, torch.float32, T * dims.H_v, "b"),
            _dev(S0, torch.float32, B * dims.H_v * dims.d_k * dims.d_v, "S0"),
            _dev(o, io, T * dims.H_v * dims.d_v, "o"))
    _check(lib().tgdn_verify_noalloc(ctypes.byref(ct), ctypes.byref(cd), *args, _stream(stream)),
           "tgdn_verify_noalloc")


def debug_set_wait_hooks(wait_limit_ns: int = 0, withhold_item: int = -1) -> None:
    """tgdn_debug_set_wait_hooks: a test hook that shortens the bounded device waits of the
    64-node verification kernel and makes its producer withhold one work item's first
    product, so that the consumer's wait expires (TGDN_SEQ_TIMEOUT, no fault or hang).
    debug_set_wait_hooks() restores the defaults."""
    _check(lib().tgdn_debug_set_wait_hooks(int(wait_limit_ns), int(withhold_item)),
           "tgdn_debug_set_wait_hooks")
