"""Benchmark: verified tree nodes/s per GDN layer on one GB300 (or N, weak scaling).

Workload (default): the 36-layer stack — 32 sequences per GPU, each a 64-node
random draft tree of depth <= 12, H_qk = 16, H_v = 32, d_k = d_v = 128, bf16
q/k/v, fp32 states (one per layer and v-head).  One step is one decode
iteration through the library's C ABI.  Default (--mode fused), the commit of
the previous step's accepted node is folded into this step's verify:
    tgdn_tree_prep -> 36 x tgdn_verify_fused -> tgdn_accept
(--mode separate: tgdn_tree_prep -> 36 x tgdn_verify -> tgdn_accept ->
36 x tgdn_commit in place), captured once per distinct step input into a CUDA
graph and replayed.
Inputs are seeded synthetic data resident in HBM; a step touches ~9 GB, far
more than the 129 MB L2, so no flush is needed between steps.

value  = 36 * B * N_nodes * steps * world / max-over-ranks elapsed time
         (the rate at which one layer's worth of tree nodes is verified).
e2e    = the same metric with the step's inputs copied from pinned host memory
         to the device and the accepted paths copied back, inside the timed
         region, every step.
roofline: the dominant kernel's algorithmic bytes per launch over its
         CUDA-event duration, against the measured HBM copy bandwidth.

--impl reference times the fp64 CPU oracle (path replay, all host cores) on a
bounded sample of the same workload, in the same metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tree_speculative_decoding_gated_gb300 import synth  # noqa: E402

CONFIG = "cfg5"
METRIC = "verified tree nodes/sec per GDN layer (1 GB300); achieved HBM GB/s % of peak"
UNIT = "nodes/s/layer"
S0_BYTES_PER_SEQ = 32 * 128 * 128 * 4                     # one layer's state of one sequence
NODE_BYTES = 2 * 16 * 128 * 2 + 32 * 128 * 2 + 2 * 32 * 4 + 32 * 128 * 2   # q,k,v,g,b in + o out
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant kernel from an ncu
# capture, with the first 16 hex digits of the SHA-256 of the kernel source it was taken on;
# the line reports it only while the source still has that hash (null otherwise).
PROFILED_TRAFFIC = {"fused": (165890816, "c6c75188da3bc32c"), "separate": (None, "")}
KERNEL_SOURCE = os.path.join(ROOT, "tree_speculative_decoding_gated_gb300", "csrc", "verify_tc.cu")


def profiled_traffic(mode: str):
    import hashlib
    value, digest = PROFILED_TRAFFIC[mode]
    if value is None:
        return None
    with open(KERNEL_SOURCE, "rb") as f:
        return value if hashlib.sha256(f.read()).hexdigest()[:16] == digest else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tgdn", choices=["tgdn", "reference"])
    ap.add_argument("--inputs", type=int, default=3,
                    help="distinct step inputs cycled through (3 lets the e2e leg copy the "
                         "next step's inputs while the current step runs)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the one-layer workload summary of the default line")
    ap.add_argument("--cpu-sample-seqs", type=int, default=4)
    ap.add_argument("--layers", type=int, default=36,
                    help="GDN layers per step (fewer only for small profiler captures)")
    ap.add_argument("--mode", default="fused", choices=["fused", "separate"],
                    help="fused: commit folded into the next step's verify; separate: own pass")
    ap.add_argument("--part", default="stack",
                    choices=["stack", "recurrent", "build", "attention", "configs"],
                    help="stack: the decode benchmark (default); recurrent: single-pass verify "
                         "vs per-branch recurrent verify by tree size; build: top-w tree "
                         "construction kernel times; attention: ancestor-masked tree "
                         "attention kernel times; configs: verify and commit per launch on "
                         "the single-layer workloads, with the oracle's time beside them")
    return ap.parse_args()


def shard_range(n_units: int, world: int, rank: int) -> range:
    """Contiguous, balanced share of `n_units` independent units (sequences) for `rank`.
    Sequences never exchange data on this path, so ranks need no collective."""
    base, extra = divmod(n_units, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def max_over_ranks(value: float, world: int) -> float:
    """The slowest rank's elapsed time (the only cross-rank reduction the benchmark does)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"tgdn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names[1:], parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- GPU arm
class StepInput:
    """One decode step's inputs for all layers, resident on the device in one flat buffer
    (so that the e2e leg moves a step's inputs with a single host-to-device copy)."""

    def __init__(self, cfg, step, layers, gen, device, tgdn, torch):
        trees = synth.make_trees(cfg, step)
        draft, target = synth.make_ids(cfg, trees, step)
        self.host_tree = trees
        T = trees.T
        parts = [torch.from_numpy(trees.cu_nodes).to(device),
                 torch.from_numpy(trees.parent).to(device),
                 torch.from_numpy(draft).to(device), torch.from_numpy(target).to(device)]
        per_layer = [synth.make_node_inputs_device(cfg, T, gen, device) for _ in range(layers)]
        for f in range(5):                 # q, k, v, g, b of every layer
            parts += [lay[f] for lay in per_layer]
        offs, total = [], 0
        for t in parts:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.flat = torch.empty(total, dtype=torch.uint8, device=device)
        views = []
        for t, off in zip(parts, offs):
            nb = t.numel() * t.element_size()
            v = self.flat[off:off + nb].view(t.dtype).view(t.shape)
            v.copy_(t)
            views.append(v)
        del parts, per_layer
        cu, parent, self.draft, self.target = views[:4]
        self.tree = tgdn.Tree(cu, parent, trees.n_max, trees.depth_max)
        L = layers
        rest = views[4:]
        self.q, self.k, self.v = rest[:L], rest[L:2 * L], rest[2 * L:3 * L]
        self.g, self.b = rest[3 * L:4 * L], rest[4 * L:5 * L]

    def tensors(self):
        return [self.tree.cu_nodes, self.tree.parent, self.draft, self.target,
                *self.q, *self.k, *self.v, *self.g, *self.b]


def run_gpu(args, rank, world, local):
    import torch
    from tree_speculative_decoding_gated_gb300 import tgdn

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = synth.CONFIGS[CONFIG]
    L, B, Nn = args.layers, cfg.B, cfg.n_nodes
    fused = args.mode == "fused"
    dims = tgdn.Dims(cfg.H_qk, cfg.H_v, cfg.dk, cfg.dv, tgdn.BF16)
    gen = torch.Generator(device=device)
    gen.manual_seed(synth.BASE_SEED + cfg.number + 1000 + 7919 * rank)

    # fused mode needs two inputs at least: a step's workspace must not be the previous one's
    R = max(2 if fused else 1, args.inputs)
    inputs = [StepInput(cfg, r + R * rank, L, gen, device, tgdn, torch) for r in range(R)]
    states = [synth.make_state_device(cfg, B, gen, device) for _ in range(L)]
    T = inputs[0].tree.T
    ws_bytes = tgdn.verify_workspace_bytes(inputs[0].tree, dims)
    # workspaces and acceptance outputs per distinct input (fused: step r commits from r - 1)
    n_ws = R if fused else 1
    ws = [[torch.empty(ws_bytes, dtype=torch.uint8, device=device) for _ in range(L)]
          for _ in range(n_ws)]
    outs = [torch.empty((T, cfg.H_v, cfg.dv), dtype=torch.bfloat16, device=device)
            for _ in range(L)]
    an = [torch.empty(B, dtype=torch.int32, device=device) for _ in range(n_ws)]
    al = [torch.empty(B, dtype=torch.int32, device=device) for _ in range(n_ws)]
    path = [torch.empty((B, cfg.depth_max + 1), dtype=torch.int32, device=device)
            for _ in range(n_ws)]

    stream = torch.cuda.Stream(device)

    def step_separate(r: int, verifies_only=False, commits_only=False):
        inp = inputs[r]
        if not commits_only:
            if not verifies_only:
                tgdn.tree_prep(inp.tree, stream)
            for l in range(L):
                tgdn.verify(inp.tree, dims, inp.q[l], inp.k[l], inp.v[l], inp.g[l], inp.b[l],
                            states[l], outs[l], ws[0][l], stream)
            if verifies_only:
                return
            tgdn.accept(inp.tree, inp.draft, inp.target, an[0], al[0], path[0], stream)
        for l in range(L):
            tgdn.commit(inp.tree, dims, an[0], inp.k[l], ws[0][l], states[l], states[l], stream)

    def step_fused(r: int, verifies_only=False):
        inp, pr = inputs[r], (r - 1) % R
        prev = inputs[pr]
        if not verifies_only:
            tgdn.tree_prep(inp.tree, stream)
        for l in range(L):
            tgdn.verify_fused(inp.tree, dims, inp.q[l], inp.k[l], inp.v[l], inp.g[l], inp.b[l],
                              states[l], outs[l], ws[r][l], prev.tree, an[pr], path[pr],
                              prev.k[l], ws[pr][l], stream)
        if not verifies_only:
            tgdn.accept(inp.tree, inp.draft, inp.target, an[r], al[r], path[r], stream)

    def first_step(r: int):
        """A plain verify + accept of input r, so that the step after it has a commit pending."""
        inp = inputs[r]
        tgdn.tree_prep(inp.tree, stream)
        for l in range(L):
            tgdn.verify(inp.tree, dims, inp.q[l], inp.k[l], inp.v[l], inp.g[l], inp.b[l],
                        states[l], outs[l], ws[r][l], stream)
        tgdn.accept(inp.tree, inp.draft, inp.target, an[r], al[r], path[r], stream)

    step = step_fused if fused else step_separate

    # capture one graph per distinct step input
    graphs = []
    with torch.cuda.stream(stream):
        if fused:
            first_step(R - 1)
        for r in range(R):        # warm the launch path before capture
            step(r)
        stream.synchronize()
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(r)
            graphs.append(g)
        # the verify launches of one step alone (as in the step graph, programmatic
        # dependent launch between them), for the dominant kernel's per-launch time
        vgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(vgraph, stream=stream):
            step(0, verifies_only=True)
        if fused:                 # leave input R - 1 as the last step run
            for r in range(R):
                step(r)
    torch.cuda.synchronize()
    launches_per_step = (1 + L + 1) if fused else (1 + L + 1 + L)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def timed(fn, K, W):
        """W warm-up steps, then K timed ones; step s runs input s % R, so the inputs follow
        each other in order across the warm-up and the timed region."""
        for s in range(W):
            fn(s)
        barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for s in range(W, W + K):
            fn(s)
        t1.record(stream)
        barrier()
        return max_over_ranks(t0.elapsed_time(t1), world)

    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.nvtx.range_push("timed")
    # W warm-up and K timed replays in input order from input 0 (the setup left input
    # R - 1 as the last step run, so each step commits its predecessor's acceptance)
    K, W = args.steps, args.warmup

    def replay(s):
        with torch.cuda.stream(stream):   # a graph replays on the current stream
            graphs[s % R].replay()

    ms = timed(replay, K, W)
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    with torch.cuda.stream(stream):       # end again on input R - 1 (for the legs below)
        for s in range(W + K, W + K + (-(W + K)) % R):
            graphs[s % R].replay()
    stream.synchronize()

    # The dominant kernel's launch time: the graph of one step's verify launches replayed
    # (back to back, as inside the step graph), divided by the launches it holds.
    def graph_us(g, n, reps=10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        return 1e3 * e0.elapsed_time(e1) / (reps * n)

    verify_us = graph_us(vgraph, L)
    if not fused:
        cgraph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(cgraph, stream=stream):
                step_separate(0, commits_only=True)
        commit_us = graph_us(cgraph, L)
    if fused:                              # the verify-only replays used input 0's step
        with torch.cuda.stream(stream):
            for r in range(1, R):
                graphs[r].replay()
        stream.synchronize()

    total_nodes = L * B * Nn * K * world
    value = total_nodes / (ms / 1e3)
    hbm, peak_kind = peaks()
    verify_bytes = B * S0_BYTES_PER_SEQ + B * Nn * NODE_BYTES
    commit_bytes = 2 * B * S0_BYTES_PER_SEQ
    if fused:
        # the fused pass also writes the committed state back (the path factors it reads,
        # under 1% of the state, are not counted)
        fv_bytes = verify_bytes + B * S0_BYTES_PER_SEQ
        dom = dict(kernel="verify_tc_kernel (with the deferred commit)", us=verify_us,
                   bytes=fv_bytes, gbs=fv_bytes / (verify_us * 1e-6) / 1e9)
        other = None
    else:
        v_gbs = verify_bytes / (verify_us * 1e-6) / 1e9
        c_gbs = commit_bytes / (commit_us * 1e-6) / 1e9
        vd = dict(kernel="verify_tc_kernel", us=verify_us, bytes=verify_bytes, gbs=v_gbs)
        cd = dict(kernel="commit128_kernel", us=commit_us, bytes=commit_bytes, gbs=c_gbs)
        dom, other = (vd, cd) if verify_us >= commit_us else (cd, vd)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, inputs, graphs, stream, an, al, path, timed, torch, R, L, B, Nn,
                      world)

    touched_gb = L * (dom["bytes"] + (0 if fused else commit_bytes)) / 1e9
    step_desc = (f"prep + {L} verify with the previous step's commit folded in + accept"
                 if fused else f"prep + {L} verify + accept + {L} in-place commit")
    roof = {"bound": "hbm", "kernel": dom["kernel"], "achieved": dom["gbs"], "peak": hbm,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": dom["gbs"] / hbm,
            "traffic": profiled_traffic(args.mode),
            "algorithmic_bytes_per_launch": dom["bytes"], "launch_us": dom["us"]}
    if other is not None:
        roof["other"] = {"kernel": other["kernel"], "achieved": other["gbs"],
                         "frac": other["gbs"] / hbm, "launch_us": other["us"],
                         "algorithmic_bytes_per_launch": other["bytes"]}
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{L}-layer GDN stack, B={B} per GPU, 64-node random trees "
                               f"(depth<=12), H_qk=16 H_v=32 d=128; {K} decode steps timed "
                               f"after {W} warm-up steps",
                   "timed_steps": K, "warmup_steps": W,
                   "layers": L, "batch_per_gpu": B, "nodes_per_tree": Nn, "depth_max": 12,
                   "H_qk": 16, "H_v": 32, "d_k": 128, "d_v": 128, "io": "bf16",
                   "state": "fp32", "accumulate": "fp32", "mode": args.mode,
                   "step": f"{step_desc} (CUDA graph)",
                   "l2": f"inputs larger than L2 (~{touched_gb:.1f} GB touched per step, "
                         f"L2 129 MB)",
                   "distinct_step_inputs": R, "parallelism": f"dp{world} (sequences)"},
        "roofline": roof,
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    if e2e is not None:
        # the end-to-end step can be no faster than its host-to-device bytes at the
        # measured link rate, nor than the device step
        e2e["bound_ms_per_step"] = max(ms / K, e2e["link_ms_per_step"])
        result["e2e"] = e2e
    return result


def run_e2e(args, inputs, graphs, stream, an, al, path, timed, torch, R, L, B, Nn, world):
    """Same step, but each step's inputs come from pinned host memory and the accepted
    paths go back to the host, inside the timed region.  an/al/path: the acceptance
    outputs per input (one shared set when there is a single one).

    A step's inputs live in one flat buffer and cross in one copy.  With at least three
    distinct inputs the host-to-device copy of step s runs on a copy stream while step
    s - 1 computes: it only waits for step s - 2, the last one that reads the same
    buffer (as its own inputs or, in the fused step, as the previous step's keys).
    Step s waits for its copy."""
    host = [inp.flat.to("cpu").pin_memory() for inp in inputs]   # one buffer per step
    res_host = [torch.empty_like(x, device="cpu").pin_memory() for x in (an[0], al[0], path[0])]
    h2d = host[0].numel()
    d2h = sum(t.numel() * t.element_size() for t in res_host)
    overlap = R >= 3
    copy_stream = torch.cuda.Stream(stream.device) if overlap else stream
    ev_copied = [torch.cuda.Event() for _ in range(R)]
    ev_done = [torch.cuda.Event() for _ in range(R)]
    done_recorded = [False] * R

    def fn(s):
        r = s % R
        a = r if len(an) > 1 else 0
        with torch.cuda.stream(copy_stream):
            if overlap and s >= 2 and done_recorded[(s - 2) % R]:
                copy_stream.wait_event(ev_done[(s - 2) % R])
            inputs[r].flat.copy_(host[r], non_blocking=True)
            if overlap:
                ev_copied[r].record(copy_stream)
        with torch.cuda.stream(stream):
            if overlap:
                stream.wait_event(ev_copied[r])
            graphs[r].replay()
            for dst, src in zip(res_host, (an[a], al[a], path[a])):
                dst.copy_(src, non_blocking=True)
            if overlap:
                ev_done[r].record(stream)
                done_recorded[r] = True

    # The host link's own rate: one step's inputs, pinned, in one copy (best of 3, untimed
    # for the metric); then input 0's buffer is restored from its host copy.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    link_ms = float("inf")
    with torch.cuda.stream(copy_stream):
        for _ in range(3):
            e0.record(copy_stream)
            inputs[0].flat.copy_(host[0], non_blocking=True)
            e1.record(copy_stream)
            copy_stream.synchronize()
            link_ms = min(link_ms, e0.elapsed_time(e1))
    torch.cuda.synchronize()
    # the previous leg ended on input R - 1, so step 0 (input 0) commits its own predecessor
    ms = timed(fn, args.steps, args.warmup)
    value = L * B * Nn * args.steps * world / (ms / 1e3)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms / args.steps,
            "link_h2d_gbs": h2d / (link_ms * 1e-3) / 1e9, "link_ms_per_step": link_ms,
            "copies": "one copy per step, overlapped with the previous step" if overlap
                      else "serial with the step"}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(n_seqs: int, step: int = 0, layer: int = 0):
    """A bounded slice of the workload: n_seqs whole sequences of one layer, all heads."""
    p = synth.make_problem(CONFIG, step=step, layer=layer)
    return synth.select_sequences(p, range(n_seqs))


def time_oracle(n_seqs: int, step: int = 0):
    import oracle
    sub = oracle_sample(n_seqs, step=step)
    t, i = sub.trees, sub.inputs
    t0 = time.perf_counter()
    o, used = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v, i.g, i.b,
                            sub.S0, return_threads=True)
    acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, sub.draft_ids,
                        sub.target_ids)
    oracle.commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b, sub.S0,
                  acc["accept_node"])
    dt = time.perf_counter() - t0
    return t.T, dt, used


def cpu_baseline(min_seconds: float = 10.0, max_layers: int = 36):
    """The oracle on whole layers of step 0 (all 32 sequences, all heads), layer after layer
    until at least `min_seconds` of CPU work has been timed."""
    import oracle
    cfg = synth.CONFIGS[CONFIG]
    nodes, dt, used, layers = 0, 0.0, 1, 0
    while layers < max_layers and dt < min_seconds:
        p = synth.make_problem(CONFIG, step=0, layer=layers)
        t, i = p.trees, p.inputs
        t0 = time.perf_counter()
        _, used = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v, i.g,
                                i.b, p.S0, return_threads=True)
        acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, p.draft_ids,
                            p.target_ids)
        oracle.commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b, p.S0,
                      acc["accept_node"])
        dt += time.perf_counter() - t0
        nodes += t.T
        layers += 1
    # one core, on 2 sequences of layer 0 (the same work per node)
    p = synth.select_sequences(synth.make_problem(CONFIG, step=0, layer=0), range(2))
    t, i = p.trees, p.inputs
    t0 = time.perf_counter()
    oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v, i.g, i.b, p.S0, 1)
    acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, p.draft_ids, p.target_ids)
    oracle.commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b, p.S0,
                  acc["accept_node"], 1)
    dt1 = time.perf_counter() - t0
    return {"value": nodes / dt, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{layers} of 36 layers of step 0, all {cfg.B} sequences x 64 nodes x "
                      f"32 v-heads: verify + accept + commit by fp64 path replay "
                      f"({dt:.1f} s)",
            "seconds": dt,
            "one_core": {"value": t.T / dt1, "unit": UNIT, "cores": 1,
                         "sample": f"2 sequences of layer 0, step 0 ({t.T} nodes x 32 v-heads, "
                                   f"{dt1:.1f} s)"}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.lib()
    n = args.cpu_sample_seqs
    for _ in range(args.warmup if args.warmup <= 1 else 1):
        time_oracle(1)
    total_nodes, total_s, used = 0, 0.0, 1
    for s in range(args.steps):
        nodes, dt, used = time_oracle(n, step=s)
        total_nodes += nodes
        total_s += dt
    value = total_nodes / total_s
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "36-layer GDN stack, 64-node random trees (depth<=12), "
                                   "H_qk=16 H_v=32 d=128; each step a bounded sample",
                       "sample_per_step": f"{n} sequences x 32 v-heads, one layer"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": f"{n} sequences of one layer per step, {args.steps} steps"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def _flush_l2(buf):
    buf.add_(1)          # 256 MiB written: nothing of the previous launch stays in L2


def _launch_times(torch, stream, fn, iters, flush):
    """Per-launch device times (us) with L2 flushed before every launch.  A ~100 us spin on
    the GPU after the flush keeps the stream busy while the host enqueues the call, so
    the events bracket the launch's device time and not the host's work for it (tensor
    maps, launch setup)."""
    ts = []
    for _ in range(iters):
        with torch.cuda.stream(stream):
            _flush_l2(flush)
            torch.cuda._sleep(200_000)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
        stream.synchronize()
        ts.append(1e3 * e0.elapsed_time(e1))
    return statistics.median(ts)


def run_recurrent_compare(args):
    """Single-pass tree verification (tgdn_verify) against per-branch recurrent verification
    (tgdn_verify_recurrent) on one GDN layer, by tree size: the pages' comparison at tree
    size 128 (7.1x on a B200)."""
    import torch
    from tree_speculative_decoding_gated_gb300 import tgdn
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    cfg = synth.CONFIGS["cfg3"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(synth.BASE_SEED + 77)
    stream = torch.cuda.Stream(dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    dims = tgdn.Dims(cfg.H_qk, cfg.H_v, cfg.dk, cfg.dv, tgdn.BF16)
    B = 16
    rng = np.random.default_rng(synth.BASE_SEED + 78)
    cases = [("random", n, 16) for n in (16, 32, 64)] + [("random", 128, 16), ("top-8", 129, 16)]
    out = []
    for kind, n, dcap in cases:
        if kind == "top-8":
            parents = [synth.top_m_tree(rng, 8, 16) for _ in range(B)]
        else:
            parents = [synth.random_recursive_tree(rng, n, dcap) for _ in range(B)]
        trees = synth.pack_trees(parents, max(len(p) for p in parents), dcap)
        tree = tgdn.Tree.from_host(trees.cu_nodes, trees.parent, trees.n_max, trees.depth_max,
                                   dev)
        q, k, v, g, b = synth.make_node_inputs_device(cfg, trees.T, gen, dev)
        S0 = synth.make_state_device(cfg, B, gen, dev)
        o = torch.empty((trees.T, cfg.H_v, cfg.dv), dtype=torch.bfloat16, device=dev)
        ws = tgdn.alloc_workspace(tree, dims, dev)
        with torch.cuda.stream(stream):
            tgdn.tree_prep(tree, stream)
        f_single = lambda: tgdn.verify(tree, dims, q, k, v, g, b, S0, o, ws, stream)
        f_rec = lambda: tgdn.verify_recurrent(tree, dims, q, k, v, g, b, S0, o, stream)
        for f in (f_single, f_rec):
            with torch.cuda.stream(stream):
                for _ in range(3):
                    f()
        t1 = _launch_times(torch, stream, f_single, 20, flush)
        t2 = _launch_times(torch, stream, f_rec, 20, flush)
        kern = ("verify_tc_kernel" if trees.n_max <= 64 else
                "verify_tc_kernel (<= 64-node sequences) + verify_tc128_kernel" if trees.n_max <= 129
                else "verify_simt_kernel")
        out.append({"tree": kind, "nodes": int(trees.n_max), "depth_max": dcap, "B": B,
                    "single_pass_us": t1, "single_pass_kernel": kern, "recurrent_us": t2,
                    "ratio": t2 / t1})
    return {"part": "recurrent", "metric": "per-branch recurrent time / single-pass time, "
            "one GDN layer (H_qk=16, H_v=32, d=128, bf16), L2 flushed before every launch",
            "unit": "x", "higher_is_better": True, "cases": out,
            "pages": "7.1x at tree size 128 on a B200 (Experimentelle Ergebnisse)"}


def run_build_times(args):
    """Top-w best-first tree construction (tgdn_tree_build): kernel time per batch."""
    import torch
    from tree_speculative_decoding_gated_gb300 import tgdn
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    out = []
    for B, budget, K, w, dmax in [(32, 64, 8, 1, 12), (32, 64, 8, 4, 12), (32, 64, 8, 8, 12),
                                  (32, 64, 8, 16, 12), (32, 128, 8, 8, 16),
                                  (32, 256, 16, 16, 30), (256, 64, 8, 8, 12)]:
        root, logp, tok = synth.make_build_tables(B, budget, K, seed=budget + w)
        d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        r, lp, tk = d(root), d(logp), d(tok)
        res = tgdn.tree_build(r, lp, tk, budget, w, dmax, stream=stream)
        fn = lambda: tgdn.tree_build(r, lp, tk, budget, w, dmax, out=res, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        t = _launch_times(torch, stream, fn, 20, flush)
        rounds = int(res["rounds"].max().item())
        out.append({"B": B, "budget": budget, "K": K, "w": w, "depth_max": dmax, "us": t,
                    "rounds": rounds, "us_per_round": t / max(rounds, 1)})
    return {"part": "build", "metric": "tgdn_tree_build kernel time per batch (one warp per "
            "sequence; latency bound)", "unit": "us", "higher_is_better": False, "cases": out}


def run_attention_times(args):
    """Ancestor-masked tree attention (tgdn_tree_attention): kernel time per layer and its
    rates against the measured peaks (the cached context is the dominant stream)."""
    import torch
    from tree_speculative_decoding_gated_gb300 import tgdn
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(synth.BASE_SEED + 91)
    rng = np.random.default_rng(synth.BASE_SEED + 92)
    hbm, kind = peaks()
    out = []
    for B, N, H_q, H_kv, P in [(16, 64, 16, 4, 1024), (16, 64, 16, 4, 4096), (32, 64, 16, 4, 4096),
                               (16, 128, 16, 4, 4096)]:
        parents = [synth.random_recursive_tree(rng, N, 16) for _ in range(B)]
        trees = synth.pack_trees(parents, N, 16)
        tree = tgdn.Tree.from_host(trees.cu_nodes, trees.parent, N, 16, dev)
        T = trees.T
        rnd = lambda *shape: torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)
        q, kt, vt = rnd(T, H_q, 128), rnd(T, H_kv, 128), rnd(T, H_kv, 128)
        kc, vc = rnd(B, P, H_kv, 128), rnd(B, P, H_kv, 128)
        pl = torch.full((B,), P, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        nb = tgdn.tree_attention_workspace_bytes(tree, H_q, H_kv, 128, P)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            tgdn.tree_prep(tree, stream)
        fn = lambda: tgdn.tree_attention(tree, q, kt, vt, kc, vc, pl, o, 128 ** -0.5, ws=ws,
                                         stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        t = _launch_times(torch, stream, fn, 20, flush)
        depth = np.concatenate([synth.tree_depths(p) for p in parents])
        keys = float(P * T + (depth + 1).sum())  # visible keys per node (one q head)
        flops = 4.0 * 128 * keys * H_q           # QK^T and PV, 2 flops per multiply-add
        cache_bytes = 2 * B * P * H_kv * 128 * 2
        node_bytes = T * (2 * H_q + 2 * H_kv) * 128 * 2
        gbs = (cache_bytes + node_bytes) / (t * 1e-6) / 1e9
        out.append({"B": B, "nodes": N, "H_q": H_q, "H_kv": H_kv, "context": P, "us": t,
                    "context_split": nb > 0,
                    "GB/s": gbs, "frac_hbm": gbs / hbm, "TFLOP/s": flops / (t * 1e-6) / 1e12})
    return {"part": "attention", "metric": "tgdn_tree_attention kernel time per layer, bf16, "
            "d=128, L2 flushed before every launch", "unit": "us", "higher_is_better": False,
            "peak_hbm_gbs": hbm, "peak_kind": kind, "cases": out}


def per_config_summary(hbm):
    """Verify and commit per launch on the one-layer workloads of 16 sequences of 64-node
    trees and of 64 mixed sequences (17-node chains and 129-node trees), L2 flushed before
    every launch, as fractions of the measured HBM bandwidth; and single-pass vs
    per-branch recurrent verification at tree size 128."""
    import torch
    from tree_speculative_decoding_gated_gb300 import tgdn
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    out = {}
    for name in ("cfg3", "cfg4"):
        cfg = synth.CONFIGS[name]
        trees = synth.make_trees(cfg, 0)
        tree = tgdn.Tree.from_host(trees.cu_nodes, trees.parent, trees.n_max, trees.depth_max,
                                   dev)
        dims = tgdn.Dims(cfg.H_qk, cfg.H_v, cfg.dk, cfg.dv, tgdn.BF16)
        gen = torch.Generator(device=dev)
        gen.manual_seed(synth.BASE_SEED + cfg.number + 1000)
        q, k, v, g, b = synth.make_node_inputs_device(cfg, trees.T, gen, dev)
        S0 = synth.make_state_device(cfg, trees.B, gen, dev)
        o = torch.empty((trees.T, cfg.H_v, cfg.dv), dtype=torch.bfloat16, device=dev)
        ws = tgdn.alloc_workspace(tree, dims, dev)
        S = torch.empty_like(S0)
        an = torch.zeros(trees.B, dtype=torch.int32, device=dev)
        with torch.cuda.stream(stream):
            tgdn.tree_prep(tree, stream)
        fv = lambda: tgdn.verify(tree, dims, q, k, v, g, b, S0, o, ws, stream)
        fc = lambda: tgdn.commit(tree, dims, an, k, ws, S0, S, stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fv()
                fc()
        tv = _launch_times(torch, stream, fv, 20, flush)
        tcm = _launch_times(torch, stream, fc, 20, flush)
        vb = trees.B * S0_BYTES_PER_SEQ + trees.T * NODE_BYTES
        cb = 2 * trees.B * S0_BYTES_PER_SEQ
        out[name] = {"verify_us": tv, "verify_frac_hbm": vb / (tv * 1e-6) / 1e9 / hbm,
                     "commit_us": tcm, "commit_frac_hbm": cb / (tcm * 1e-6) / 1e9 / hbm}
    out["recurrent_vs_single_pass_128"] = recurrent_ratio(128)
    return out


def recurrent_ratio(n_nodes: int):
    """Per-branch recurrent over single-pass verification time, one layer of 16 sequences of
    n_nodes-node random trees (depth <= 16), L2 flushed before every launch."""
    import torch
    from tree_speculative_decoding_gated_gb300 import tgdn
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    cfg = synth.CONFIGS["cfg3"]
    rng = np.random.default_rng(synth.BASE_SEED + 78)
    parents = [synth.random_recursive_tree(rng, n_nodes, 16) for _ in range(16)]
    trees = synth.pack_trees(parents, n_nodes, 16)
    tree = tgdn.Tree.from_host(trees.cu_nodes, trees.parent, trees.n_max, trees.depth_max, dev)
    dims = tgdn.Dims(cfg.H_qk, cfg.H_v, cfg.dk, cfg.dv, tgdn.BF16)
    gen = torch.Generator(device=dev)
    gen.manual_seed(synth.BASE_SEED + 77)
    q, k, v, g, b = synth.make_node_inputs_device(cfg, trees.T, gen, dev)
    S0 = synth.make_state_device(cfg, 16, gen, dev)
    o = torch.empty((trees.T, cfg.H_v, cfg.dv), dtype=torch.bfloat16, device=dev)
    ws = tgdn.alloc_workspace(tree, dims, dev)
    with torch.cuda.stream(stream):
        tgdn.tree_prep(tree, stream)
    f1 = lambda: tgdn.verify(tree, dims, q, k, v, g, b, S0, o, ws, stream)
    f2 = lambda: tgdn.verify_recurrent(tree, dims, q, k, v, g, b, S0, o, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            f1()
            f2()
    t1 = _launch_times(torch, stream, f1, 10, flush)
    t2 = _launch_times(torch, stream, f2, 10, flush)
    return {"nodes": n_nodes, "single_pass_us": t1, "recurrent_us": t2, "ratio": t2 / t1,
            "pages": "7.1x at tree size 128 on a B200 (Experimentelle Ergebnisse)"}


def run_config_times(args):
    """tgdn_verify and tgdn_commit per launch on the single-layer workloads (one B=1 top-4
    tree; 16 x 64-node random trees; 64 mixed chains and 129-node top-8 trees), against the
    measured HBM copy bandwidth, with the oracle's all-core time for the same launch."""
    import torch
    import oracle
    from tree_speculative_decoding_gated_gb300 import tgdn
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    hbm, kind = peaks()
    out = []
    for name in ("cfg2", "cfg3", "cfg4"):
        p = synth.make_problem(name)
        cfg, t, i = p.cfg, p.trees, p.inputs
        tree = tgdn.Tree.from_host(t.cu_nodes, t.parent, t.n_max, t.depth_max, dev)
        dims = tgdn.Dims(cfg.H_qk, cfg.H_v, cfg.dk, cfg.dv, tgdn.BF16)
        bf = lambda x: torch.from_numpy(synth.bf16_bits(x)).view(torch.bfloat16).to(dev)
        f32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
        q, k, v, g, b, S0 = bf(i.q), bf(i.k), bf(i.v), f32(i.g), f32(i.b), f32(p.S0)
        o = torch.empty((t.T, cfg.H_v, cfg.dv), dtype=torch.bfloat16, device=dev)
        ws = tgdn.alloc_workspace(tree, dims, dev)
        S = torch.empty_like(S0)
        an = torch.empty(t.B, dtype=torch.int32, device=dev)
        al = torch.empty_like(an)
        path = torch.empty((t.B, t.depth_max + 1), dtype=torch.int32, device=dev)
        draft = torch.from_numpy(p.draft_ids).to(dev)
        target = torch.from_numpy(p.target_ids).to(dev)
        with torch.cuda.stream(stream):
            tgdn.tree_prep(tree, stream)
            tgdn.verify(tree, dims, q, k, v, g, b, S0, o, ws, stream)
            tgdn.accept(tree, draft, target, an, al, path, stream)
        fv = lambda: tgdn.verify(tree, dims, q, k, v, g, b, S0, o, ws, stream)
        fc = lambda: tgdn.commit(tree, dims, an, k, ws, S0, S, stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fv()
                fc()
        tv = _launch_times(torch, stream, fv, 30, flush)
        tcm = _launch_times(torch, stream, fc, 30, flush)
        vb = t.B * S0_BYTES_PER_SEQ + t.T * NODE_BYTES
        cb = 2 * t.B * S0_BYTES_PER_SEQ
        t0 = time.perf_counter()
        _, used = oracle.verify(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.q, i.k, i.v, i.g,
                                i.b, p.S0, return_threads=True)
        acc = oracle.accept(t.cu_nodes, t.parent, t.n_max, t.depth_max, p.draft_ids,
                            p.target_ids)
        oracle.commit(t.cu_nodes, t.parent, t.n_max, t.depth_max, i.k, i.v, i.g, i.b, p.S0,
                      acc["accept_node"])
        t_or = time.perf_counter() - t0
        kern = ("verify_tc_kernel" if t.n_max <= 64 else
                "verify_tc_kernel (<= 64-node sequences) + verify_tc128_kernel" if t.n_max <= 129
                else "verify_simt_kernel")
        out.append({"workload": name, "B": t.B, "nodes": t.T, "verify_kernel": kern,
                    "verify_us": tv, "verify_frac_hbm": vb / (tv * 1e-6) / 1e9 / hbm,
                    "commit_us": tcm, "commit_frac_hbm": cb / (tcm * 1e-6) / 1e9 / hbm,
                    "nodes_per_s_verify": t.T / (tv * 1e-6),
                    "nodes_per_s_verify_commit": t.T / ((tv + tcm) * 1e-6),
                    "oracle_ms": 1e3 * t_or, "oracle_cores": used})
    return {"part": "configs", "metric": "per-launch verify and commit on the single-layer "
            "workloads, L2 flushed before every launch", "unit": "us", "peak_hbm_gbs": hbm,
            "peak_kind": kind, "cases": out}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.part != "stack":
        if rank == 0:
            fn = {"recurrent": run_recurrent_compare, "build": run_build_times,
                  "attention": run_attention_times, "configs": run_config_times}[args.part]
            print(json.dumps(fn(args)), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    res = run_gpu(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_per_config:
        res["per_config"] = per_config_summary(peaks()[0])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
