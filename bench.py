#!/usr/bin/env python
"""Benchmark of the GB300 verify-and-accept path.

Default workload: greedy chain verification, B = 64 requests, k = 5 drafts,
V = 128256, bf16 target logits [64, 6, 128256] drawn N(0, 3^2); each draft
token equals the row argmax with probability 0.8, else uniform.  One step is
one pass of the hot path over that batch: spec_verify_chain_fused, the
verify with the fix-up of the batch's [64, 6] int64 slot_mapping in the same
launch (the oracle's step is the verify followed by the fix-up).

Metric: verified draft positions per second (B * k per step), with the
achieved HBM bandwidth of the verify kernel against the measured copy peak.

Timing: CUDA graphs (one per input copy) replayed on one stream; inputs rotate
over enough device copies that the bytes touched between two uses of a copy
exceed 4x the L2 size, so every step reads its logits from HBM.  CUDA events
bracket exactly K steps, with a barrier and a device synchronisation on both
sides; the time is the max over ranks.

``--impl reference`` times the CPU oracle instead (the only reference this
path has), on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "verified draft positions/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
OTHER_NAMES = ["sampled_chain", "sweep", "greedy_tree", "ragged", "ngram", "sampled_tree", "next_step"]
_CSRC = os.path.join(ROOT, "speculative_decoding_verification_chain_gb300", "csrc")
KERNEL_SRCS = [os.path.join(_CSRC, f) for f in ("spec_verify.cu", "ptx.cuh", "twofloat.cuh")]
# the sources each profiled kernel is compiled from (its profile's hash covers them)
PROFILED_SRCS = {
    "verify_kernel": KERNEL_SRCS,
    "chain_cluster_kernel": [os.path.join(_CSRC, f) for f in ("chain_cluster.cu", "ptx.cuh", "twofloat.cuh")],
    "greedy_cluster_kernel": [os.path.join(_CSRC, f) for f in ("greedy_cluster.cu", "ptx.cuh")],
    "tree_sampled_kernel": [os.path.join(_CSRC, f) for f in ("tree_sampled.cu", "ptx.cuh", "twofloat.cuh")],
}


# ------------------------------------------------------------------ setup --
def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200, help="steps of the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--only", choices=OTHER_NAMES, default=None,
                    help="run just this secondary workload (kernel-only timing) and print its JSON")
    ap.add_argument("--sweep-b", type=int, default=None,
                    help="one batch of the sweep workload (default: B = 1, 8, 64 and 256)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the baseline leg")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: time the verify kernel over exactly --steps launches, no clock sampling")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, use_cuda):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return dist


def reduce_max(dist, value: float, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(srcs=None) -> str:
    """Hash of the code a kernel is compiled from (the verify kernel's by
    default): comments removed and whitespace collapsed, so a change to the code
    (not to its comments) orphans the profiled counters."""
    h = hashlib.sha256()
    for path in (srcs or KERNEL_SRCS):
        with open(path, encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode("utf-8"))
        h.update(b"\0")
    return h.hexdigest()[:16]


def profiled_traffic(name: str, kernel: str = "verify_kernel"):
    """dram read+write bytes per launch from a committed ncu summary, if it was
    taken on the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash(PROFILED_SRCS[kernel]):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while work runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if _isfloat(r[3])) if any(_isfloat(r[3]) for r in rows) else None}


def _isfloat(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


# --------------------------------------------------------------- bytes ---
def chain_bytes(num_accepted, temperature, k, V, s_z):
    """Bytes per launch: algorithmic (rows up to the first rejection; for a
    sampled request rejected before row k also that row's q and one 4-byte q
    gather per accept test), position-parallel (every logits row plus q only at
    the rejection), and dense (every input byte)."""
    a = np.asarray(num_accepted, np.int64)
    sampled = np.asarray(temperature) > 0
    row = V * s_z
    alg = ((a + 1) * row).sum()
    alg += (sampled * (np.minimum(a + 1, k) * 4)).sum()
    alg += (sampled * (a < k) * (V * 4)).sum()
    B = len(a)
    par = B * (k + 1) * row + (sampled * (a < k) * (V * 4)).sum() + (sampled * k * 4).sum()
    dense = B * (k + 1) * row + (sampled.sum() * k * V * 4)
    return float(alg), float(par), float(dense)


def tree_greedy_bytes(parent, node_tokens, g_rows, path, length, V, s_z):
    """Algorithmic bytes of greedy tree verification: per request the root row,
    the row of every accepted node that has children, and the chosen node's row
    (its bonus or correction token).  A node is accepted iff its parent is and
    its token equals the argmax of its parent's row; the GPU's path fixes the
    argmaxes along the path only, so the accepted nodes off it come from the
    row argmaxes g_rows [B, N+1] (first index on ties)."""
    N = len(parent) - 1
    has_child = np.zeros(N + 1, bool)
    has_child[np.asarray(parent)[1:]] = True
    rows = 0
    for b in range(len(length)):
        acc = np.zeros(N + 1, bool)
        acc[0] = True
        for n in range(1, N + 1):
            acc[n] = acc[parent[n]] and node_tokens[b, n - 1] == g_rows[b, parent[n]]
        best = path[b, length[b] - 1]
        rows += sum(1 for n in range(N + 1) if n == 0 or n == best or (acc[n] and has_child[n]))
    return float(rows * V * s_z)


# ------------------------------------------------------------ GPU timing --
def to_dev(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def l2_bytes(dev):
    import torch
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        return 129 * 2 ** 20


class ChainCase:
    """Device copies, outputs and captured graphs of one chain workload."""

    def __init__(self, sv, x, dev, with_fixup=True):
        import torch
        self.sv, self.x, self.dev = sv, x, dev
        sampled = x.draft_probs is not None
        per_copy = x.logits.nbytes + (x.draft_probs.nbytes if sampled else 0)
        self.ncopy = max(2, int(np.ceil(4 * l2_bytes(dev) / per_copy)) + 1)
        self.ncopy = min(self.ncopy, 64)
        self.copies = []
        for _ in range(self.ncopy):
            c = dict(z=to_dev(x.logits, dev), tok=to_dev(x.draft_tokens, dev),
                     slots=to_dev(x.slot_mapping, dev),
                     out=torch.empty((x.B, x.k + 1), dtype=torch.int32, device=dev),
                     na=torch.empty((x.B,), dtype=torch.int32, device=dev))
            if sampled:
                c.update(T=to_dev(x.temperature, dev), ua=to_dev(x.u_accept, dev), us=to_dev(x.u_sample, dev),
                         q=to_dev(x.draft_probs, dev))
            self.copies.append(c)
        code = sv.SPEC_BF16 if x.dtype == 0 else sv.SPEC_FP32
        self.ws = torch.zeros(sv.workspace_bytes(x.B, x.k + 1, x.V, code), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.with_fixup = with_fixup
        self.graphs_step = None
        self.graphs_verify = None

    def _verify(self, c):
        # With the fix-up the step is one launch: the slot_mapping fix-up runs in
        # the verify kernel's request finalisation.  It is idempotent for a fixed
        # num_accepted, so replaying a step on its own (already fixed) slot map
        # does the same work every time.
        return self.sv.verify_chain(c["z"], c["tok"], c.get("T"), c.get("ua"), c.get("us"), c.get("q"),
                                    out_tokens=c["out"], out_num_accepted=c["na"], status=self.status,
                                    workspace=self.ws, slot_mapping=c["slots"] if self.with_fixup else None)

    def _step(self, c, fixup=True):
        self._verify(c)

    def capture(self):
        import torch
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            for c in self.copies:          # eager warm-up outside capture
                self._step(c, self.with_fixup)
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize(self.dev)
        # one graph per copy (for remainders) and one graph that runs one step
        # on every copy in turn, so the host launches one graph per ncopy steps
        self.graphs_step, self.graphs_verify = [], []
        for c in self.copies:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._step(c, self.with_fixup)
            self.graphs_step.append(g)
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2):
                self._verify(c)
            self.graphs_verify.append(g2)
        self.round_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.round_step):
            for c in self.copies:
                self._step(c, self.with_fixup)
        self.round_verify = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.round_verify):
            for c in self.copies:
                self._verify(c)
        torch.cuda.synchronize(self.dev)

    def run(self, steps, verify_only=False):
        """Exactly `steps` steps, rotating over the copies."""
        gs = self.graphs_verify if verify_only else self.graphs_step
        rg = self.round_verify if verify_only else self.round_step
        n = len(gs)
        for _ in range(steps // n):
            rg.replay()
        for i in range(steps % n):
            gs[i].replay()

    def launches_per_step(self):
        return 1   # verify with the fused slot fix-up


def time_steps(case, steps, dev, dist=None, verify_only=False):
    import torch
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    st = torch.cuda.current_stream(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    case.run(steps, verify_only=verify_only)
    e1.record(st)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    ms = e0.elapsed_time(e1)
    return reduce_max(dist, ms, dev)


def e2e_leg(sv, x, dev, steps, dist=None):
    """Host buffers in pinned memory; per step: H2D of the step's inputs, the
    C-ABI verify (slot fix-up fused), D2H of the step's results; events on the
    streams.  Two device input sets alternate: the copy stream loads step i+1's
    inputs while the compute stream verifies step i (the host link, not the
    kernel, bounds the step), and each step's results are read back before its
    input set is refilled."""
    import torch
    sampled = x.draft_probs is not None
    host = dict(z=x.logits, tok=x.draft_tokens, slots=x.slot_mapping)
    if sampled:
        host.update(T=x.temperature, ua=x.u_accept, us=x.u_sample, q=x.draft_probs)
    pinned = {}
    for k_, a in host.items():
        a = np.ascontiguousarray(a)
        pinned[k_] = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
    sets = [{k_: torch.empty_like(t, device=dev) for k_, t in pinned.items()} for _ in range(2)]
    outs = [dict(out=torch.empty((x.B, x.k + 1), dtype=torch.int32, device=dev),
                 na=torch.empty((x.B,), dtype=torch.int32, device=dev)) for _ in range(2)]
    out_h = torch.empty((x.B, x.k + 1), dtype=torch.int32).pin_memory()
    na_h = torch.empty((x.B,), dtype=torch.int32).pin_memory()
    slots_h = torch.empty_like(pinned["slots"]).pin_memory()
    h2d = sum(int(t.numel() * t.element_size()) for t in pinned.values())
    d2h = int(out_h.numel() * 4 + na_h.numel() * 4 + slots_h.numel() * 8)
    compute = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    loaded = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]
    for e in freed:
        e.record(compute)

    def load(i):
        s_ = i & 1
        copy.wait_event(freed[s_])          # the set's previous step has read it and its results are out
        with torch.cuda.stream(copy):
            for k_, t in pinned.items():
                sets[s_][k_].copy_(t, non_blocking=True)
        loaded[s_].record(copy)

    def verify(i):
        s_ = i & 1
        d, o = sets[s_], outs[s_]
        compute.wait_event(loaded[s_])
        z = d["z"].view(torch.bfloat16) if x.dtype == 0 else d["z"]
        sv.verify_chain(z, d["tok"], d.get("T"), d.get("ua"), d.get("us"), d.get("q"), out_tokens=o["out"],
                        out_num_accepted=o["na"], slot_mapping=d["slots"])
        out_h.copy_(o["out"], non_blocking=True)
        na_h.copy_(o["na"], non_blocking=True)
        slots_h.copy_(d["slots"], non_blocking=True)
        freed[s_].record(compute)

    def run(n):
        load(0)
        for i in range(n):
            if i + 1 < n:
                load(i + 1)
            verify(i)

    run(3)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    copy.wait_event(e0)
    run(steps)
    e1.record(compute)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    ms = reduce_max(dist, e0.elapsed_time(e1), dev)
    return ms, h2d, d2h, (out_h.numpy().copy(), na_h.numpy().copy())


# ------------------------------------------------------------ CPU leg ---
# Sampled workloads whose GPU results the CPU leg checks against the oracle:
# (kind, the workload's result line, inputs, GPU outputs).
_PARITY_JOBS = []


def cpu_parity_leg():
    """Part of the CPU-baseline leg: the oracle on each sampled secondary
    workload's batch, compared with the GPU's results of that batch.  Adds to
    each result line the fraction of positions (B x (k+1) rows, B x (N+1)
    tree nodes) the oracle flags and the fraction where the GPU differs."""
    from oracle import oracle as O
    threads = os.cpu_count() or 1
    for kind, res, x, got in _PARITY_JOBS:
        if kind == "chain":
            ref = O.verify_chain(x.logits, x.dtype, x.draft_tokens, x.temperature, x.u_sample, x.draft_probs,
                                 x.u_accept, nthreads=threads)
            ot, na = got
            a, ra = na.astype(np.int64), ref["num_accepted"].astype(np.int64)
            tok_differ = np.array([a[b] == ra[b] and ot[b, a[b]] != ref["out_tokens"][b, a[b]]
                                   for b in range(x.B)])
            differ = int((a != ra).sum() + tok_differ.sum())
            positions = x.B * (x.k + 1)
        else:
            ref = O.verify_tree_sampled(x.logits, x.dtype, x.node_tokens, x.parent, x.temperature, x.u_accept,
                                        x.u_sample, x.draft_probs)
            path, toks, ln = got
            differ = int(sum(1 for b in range(x.B) if not (ln[b] == ref["length"][b]
                                                            and (path[b] == ref["path"][b]).all()
                                                            and (toks[b] == ref["tokens"][b]).all())))
            positions = x.B * (x.N + 1)
        flagged = int(ref["flag_accept"].sum() + ref["flag_sample"].sum())
        res["parity_vs_oracle"] = {"positions": positions, "flagged_frac": flagged / positions,
                                   "differ_frac": differ / positions}
    _PARITY_JOBS.clear()


def oracle_leg(x, seconds, rows_hint=None):
    """Times the CPU oracle on whole-request samples of the workload on all host
    cores; returns (positions/s, threads, sample description, oracle result of
    the first sample)."""
    from oracle import oracle as O
    threads = os.cpu_count() or 1
    B = x.B
    first = None
    t0 = time.perf_counter()
    done = 0
    reps = 0
    while True:
        rows = np.arange(B) if rows_hint is None else rows_hint
        r = O.verify_chain(x.logits[rows], x.dtype, x.draft_tokens[rows], x.temperature[rows],
                           x.u_sample[rows], None if x.draft_probs is None else x.draft_probs[rows],
                           None if x.u_accept is None else x.u_accept[rows], nthreads=threads)
        if first is None:
            first = r
        done += len(rows)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    pos = done * x.k / dt
    return pos, threads, "%d passes over the %d-request batch (%d requests, %.1f s)" % (reps, B, done, dt), first


# ---------------------------------------------------------------- main ---
def workload_default():
    from speculative_decoding_verification_chain_gb300 import workloads as W
    return W.chain_greedy(seed=2, B=64, k=5, V=128256, p_match=0.8)


WORKLOAD_NAME = ("greedy chain: B=64 requests, k=5 drafts, V=128256, bf16 logits N(0,3^2), "
                 "draft = row argmax w.p. 0.8 else uniform; step = verify + slot_mapping fix-up")


def reference_main(args, world, rank):
    """CPU oracle arm: rank 0 only, a bounded sample of the batch per step."""
    if rank != 0:
        return 0
    from oracle import oracle as O
    x = workload_default()
    threads = os.cpu_count() or 1
    # calibrate: time one request, then size the per-step sample
    t0 = time.perf_counter()
    O.verify_chain(x.logits[:1], x.dtype, x.draft_tokens[:1], x.temperature[:1], x.u_sample[:1], nthreads=1)
    per_req = max(1e-5, time.perf_counter() - t0)
    budget = 120.0 / max(1, args.steps + args.warmup)
    nreq = int(max(1, min(x.B, budget * min(threads, x.B) / per_req)))
    rows = np.arange(nreq)
    sub = lambda a: a[rows]

    def step():
        O.verify_chain(sub(x.logits), x.dtype, sub(x.draft_tokens), sub(x.temperature), sub(x.u_sample),
                       nthreads=threads)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = nreq * x.k * args.steps / dt
    sample = "first %d of %d requests per step (whole requests, all rows)" % (nreq, x.B)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "global_batch": x.B, "k": x.k, "V": x.V,
                   "reference": "CPU fp64 oracle (plain C), the path has no other reference implementation"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        return reference_main(args, world, rank)
    import torch
    import speculative_decoding_verification_chain_gb300 as sv
    from speculative_decoding_verification_chain_gb300 import workloads as W
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, True)
    sv.load_library()
    if args.only:
        res = others(sv, W, dev, dist, measured_peak()[0], args)
        if rank == 0:
            print(json.dumps({"only": args.only, "also": res}))
        return 0

    x = workload_default()
    case = ChainCase(sv, x, dev, with_fixup=True)
    case.capture()
    peak, peak_kind = measured_peak()

    sampler = ClockSampler(local)
    if not args.quick:
        sampler.start()
    case.run(args.warmup)
    torch.cuda.synchronize(dev)
    ms = time_steps(case, args.steps, dev, dist)
    # the verify kernel alone, same rotation, for the roofline (>= ~1.5 s of replays)
    ws_counters0 = sv.workspace_counters(case.ws)
    kv_steps = args.steps if args.quick else max(args.steps, 2000)
    ms_k = time_steps(case, kv_steps, dev, dist, verify_only=True)
    t_target = 1.5
    if not args.quick and ms_k / 1e3 < t_target:
        extra = int(kv_steps * (t_target / max(ms_k / 1e3, 1e-6)))
        ws_counters0 = sv.workspace_counters(case.ws)
        ms_k2 = time_steps(case, extra, dev, dist, verify_only=True)
        kv_steps, ms_k = extra, ms_k2
    ws_counters1 = sv.workspace_counters(case.ws)
    clocks = sampler.stop() if not args.quick else {"sm_mhz": None, "sm_max_mhz": None,
                                                     "reasons": ["not sampled (--quick)"], "samples": 0}

    na = case.copies[0]["na"].cpu().numpy()
    st = int(case.status.item())
    kernel_us = ms_k * 1e3 / kv_steps
    b_alg, b_par, b_dense = chain_bytes(na, x.temperature, x.k, x.V, 2)
    streamed = (ws_counters1["bytes_loaded"] - ws_counters0["bytes_loaded"]) / kv_steps
    achieved = b_alg / (kernel_us * 1e-6) / 1e9
    positions = x.B * x.k
    value = positions * world * args.steps / (ms / 1e3)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "global_batch": x.B * world, "k": x.k, "V": x.V,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs rotate over %d device copies (%.0f MB > 4x L2); CUDA graph per step"
                         % (case.ncopy, case.ncopy * x.logits.nbytes / 1e6)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic("verify_kernel_greedy_chain_B64_k5_V128256.md"),
                     "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy burst)",
                     "bytes_per_launch": {"algorithmic": b_alg, "position_parallel": b_par, "dense": b_dense,
                                          "streamed_by_kernel": streamed},
                     "frac_position_parallel": b_par / (kernel_us * 1e-6) / 1e9 / peak,
                     "frac_dense": b_dense / (kernel_us * 1e-6) / 1e9 / peak,
                     "frac_alg_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                     "kernel": "verify_kernel<2>", "kernel_us": kernel_us, "kernel_launches_timed": kv_steps},
        "gpu_launches": args.steps * case.launches_per_step(),
        "clocks": clocks,
        "device_status": st,
    }

    if not args.no_e2e:
        e_ms, h2d, d2h, _ = e2e_leg(sv, x, dev, args.e2e_steps, dist)
        line["e2e"] = {"value": positions * world * args.e2e_steps / (e_ms / 1e3), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                       "ms_per_step": e_ms / args.e2e_steps}

    if not args.no_others:
        line["also"] = others(sv, W, dev, dist, peak, args)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pos, threads, sample, ref = oracle_leg(x, args.cpu_seconds)
        got_t = case.copies[0]["out"].cpu().numpy()
        line["cpu_baseline"] = {"value": pos, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
                                "parity_vs_gpu": {"requests": int(x.B),
                                                  "mismatched_requests": int((got_t != ref["out_tokens"]).any(1).sum())}}
        cpu_parity_leg()
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def others(sv, W, dev, dist, peak, args):
    """Secondary workloads (kernel-only device time): sampled chain, the k = 8,
    V = 152064 sampled sweep, greedy tree, the ragged greedy chain, n-gram
    lookup drafting, the sampled tree, next-step preparation and tree KV
    compaction (or only the one --only names)."""
    want = lambda name: args.only is None or args.only == name
    out = []
    if want("sampled_chain"):
        # the draft's closeness to the target at three levels (lambda = 0.3 first)
        for lam in (0.3, 0.1, 0.6):
            x = W.chain_sampled(seed=3, B=32, k=4, V=128256, temperature=0.7, lam=lam)
            out.append(_other_chain(sv, x, dev, dist, peak,
                                    "sampled chain B=32 k=4 V=128256 T=0.7 lambda=%g (Zipf)" % lam))
            if lam == 0.3:
                out[-1]["kernel"] = "chain_cluster_kernel<2>"
                out[-1]["profiled_traffic"] = profiled_traffic(
                    "chain_cluster_kernel_sampled_chain_B32_k4_V128256.md", "chain_cluster_kernel")
    if want("sweep"):
        for Bs in ([args.sweep_b] if args.sweep_b else [64, 1, 8, 256]):
            x = W.chain_sampled(seed=5, B=Bs, k=8, V=152064, temperature=1.0, lam=0.3)
            out.append(_other_chain(sv, x, dev, dist, peak,
                                    "sampled sweep B=%d k=8 V=152064 T=1 lambda=0.3 (Zipf)" % Bs))
    if want("greedy_tree"):
        out.append(_other_tree(sv, W, dev, dist, peak))
        out[-1]["kernel"] = "greedy_cluster_kernel<2>"
        out[-1]["profiled_traffic"] = profiled_traffic("greedy_cluster_kernel_greedy_tree_B16_N60_V128256.md",
                                                       "greedy_cluster_kernel")
    if want("ragged"):
        out.append(_other_ragged(sv, W, dev, dist, peak))
    if want("ngram"):
        out.append(_other_ngram(sv, W, dev, dist, peak))
    if want("sampled_tree"):
        out.append(_other_tree_sampled(sv, W, dev, dist, peak))
        out[-1]["kernel"] = "tree_sampled_kernel<2>"
        out[-1]["profiled_traffic"] = profiled_traffic("tree_sampled_kernel_B16_N60_V128256.md", "tree_sampled_kernel")
    if want("next_step"):
        out.extend(_other_next_step(sv, W, dev, dist, peak))
    return out


def _other_chain(sv, x, dev, dist, peak, name, target_s=0.5):
    import torch
    case = ChainCase(sv, x, dev, with_fixup=False)
    case.capture()
    case.run(20)
    ms = time_steps(case, 200, dev, dist, verify_only=True)
    n = max(200, int(200 * target_s / max(ms / 1e3, 1e-6)))
    c0 = sv.workspace_counters(case.ws)
    ms = time_steps(case, n, dev, dist, verify_only=True)
    c1 = sv.workspace_counters(case.ws)
    us = ms * 1e3 / n
    na = case.copies[0]["na"].cpu().numpy()
    s_z = 2 if x.dtype == 0 else 4
    b_alg, b_par, b_dense = chain_bytes(na, x.temperature, x.k, x.V, s_z)
    ach = b_alg / (us * 1e-6) / 1e9
    res = {"workload": name, "positions_per_s": x.B * x.k / (us * 1e-6), "kernel_us": us,
           "achieved_gbs_alg": ach, "frac_alg": ach / peak, "frac_position_parallel": b_par / (us * 1e-6) / 1e9 / peak,
           "frac_dense": b_dense / (us * 1e-6) / 1e9 / peak,
           "bytes_per_launch": {"algorithmic": b_alg, "position_parallel": b_par, "dense": b_dense,
                                "streamed_by_kernel": (c1["bytes_loaded"] - c0["bytes_loaded"]) / n},
           "mean_accepted": float(na.mean())}
    if x.draft_probs is not None:
        a = na.astype(np.int64)
        res["alpha_achieved"] = float(a.sum() / max(1, (a + (a < x.k)).sum()))
        _PARITY_JOBS.append(("chain", res, x, (case.copies[0]["out"].cpu().numpy(), na)))
    del case
    torch.cuda.empty_cache()
    return res


def _other_tree(sv, W, dev, dist, peak, target_s=0.5):
    import torch
    t = W.tree_greedy(seed=4, B=16, V=128256)
    per_copy = t.logits.nbytes
    ncopy = min(64, max(2, int(np.ceil(4 * l2_bytes(dev) / per_copy)) + 1))
    zs = [to_dev(t.logits, dev) for _ in range(ncopy)]
    tok = to_dev(t.node_tokens, dev)
    D1 = 6   # depth 5 plus the root
    outs = [(torch.empty((t.B, D1), dtype=torch.int32, device=dev), torch.empty((t.B, D1), dtype=torch.int32, device=dev),
             torch.empty((t.B,), dtype=torch.int32, device=dev)) for _ in range(ncopy)]
    ws = torch.zeros(sv.workspace_bytes(t.B, t.N + 1, t.V, 0), dtype=torch.uint8, device=dev)
    parent = t.parent

    def call(i):
        sv.verify_tree(zs[i], tok, parent, 5, out_path=outs[i][0], out_tokens=outs[i][1], out_len=outs[i][2],
                       workspace=ws)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for i in range(ncopy):
            call(i)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    graphs = []
    for i in range(ncopy):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(i)
        graphs.append(g)

    class _C:
        def run(self, steps, verify_only=False):
            for j in range(steps):
                graphs[j % ncopy].replay()
    case = _C()
    case.run(20)
    ms = time_steps(case, 200, dev, dist)
    n = max(200, int(200 * target_s / max(ms / 1e3, 1e-6)))
    c0 = sv.workspace_counters(ws)
    ms = time_steps(case, n, dev, dist)
    c1 = sv.workspace_counters(ws)
    us = ms * 1e3 / n
    g_rows = np.argmax(W.logits_as_f32(t.logits, t.dtype), axis=-1)
    b_alg = tree_greedy_bytes(t.parent, t.node_tokens, g_rows, outs[0][0].cpu().numpy(),
                              outs[0][2].cpu().numpy(), t.V, 2)
    b_dense = float(t.logits.nbytes)
    ach = b_alg / (us * 1e-6) / 1e9
    return {"workload": "greedy tree B=16 N=60 levels (4,8,16,16,16) V=128256 bf16",
            "positions_per_s": t.B * t.N / (us * 1e-6), "kernel_us": us, "achieved_gbs_alg": ach,
            "frac_alg": ach / peak, "frac_dense": b_dense / (us * 1e-6) / 1e9 / peak,
            "bytes_per_launch": {"algorithmic": b_alg, "dense": b_dense,
                                 "streamed_by_kernel": (c1["bytes_loaded"] - c0["bytes_loaded"]) / n}}


def _other_ragged(sv, W, dev, dist, peak, target_s=0.5):
    """Ragged greedy chain: B = 64 requests with k_b uniform in [1, 8] drafts,
    V = 128256 bf16, packed by cu_num_draft_tokens (the headline recipe per
    request)."""
    import torch
    x = W.chain_ragged(seed=7, B=64, max_k=8, V=128256, mode="greedy", min_k=1)
    per_copy = x.logits.nbytes
    ncopy = min(64, max(2, int(np.ceil(4 * l2_bytes(dev) / per_copy)) + 1))
    zs = [to_dev(x.logits, dev) for _ in range(ncopy)]
    tok, cu = to_dev(x.draft_tokens, dev), to_dev(x.cu, dev)
    mk = x.max_k
    outs = [(torch.empty((x.B, mk + 1), dtype=torch.int32, device=dev), torch.empty((x.B,), dtype=torch.int32, device=dev))
            for _ in range(ncopy)]
    ws = torch.zeros(sv.workspace_bytes(x.B, mk + 1, x.V, 0), dtype=torch.uint8, device=dev)

    def call(i):
        sv.verify_chain_ragged(zs[i], tok, cu, mk, out_tokens=outs[i][0], out_num_accepted=outs[i][1], workspace=ws)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for i in range(ncopy):
            call(i)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    graphs = []
    for i in range(ncopy):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(i)
        graphs.append(g)

    class _C:
        def run(self, steps, verify_only=False):
            for j in range(steps):
                graphs[j % ncopy].replay()
    case = _C()
    case.run(20)
    ms = time_steps(case, 200, dev, dist)
    n = max(200, int(200 * target_s / max(ms / 1e3, 1e-6)))
    c0 = sv.workspace_counters(ws)
    ms = time_steps(case, n, dev, dist)
    c1 = sv.workspace_counters(ws)
    us = ms * 1e3 / n
    a = outs[0][1].cpu().numpy().astype(np.int64)
    ks = np.diff(x.cu).astype(np.int64)
    b_alg = float(((np.minimum(a, ks) + 1) * x.V * 2).sum())
    b_dense = float(x.logits.nbytes)
    ach = b_alg / (us * 1e-6) / 1e9
    return {"workload": "ragged greedy chain B=64 k_b uniform in [1, 8] (sum %d) V=128256 bf16" % int(ks.sum()),
            "positions_per_s": float(ks.sum()) / (us * 1e-6), "kernel_us": us, "achieved_gbs_alg": ach,
            "frac_alg": ach / peak, "frac_dense": b_dense / (us * 1e-6) / 1e9 / peak,
            "bytes_per_launch": {"algorithmic": b_alg, "dense": b_dense,
                                 "streamed_by_kernel": (c1["bytes_loaded"] - c0["bytes_loaded"]) / n},
            "mean_accepted": float(a.mean())}


def _other_ngram(sv, W, dev, dist, peak, target_s=0.5):
    """n-gram lookup drafting: B = 64 copy-heavy texts, lengths uniform in
    [1, 8192], n in [2, 8], k = 8 (the draft length of the chain workloads).
    Input copies rotate so the token buffers together exceed L2 four times."""
    import torch
    t, ln = W.ngram_texts(seed=11, B=64, Lmax=8192, V=128256)
    n_min, n_max, k = 2, 8, 8
    ncopy = min(256, max(2, int(np.ceil(4 * l2_bytes(dev) / t.nbytes)) + 1))
    ts = [to_dev(t, dev) for _ in range(ncopy)]
    lt = to_dev(ln, dev)
    outs = [tuple(torch.empty(shape, dtype=torch.int32, device=dev) for shape in ((64, k), (64,), (64,), (64,)))
            for _ in range(ncopy)]

    def call(i):
        o = outs[i]
        sv.ngram_propose(ts[i], lt, n_min, n_max, k, out_draft=o[0], out_count=o[1], out_match_len=o[2],
                         out_match_end=o[3])
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for i in range(ncopy):
            call(i)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(ncopy):
            call(i)

    class _C:
        def run(self, steps, verify_only=False):
            for _ in range(steps):
                g.replay()
    case = _C()
    case.run(3)
    ms = time_steps(case, 10, dev, dist)
    n = max(10, int(10 * target_s / max(ms / 1e3, 1e-6)))
    ms = time_steps(case, n, dev, dist)
    us = ms * 1e3 / (n * ncopy)
    b_alg = float(ln.astype(np.int64).sum() * 4 + 64 * 4 + 64 * (k + 3) * 4)
    ach = b_alg / (us * 1e-6) / 1e9
    cnt = outs[0][1].cpu().numpy()
    return {"workload": "n-gram lookup B=64 copy-heavy texts L uniform in [1, 8192] (sum %d) n in [2, 8] k=8"
            % int(ln.sum()), "sequences_per_s": 64 / (us * 1e-6), "kernel_us": us, "achieved_gbs_alg": ach,
            "frac_alg": ach / peak, "bytes_per_launch": {"algorithmic": b_alg},
            "mean_draft_len": float(cnt.mean())}


def tree_sampled_bytes(parent, path, length, V, zbytes):
    """Algorithmic bytes of one sampled-tree walk, from its path: the logits
    row of every node on the path; the q row of a node where a child was
    rejected (the next node is not its first child, or the walk stopped at a
    node with children); 4 bytes per q(x) gather (one per child tested)."""
    par = np.asarray(parent)
    kids = [np.flatnonzero(par == c) for c in range(par.shape[0])]
    total = 0.0
    for b in range(path.shape[0]):
        L = int(length[b])
        nodes = [int(v) for v in path[b, :L]]
        total += L * V * zbytes
        for i, c in enumerate(nodes):
            ch = kids[c]
            if i + 1 < L:
                tested = int(np.flatnonzero(ch == nodes[i + 1])[0]) + 1
                rejected = tested > 1
            else:
                tested = ch.size
                rejected = ch.size > 0
            total += 4.0 * tested + (V * 4.0 if rejected else 0.0)
    return total


def _other_tree_sampled(sv, W, dev, dist, peak, target_s=0.5):
    """Sampled tree: B = 16 requests, the 60-node tree of the greedy tree
    workload, V = 128256 bf16 logits and fp32 q rows, T = 0.7, lambda = 0.3.
    Input copies rotate so the rows the walks read never come from L2."""
    import torch
    x = W.tree_sampled(seed=13, B=16, V=128256)
    per_copy = x.logits.nbytes + x.draft_probs.nbytes
    z0 = to_dev(x.logits, dev)
    q0 = to_dev(x.draft_probs, dev)
    small = dict(tok=to_dev(x.node_tokens, dev), T=to_dev(x.temperature, dev), ua=to_dev(x.u_accept, dev),
                 us=to_dev(x.u_sample, dev))
    ncopy = 8
    zs = [z0] + [z0.clone() for _ in range(ncopy - 1)]
    qs = [q0] + [q0.clone() for _ in range(ncopy - 1)]
    D1 = int(tree_depth(x.parent)) + 1
    outs = [tuple(torch.empty(sh, dtype=torch.int32, device=dev) for sh in ((x.B, D1), (x.B, D1), (x.B,)))
            for _ in range(ncopy)]

    def call(i):
        o = outs[i]
        sv.verify_tree_sampled(zs[i], qs[i], small["tok"], x.parent, small["T"], small["ua"], small["us"],
                               out_path=o[0], out_tokens=o[1], out_len=o[2])
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for i in range(ncopy):
            call(i)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(ncopy):
            call(i)

    class _C:
        def run(self, steps, verify_only=False):
            for _ in range(steps):
                g.replay()
    case = _C()
    case.run(3)
    ms = time_steps(case, 10, dev, dist)
    n = max(10, int(10 * target_s / max(ms / 1e3, 1e-6)))
    ms = time_steps(case, n, dev, dist)
    us = ms * 1e3 / (n * ncopy)
    path, length = outs[0][0].cpu().numpy(), outs[0][2].cpu().numpy()
    b_alg = tree_sampled_bytes(x.parent, path, length, x.V, 2)
    ach = b_alg / (us * 1e-6) / 1e9
    res = {"workload": "sampled tree B=16 N=60 levels (4,8,16,16,16) V=128256 bf16 T=0.7 lambda=0.3 (Zipf)",
           "positions_per_s": float(x.B * x.N) / (us * 1e-6), "tokens_per_s": float(length.sum()) / (us * 1e-6),
           "kernel_us": us, "achieved_gbs_alg": ach, "frac_alg": ach / peak,
           "bytes_per_launch": {"algorithmic": b_alg, "dense_inputs": float(per_copy)},
           "mean_tokens_per_request": float(length.mean())}
    _PARITY_JOBS.append(("tree", res, x, (path, outs[0][1].cpu().numpy(), length)))
    return res


def _other_next_step(sv, W, dev, dist, peak, target_s=0.3):
    """Post-verify work.  (1) Tree KV compaction: B = 16 requests, the 60-node
    tree, one token's KV = 32 layers x (K, V) x 8 heads x 128 x bf16 = 128 KiB
    a row; paths from the sampled-tree walks of the same tree; 8 slot maps over
    a 4096-slot (512 MiB) cache rotate so consecutive launches touch different
    rows.  (2) Next-step preparation for the greedy chain batch: B = 64, k = 5,
    6 next slots from 64-block tables, 4096-wide bf16 hidden rows."""
    import torch
    res = []
    # (1) compaction
    x = W.tree_sampled(seed=17, B=16, V=4096)
    p, t, n = sv.verify_tree_sampled(to_dev(x.logits, dev).view(torch.bfloat16), to_dev(x.draft_probs, dev),
                                     to_dev(x.node_tokens, dev), x.parent, to_dev(x.temperature, dev),
                                     to_dev(x.u_accept, dev), to_dev(x.u_sample, dev))
    row = 32 * 2 * 8 * 128 * 2
    num_slots = 4096
    kv = torch.zeros((num_slots, row // 2), dtype=torch.bfloat16, device=dev)
    g = np.random.default_rng(19)
    nmap = 8
    maps = [torch.from_numpy(g.permutation(num_slots)[:x.B * (x.N + 1)].reshape(x.B, x.N + 1).astype(np.int64)).to(dev)
            for _ in range(nmap)]
    torch.cuda.synchronize(dev)
    lens = n.cpu().numpy()
    moved = sum(int(np.sum(p.cpu().numpy()[b, 1:lens[b]] != np.arange(1, lens[b]))) for b in range(x.B))

    gk = _graph_of(dev, lambda: [sv.compact_tree_kv(kv, maps[j], p, n) for j in range(nmap)])
    us = _time_graph(gk, nmap, dev, dist, target_s)
    b_alg = 2.0 * moved * row
    res.append({"workload": "tree KV compaction B=16 N=60 (4,8,16,16,16), 128 KiB KV rows, %d rows moved" % moved,
                "kernel_us": us, "achieved_gbs_alg": b_alg / (us * 1e-6) / 1e9,
                "frac_alg": b_alg / (us * 1e-6) / 1e9 / peak, "bytes_per_launch": {"algorithmic": b_alg},
                "note": "CUDA-graph replays of 8 launches, rotating slot maps"})
    # (2) next-step preparation
    B, k1, H = 64, 6, 4096
    ot = torch.from_numpy(g.integers(0, 128256, size=(B, k1)).astype(np.int32)).to(dev)
    na = torch.from_numpy(g.integers(0, k1, size=B).astype(np.int32)).to(dev)
    pos = torch.from_numpy(g.integers(0, 900, size=B).astype(np.int32)).to(dev)
    bt = torch.from_numpy(g.integers(0, 20000, size=(B, 64)).astype(np.int32)).to(dev)
    hid = torch.zeros((B * k1, H), dtype=torch.bfloat16, device=dev)

    gp = _graph_of(dev, lambda: [sv.prepare_next_step(ot, na, pos, bt, 16, k1, rows_per_req=k1, hidden=hid)
                                 for _ in range(16)])
    us = _time_graph(gp, 16, dev, dist, target_s)
    b_alg = float(B * (2 * H * 2 + 4 * 4 + k1 * 8 + 4))
    res.append({"workload": "next-step preparation B=64 k=5, 6 next slots, 4096-wide bf16 hidden rows",
                "kernel_us": us, "achieved_gbs_alg": b_alg / (us * 1e-6) / 1e9,
                "bytes_per_launch": {"algorithmic": b_alg},
                "note": "CUDA-graph replays of 16 launches; 1.1 MB a launch, so launch latency dominates"})
    return res


def _graph_of(dev, fn):
    """fn() enqueues work; warm it up on a side stream, then capture it."""
    import torch
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _time_graph(g, launches_per_replay, dev, dist, target_s):
    """Mean device time of one launch over graph replays (CUDA events)."""
    class _C:
        def run(self, steps, verify_only=False):
            for _ in range(steps):
                g.replay()
    case = _C()
    case.run(3)
    ms = time_steps(case, 10, dev, dist)
    n = max(10, int(10 * target_s / max(ms / 1e3, 1e-6)))
    ms = time_steps(case, n, dev, dist)
    return ms * 1e3 / (n * launches_per_replay)


def tree_depth(parent):
    par = np.asarray(parent)
    d = np.zeros(par.shape[0], np.int64)
    for n in range(1, par.shape[0]):
        d[n] = d[par[n]] + 1
    return d.max()


if __name__ == "__main__":
    sys.exit(main())
