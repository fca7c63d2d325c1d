"""Benchmark of one tree-attention speculative verification step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload c4]
                    [--sub c3,c5,c2,c1]

A step is one pass of the whole hot path over one batch of synthetic input:
tree_build_ancestry -> tree_attn_fwd -> tree_verify_greedy.  The metric is tree
tokens verified per second (B * N / step time).  Prints ONE JSON line.

The headline workload is c4, the 70B-shaped layer (batch 64, 64-node trees,
8192-token paged prefixes, vocab 128256), the largest configuration; the
line also carries sub-records for c3 (batched serving), c5 (131072-token
prefixes), c2 and c1, each with its step time, per-call times and rooflines.

Timing (impl=ours): the K timed steps are captured into CUDA graphs (chunks of
S steps) and replayed back to back; the whole timed region is bracketed by a
barrier and a synchronize, with CUDA events on the launching stream around it.
The library's kernels use programmatic dependent launch, so a graph with event
nodes between the kernels would serialise them; the per-call durations are
therefore taken in a second region right after, from a graph of the same
steps with a timing event node around every library call.  Where one input
set is smaller than twice the 129 MB L2, steps rotate over several
independent sets whose union is larger, so every step reads its inputs from
HBM.  ``e2e`` repeats the headline step through the same public calls from
pinned host buffers, with the host->device copies of all inputs and the
device->host read of the accepted path inside the timed region.
``cpu_baseline`` (and impl=reference) time the CPU oracle on bounded samples
of the same workloads.

Under torchrun (--gpus N > 1) every rank runs an independent replica of the
workload on its own GPU (the path has no exchange step); rank 0 prints the
job-wide value = all ranks' tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------- accounting

def algorithmic(case) -> dict:
    """Bytes each kernel must move and flops it must do for one step of ``case``."""
    B, N, Hq, Hkv, D, W = case.B, case.N, case.Hq, case.Hkv, case.D, case.W
    P = case.prefix_len.astype(np.int64)
    anc_bytes = B * N * 4 + B * 4 + B * N * W * 8 + B * N * 8 + B * 4
    nblk = int(sum(-(-int(p) // case.bs) for p in P))
    attn_bytes = (int(P.sum()) * Hkv * D * 2 * 2 + B * N * Hq * D * 2 + B * N * Hkv * D * 2 * 2
                  + B * N * W * 8 + nblk * 4 + B * 4 + B * N * Hq * D * 2 + B * N * Hq * 4)
    # |A(i)| = depth + 1, counted here without the oracle: walk parent pointers
    vis = 0
    for b in range(B):
        par = case.parent[b]
        dep = np.zeros(N, np.int64)
        for i in range(1, N):
            dep[i] = dep[par[i]] + 1
        vis += int(N * P[b] + (dep + 1).sum())
    attn_flops = 4 * D * (Hq // Hkv) * Hkv * vis
    ver_bytes = (B * N * case.vocab * 4 + 2 * B * N * 4 + B * N * 4 + B * 12) if case.vocab else 0
    return {"tree_build_ancestry": {"bytes": anc_bytes, "flops": 0},
            "tree_attn_fwd": {"bytes": attn_bytes, "flops": attn_flops},
            "tree_verify_greedy": {"bytes": ver_bytes, "flops": 0}}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel's source changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}.{workload}.traffic.txt")
    if not os.path.exists(path):
        return None
    rec = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
    try:
        if code_digest(rec["sources"].split()) != rec["sources_sha256_16"]:
            return None
        return int(float(rec["dram_bytes_per_launch"]))
    except Exception:
        return None


def code_digest(sources) -> str:
    """First 16 hex digits of the sha256 of the sources' code: '//' comments,
    trailing blanks and empty lines removed, so that editing a comment does not
    disown a capture of an unchanged kernel."""
    h = hashlib.sha256()
    for s in sources:
        for line in open(os.path.join(ROOT, s), encoding="utf-8"):
            code = re.sub(r"//.*$", "", line).rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str, period_ms: int = 50):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.period = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        def parse(s):
            parts = [p.strip() for p in s.split(",")]
            try:
                return float(parts[0]), float(parts[1]), parts
            except Exception:
                return None

        win = [(t, parse(s)) for t, s in self.samples if t0 <= t <= t1]
        win = [(t, p) for t, p in win if p]
        note = "samples inside the timed region"
        if not win:   # a short timed region: take the samples closest to it
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:3]
            win = [(t, parse(s)) for t, s in near]
            win = [(t, p) for t, p in win if p]
            note = "no sample inside the timed region; nearest samples"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [p[0] for _, p in win]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in win:
            for name, val in zip(names, p[2][4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(p[1] for _, p in win),
                "reasons": sorted(reasons), "samples": len(win), "note": note}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- oracle timing

def oracle_part(case, seqs, units):
    """Run the oracle on part of one step and return the seconds it took:
    ancestry of the trees of ``seqs``, attention of the (sequence, kv-head)
    ``units``, and (with logits) the argmax of every row of ``seqs`` plus
    their acceptance walks."""
    import oracle
    import workloads as W
    seqs = list(seqs)
    forest = bool((case.parent[:, 1:] < 0).any())
    t0 = time.perf_counter()
    (oracle.forest.build_ancestry_forest if forest else oracle.tree.build_ancestry)(case.parent[seqs],
                                                                                   case.prefix_len[seqs])
    if units:
        oracle.attention.tree_attention_case(case, units=list(units))
    if case.vocab:
        am = oracle.verify.greedy_argmax(case.logits[seqs])
        walk = oracle.forest.accept_walk_forest if forest else oracle.verify.accept_walk
        for i, b in enumerate(seqs):
            walk(case.parent[b], case.draft[b], am[i], W.LEVELS.get(case.name, case.N - 1))
    return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def _one_thread():
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(1)
    except Exception:   # pragma: no cover
        import contextlib
        return contextlib.nullcontext()


def oracle_throughput(case, budget_s: float, mode: str):
    """Tree tokens verified per second by the CPU oracle on ``case``.

    mode "full": the whole step (every tree, every unit, every row), repeated
    until ``budget_s`` is spent.  mode "sequences": whole sequences, one after
    another from sequence 0, until ``budget_s`` is spent; nothing is
    extrapolated (tokens = the sequences' nodes).  mode "units": ancestry and
    verification of the whole batch plus attention of seeded (sequence,
    kv-head) units until ``budget_s`` is spent, the attention time scaled by
    the unit count (stated in the sample).  Returns (tokens/s, description)."""
    B, N, Hkv = case.B, case.N, case.Hkv
    allu = [(b, g) for b in range(B) for g in range(Hkv)]
    if mode == "full":
        ts = []
        while not ts or sum(ts) < budget_s:
            ts.append(oracle_part(case, range(B), allu))
        t = float(np.median(ts))
        return B * N / t, f"the whole step (all {B} trees, {B * Hkv} units, {B * N} rows), median of {len(ts)}"
    if mode == "sequences":
        spent, seqs = 0.0, 0
        while seqs < B and (seqs == 0 or spent < budget_s):
            spent += oracle_part(case, [seqs], [(seqs, g) for g in range(Hkv)])
            seqs += 1
        return seqs * N / spent, (f"sequences 0..{seqs - 1} of {B}, each whole (ancestry, attention of all "
                                  f"{Hkv} kv heads, argmax of its {N} rows, walk); {spent:.1f} s, no extrapolation")
    # units
    t_rest = oracle_part(case, range(B), [])
    g = np.random.default_rng(12345)
    order = [allu[i] for i in g.permutation(len(allu))]
    spent, k = 0.0, 0
    while k < len(order) and (k == 0 or spent < budget_s):
        spent += oracle_part(case, [order[k][0]], [order[k]])
        k += 1
    # each unit's call also re-ran its sequence's ancestry/argmax/walk: remove that share
    t_unit = max(spent / k - t_rest / B, 1e-9)
    t = t_rest + t_unit * len(allu)
    return B * N / t, (f"ancestry, argmax and walks of all {B} sequences ({t_rest:.2f} s) + attention of {k} "
                       f"seeded of {len(allu)} (sequence, kv-head) units ({t_unit:.2f} s each, net of their "
                       f"sequence's verify), extrapolated x{len(allu)}")


CPU_MODES = {"c1": "full", "c2": "full", "c3": "full", "c4": "sequences", "c5": "units"}


# ----------------------------------------------------------------------------- GPU bench

def measure_gpu(name, args, dev, world, K, overrides, with_e2e=False, sampler=None, warmup=5):
    """Time K steps of workload ``name`` (graph-captured, barrier + synchronize
    on both sides, CUDA events, max over ranks) and each library call's share;
    optionally the e2e step from pinned host buffers.  Returns a record."""
    import torch
    import workloads as W
    from tree_attention_speculative_gb300.step import PackedInputs, TreeVerifyStep
    from tests.gpu_util import to_dev

    base = W.make(name, **overrides)
    set_bytes = sum(x.nbytes for x in (base.q, base.k_cache, base.v_cache, base.k_tree, base.v_tree)) + \
        (base.logits.nbytes if base.logits is not None else 0)
    nsets = max(1, min(16, math.ceil(2 * L2_BYTES / set_bytes))) if set_bytes < 2 * L2_BYTES else 1
    cases = [base] + [W.make(name, seed=20270000 + 97 * k, **overrides) for k in range(1, nsets)]
    dsets = [to_dev(c, dev) for c in cases]
    forest = bool(overrides.get("forest_roots"))
    steps = [TreeVerifyStep(c.B, c.N, c.Hq, c.Hkv, c.D, c.prefix_len, vocab=c.vocab,
                            max_depth=W.LEVELS.get(name, c.N - 1), device=dev, forest=forest) for c in cases]

    def enqueue(k, evs=None):
        enqueue_on(dsets[k % nsets], steps[k % nsets], evs)

    def enqueue_on(t, st, evs=None):
        if evs: evs[0].record()
        st.ancestry(t["parent"], t["prefix_len"])
        if evs: evs[1].record()
        st.attention(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["prefix_len"], t["k_tree"],
                     t["v_tree"])
        if evs: evs[2].record()
        if base.vocab:
            st.verify(t["draft"], t["logits"], t["parent"])
        if evs: evs[3].record()

    for k in range(nsets):    # allocate workspaces eagerly
        enqueue(k)
    torch.cuda.synchronize()
    for k in range(warmup):
        enqueue(k)
    torch.cuda.synchronize()

    S = min(K, max(nsets, 8 * nsets))
    S = S - S % nsets if S >= nsets else S
    stream = torch.cuda.Stream(device=dev)

    def capture(nsteps, timed_calls):
        g = torch.cuda.CUDAGraph()
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)] for _ in range(nsteps)]
        with torch.cuda.graph(g, stream=stream):
            for k in range(nsteps):
                enqueue(k, evs[k] if timed_calls else None)
        return g, evs

    full, last = divmod(K, S)
    g_main = capture(S, False)[0] if full else None
    g_rem = capture(last, False)[0] if last else None
    if g_main: g_main.replay()    # one untimed replay of each graph uploads it
    if g_rem: g_rem.replay()
    torch.cuda.synchronize()

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(full):
        g_main.replay()
    if g_rem:
        g_rem.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    ms_step = max_over_ranks(e0.elapsed_time(e1), world, dev) / K

    # per-call durations: the same steps again, with an event node around every call
    S_ev = min(K, S)
    g_ev, evs = capture(S_ev, True)
    g_ev.replay()
    torch.cuda.synchronize()
    g_ev.replay()
    torch.cuda.synchronize()
    per = {"tree_build_ancestry": [], "tree_attn_fwd": [], "tree_verify_greedy": []}
    for e in evs:
        per["tree_build_ancestry"].append(e[0].elapsed_time(e[1]))
        per["tree_attn_fwd"].append(e[1].elapsed_time(e[2]))
        if base.vocab:
            per["tree_verify_greedy"].append(e[2].elapsed_time(e[3]))
    kern_ms = {k: float(np.mean(v)) for k, v in per.items() if v}
    ws_attn = steps[0].ws_attn.numel() if steps[0].ws_attn is not None else 0
    kernels_per_step = 2 + (1 if ws_attn > 256 else 0) + (1 if base.vocab else 0)
    for st in steps:
        assert (st.status.cpu().numpy() == 0).all(), f"{name}: a timed step reported an error status"
    del g_main, g_rem, g_ev

    rec = {"name": name, "case": base, "K": K, "ms_step": ms_step, "kern_ms": kern_ms, "w0": w0, "w1": w1,
           "S": S, "S_ev": S_ev, "nsets": nsets, "set_bytes": set_bytes, "kernels_per_step": kernels_per_step}

    if with_e2e:
        # e2e through the public calls.  Each input set is packed into one
        # pinned host buffer (PackedInputs), so a step's whole upload is one
        # copy; uploads run on a copy stream, step k+1's overlapping step k's
        # kernels, and an upload into a set waits until the kernels that last
        # read it are done.  Every step's upload and its result read-back are
        # inside the timed region.
        def host_arrays(c):
            h = {}
            for nm, arr in (("parent", c.parent), ("prefix_len", c.prefix_len), ("block_table", c.block_table)):
                h[nm] = torch.from_numpy(np.ascontiguousarray(arr, np.int32))
            for nm in ("q", "k_cache", "v_cache", "k_tree", "v_tree"):
                h[nm] = torch.from_numpy(np.ascontiguousarray(getattr(c, nm)).view(np.int16)).view(torch.bfloat16)
            if c.vocab:
                h["draft"] = torch.from_numpy(np.ascontiguousarray(c.draft, np.int32))
                h["logits"] = torch.from_numpy(np.ascontiguousarray(c.logits, np.float32))
            return h

        packs = [PackedInputs(host_arrays(c), dev) for c in cases]
        pviews = [{nm: pk.device(nm) for nm in pk.layout} for pk in packs]
        outs = {"accepted": torch.empty((base.B, W.LEVELS.get(name, base.N - 1) + 1), dtype=torch.int32).pin_memory(),
                "accept_len": torch.empty(base.B, dtype=torch.int32).pin_memory(),
                "bonus": torch.empty(base.B, dtype=torch.int32).pin_memory(),
                "status": torch.empty(base.B, dtype=torch.int32).pin_memory()}
        h2d = packs[0].nbytes
        d2h = sum(v.numel() * v.element_size() for v in outs.values())
        K_e2e = min(K, max(3 * nsets, int(2.0e-3 * K) + 3 * nsets)) if K > 200 else K
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(nsets)]
        consumed = [torch.cuda.Event() for _ in range(nsets)]

        def e2e_step(k):
            i = k % nsets
            main = torch.cuda.current_stream(dev)
            copy_stream.wait_event(consumed[i])
            packs[i].upload(copy_stream)
            copied[i].record(copy_stream)
            main.wait_event(copied[i])
            enqueue_on(pviews[i], steps[i])
            consumed[i].record(main)
            st = steps[i]
            if base.vocab:
                outs["accepted"].copy_(st.accepted, non_blocking=True)
                outs["accept_len"].copy_(st.accept_len, non_blocking=True)
                outs["bonus"].copy_(st.bonus, non_blocking=True)
            outs["status"].copy_(st.status, non_blocking=True)

        for k in range(min(3, K_e2e)):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        x0 = torch.cuda.Event(enable_timing=True)
        x1 = torch.cuda.Event(enable_timing=True)
        x0.record()
        copy_stream.wait_stream(torch.cuda.current_stream(dev))
        for k in range(K_e2e):
            e2e_step(k)
        torch.cuda.current_stream(dev).wait_stream(copy_stream)
        x1.record()
        torch.cuda.synchronize()
        barrier(world)
        ms_e2e = max_over_ranks(x0.elapsed_time(x1), world, dev) / K_e2e
        rec["e2e"] = {"value": world * base.B * base.N / (ms_e2e * 1e-3), "unit": "tree tokens/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K_e2e, "ms_per_step": ms_e2e,
                      "staging": "each step's inputs in one pinned buffer, uploaded by one copy on a copy stream "
                                 "that overlaps the previous step's kernels; results read back every step"}
        del packs, pviews
    del dsets, steps, cases
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def roofline_of(rec, pk, world=1):
    """Per-call throughput against the measured peaks; the attention call gets
    both its tensor and its HBM fraction.  Tensor fractions use the burst
    bf16 peak: these calls run at the full SM clock, and the sustained figure
    was taken under the power cap at a lower clock."""
    alg = algorithmic(rec["case"])
    kern = {}
    for k, ms in rec["kern_ms"].items():
        kb = alg[k]
        gbs = kb["bytes"] / (ms * 1e-3) / 1e9
        kern[k] = {"ms": ms, "share": ms / sum(rec["kern_ms"].values()), "GB/s": gbs, "hbm_frac": gbs / pk["hbm_gbs"]}
        if kb["flops"]:
            tf = kb["flops"] / (ms * 1e-3) / 1e12
            kern[k]["TFLOP/s"] = tf
            kern[k]["tensor_frac"] = tf / pk["bf16_tflops"]
    dom = max(rec["kern_ms"], key=rec["kern_ms"].get)
    a = alg[dom]
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if a["flops"] and a["flops"] / max(a["bytes"], 1) > ridge:
        roof = {"bound": "tensor", "achieved": kern[dom]["TFLOP/s"], "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": kern[dom]["tensor_frac"], "hbm_achieved_GBs": kern[dom]["GB/s"],
                "hbm_frac": kern[dom]["hbm_frac"]}
    else:
        roof = {"bound": "hbm", "achieved": kern[dom]["GB/s"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": kern[dom]["hbm_frac"]}
        if "TFLOP/s" in kern[dom]:
            roof["tensor_achieved_TFs"] = kern[dom]["TFLOP/s"]
            roof["tensor_frac"] = kern[dom]["tensor_frac"]
    roof["traffic"] = recorded_traffic(dom, rec["name"])
    roof["kernel"] = dom
    roof["algorithmic_bytes"] = a["bytes"]
    roof["algorithmic_flops"] = a["flops"]
    roof["peak_source"] = f"{pk['source']} ({'hbm copy' if roof['unit'] == 'GB/s' else 'bf16 burst'})"
    return roof, kern


def workload_record(rec, pk, world, cpu=None):
    """The sub-record of one workload inside the bench line."""
    c = rec["case"]
    roof, kern = roofline_of(rec, pk, world)
    out = {"workload": f"{rec['name']}: " + WORKLOAD_DESC[rec["name"]],
           "value": world * c.B * c.N / (rec["ms_step"] * 1e-3), "unit": "tree tokens/s",
           "ms_per_step": rec["ms_step"], "steps": rec["K"], "roofline": roof, "kernels": kern,
           "l2": l2_note(rec)}
    if cpu is not None:
        out["cpu_baseline"] = cpu
    return out


def l2_note(rec):
    tot = rec["nsets"] * rec["set_bytes"]
    if tot > L2_BYTES:
        return (f"{rec['nsets']} rotating input set(s) of {rec['set_bytes'] / 2**20:.1f} MiB "
                f"({tot / 2**20:.0f} MiB > 129 MiB L2)")
    return f"{rec['nsets']} input sets of {rec['set_bytes'] / 2**20:.2f} MiB: L2-resident (launch-bound case)"


def cpu_record(case, budget_s, mode, one_thread_budget=None):
    v, desc = oracle_throughput(case, budget_s, mode)
    out = {"value": v, "unit": "tree tokens/s", "cores": blas_threads(), "kind": "oracle",
           "sample": f"{desc}; numpy fp64 oracle, BLAS threads as reported"}
    if one_thread_budget is not None:
        with _one_thread():
            v1, d1 = oracle_throughput(case, one_thread_budget, mode)
        out["one_thread"] = {"value": v1, "cores": 1, "sample": d1}
    return out


SUB_STEPS = {"c1": 2000, "c2": 2000, "c3": 1000, "c4": 200, "c5": 100}


def run_ours(args, world, rank, local):
    import torch
    from tree_attention_speculative_gb300 import _build
    _build.build()

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pk = peaks()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)

    head = measure_gpu(args.workload, args, dev, world, args.steps, workload_overrides(args), with_e2e=True,
                       warmup=args.warmup)
    time.sleep(0.2)
    subs = {}
    for name in args.sub:
        if name == args.workload:
            continue
        subs[name] = measure_gpu(name, args, dev, world, max(args.steps, SUB_STEPS[name]), {}, warmup=args.warmup)
    sampler.stop()

    base = head["case"]
    roof, kern = roofline_of(head, pk, world)
    cpu = None
    sub_cpu = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_record(base, args.cpu_budget, CPU_MODES[args.workload],
                         one_thread_budget=args.cpu_budget / 4)
        for name, rec in subs.items():
            mode = CPU_MODES[name]
            sub_cpu[name] = cpu_record(rec["case"], 2.0 if mode == "full" else 4.0, mode,
                                       one_thread_budget=(0.5 if mode == "full" else None))
    line = {
        "metric": "tree-verify step: tree tokens verified/s",
        "value": world * base.B * base.N / (head["ms_step"] * 1e-3), "unit": "tree tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: " + WORKLOAD_DESC[args.workload] +
                               (f"; each tree replaced by a forest of {args.forest} trees" if args.forest else ""),
                   "batch": base.B, "tree_nodes": base.N, "q_heads": base.Hq, "kv_heads": base.Hkv,
                   "head_dim": base.D, "prefix": [int(x) for x in np.unique(base.prefix_len)][:4],
                   "kv_block": base.bs, "vocab": base.vocab, "parallelism": f"replicas x{world}",
                   "l2": l2_note(head),
                   "timing": f"CUDA graphs of {head['S']} steps replayed back to back, CUDA events around the K "
                             f"steps; per-call times from {head['S_ev']} more steps with an event node around "
                             f"each call"},
        "roofline": roof,
        "kernels": kern,
        "e2e": head["e2e"],
        "gpu_launches": args.steps * head["kernels_per_step"],
        "clocks": sampler.summary(head["w0"], head["w1"]),
        "cpu_baseline": cpu,
        "workloads": {name: workload_record(rec, pk, world, sub_cpu.get(name)) for name, rec in subs.items()},
    }
    for name, rec in subs.items():
        line["workloads"][name]["clocks"] = sampler.summary(rec["w0"], rec["w1"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


WORKLOAD_DESC = {
    "c1": "5-node demo tree, B1, prefix 16, 2 heads, D64, vocab 1000",
    "c2": "Llama-3-8B-shaped layer, B1, 64-node depth-6 tree, 32q/8kv heads, D128, contiguous 4096 prefix, "
          "verify over vocab 128256",
    "c3": "batched serving, B16, prefixes U[1024,16384], 26-node [4,3,2,1,1] tree, 32q/8kv, D128, paged bs16",
    "c4": "70B-shaped layer, B64, 64-node depth-8 trees, 64q/8kv, D128, paged bs16 prefix 8192, vocab 128256",
    "c5": "long context, B4, prefix 131072, 192-node depth-10 tree, 32q/8kv, D128, paged bs64, vocab 128256",
}


def run_commit(args, world, rank, local):
    """--part commit: time tree_commit_accepted (appending every sequence's accepted
    path to its paged cache) on the workload, after one real verification step."""
    import torch
    import workloads as W
    import oracle
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts
    from tree_attention_speculative_gb300.step import TreeVerifyStep
    from tests.gpu_util import to_dev

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kw = workload_overrides(args)
    if args.workload not in W.VOCAB:
        raise SystemExit("--part commit needs a workload with logits (c1, c2, c4, c5)")
    depth = W.LEVELS[args.workload]
    case = W.make(args.workload, spare_tokens=depth + 1, **kw)
    t = to_dev(case, dev)
    st = TreeVerifyStep(case.B, case.N, case.Hq, case.Hkv, case.D, case.prefix_len, vocab=case.vocab,
                        max_depth=depth, device=dev)
    st.run(t["parent"], t["prefix_len"], t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["k_tree"],
           t["v_tree"], t["draft"], t["logits"])
    torch.cuda.synchronize()
    new_len = torch.empty_like(t["prefix_len"])

    def commit():
        ts.tree_commit_accepted(t["k_tree"], t["v_tree"], st.accepted, st.accept_len, t["prefix_len"],
                                t["k_cache"], t["v_cache"], t["block_table"], new_len, st.status)

    for _ in range(args.warmup):
        commit()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(args.steps):
            commit()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    L = st.accept_len.cpu().numpy()
    assert (st.status.cpu().numpy() == 0).all()
    tokens = int((L + 1).sum())
    nbytes = tokens * case.Hkv * case.D * 2 * 2 * 2 + case.B * 4 * 4   # read tree + write cache, K and V
    pk = peaks()
    acc = st.accepted.cpu().numpy()
    c0 = time.perf_counter()
    reps = 0
    while time.perf_counter() - c0 < 2.0 or reps < 1:
        oracle.commit.commit_accepted(case.k_tree, case.v_tree, acc, L, np.zeros(case.B, np.int32), case.prefix_len,
                                      case.k_cache, case.v_cache, case.block_table)
        reps += 1
    t_cpu = (time.perf_counter() - c0) / reps
    line = {
        "metric": "commit of accepted paths: tokens appended/s", "value": tokens / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: " + WORKLOAD_DESC[args.workload], "part": "commit",
                   "tokens_per_step": tokens, "timing": "CUDA graph of the commit call alone, CUDA events"},
        "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "traffic": None,
                     "kernel": "tree_commit_accepted", "algorithmic_bytes": nbytes},
        "gpu_launches": args.steps,
        "cpu_baseline": {"value": tokens / t_cpu, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"the whole commit of this workload, {reps} repeats"},
    }
    print(json.dumps(line), flush=True)


def run_stochastic(args, world, rank, local):
    """--part stochastic: time tree_verify_stochastic (rejection-sampling
    verification at --temperature) on the workload's trees."""
    import torch
    import workloads as W
    import oracle
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    batch = args.batch or 64
    if args.batch and args.workload != "c4":
        raise SystemExit("--batch applies to c4 only")
    # two input sets, used alternately: a call never finds the previous call's rows in L2
    sets = []
    for k in range(2):
        parent, si = W.stochastic_workload(args.workload, temperature=args.temperature, batch=batch, tag=f"stoch{k}")
        sets.append((parent, si))
    parent = sets[0][0]
    B, N = parent.shape
    V = sets[0][1].logits.shape[2]
    depth = W.LEVELS[args.workload]
    dsets = []
    for _, si in sets:
        dsets.append(dict(draft=torch.from_numpy(si.draft).to(dev), logits=torch.from_numpy(si.logits).to(dev),
                          q=torch.from_numpy(si.q).to(dev), coins=torch.from_numpy(si.coins).to(dev)))
    par = torch.from_numpy(np.ascontiguousarray(parent, np.int32)).to(dev)
    outs = [dict(acc=torch.empty((B, depth + 1), dtype=torch.int32, device=dev),
                 L=torch.empty(B, dtype=torch.int32, device=dev), bonus=torch.empty(B, dtype=torch.int32, device=dev),
                 st=torch.zeros(B, dtype=torch.int32, device=dev)) for _ in range(2)]

    def call(k):
        d, o = dsets[k], outs[k]
        ts.tree_verify_stochastic(d["draft"], d["logits"], d["q"], par, d["coins"], args.temperature, o["acc"],
                                  o["L"], o["bonus"], o["st"])

    for i in range(args.warmup):
        call(i & 1)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(args.steps):
            call(i & 1)
    g.replay()
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    w0 = time.time()
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    w1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(w0, w1)
    ms = e0.elapsed_time(e1) / args.steps
    # rows the walks had to read: every visited node's logits, plus its draft row when it has children
    nbytes = 0
    for k in range(2):
        L = outs[k]["L"].cpu().numpy()
        acc = outs[k]["acc"].cpu().numpy()
        assert (outs[k]["st"].cpu().numpy() == 0).all()
        for b in range(B):
            kids = np.bincount(parent[b][1:], minlength=N)
            for u in acc[b][: L[b] + 1]:
                nbytes += V * 4 * (2 if kids[u] else 1)
    nbytes = nbytes / 2 + B * N * 4 * 3   # per call; + drafts, parents, coins
    pk = peaks()
    parent0, si0 = sets[0]
    cpu = None
    if not args.no_cpu_baseline:
        c0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - c0 < 3.0 or reps < 1:
            oracle.stochastic.verify_stochastic(si0.draft, si0.logits, si0.q, parent0, si0.coins, args.temperature,
                                                depth)
            reps += 1
        t_cpu = (time.perf_counter() - c0) / reps
        cpu = {"value": B * N / t_cpu, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"the whole batch of this workload, {reps} repeats"}
    lens = np.concatenate([o["L"].cpu().numpy() for o in outs])
    line = {
        "metric": "stochastic tree verification: tree tokens verified/s", "value": B * N / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload} trees, vocab {V}, B{B}, N{N}; logits 2*N(0,1), draft = target "
                               f"logits + 0.5*N(0,1), temperature {args.temperature}",
                   "part": "stochastic", "mean_accept_len": float(lens.mean()),
                   "timing": "CUDA graph of the call alone, CUDA events; two input sets alternate, so no call "
                             "finds its rows in L2"},
        "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "traffic": None,
                     "kernel": "tree_verify_stochastic", "algorithmic_bytes": nbytes,
                     "note": "bytes = rows of the visited nodes only (the walk is sequential per sequence)"},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_dynamic(args, world, rank, local):
    """--part dynamic: time tree_build_dynamic (rerank a draft's candidate pool
    into the N-node tree and build its masks, depths and positions) on pools
    shaped for the workload's trees, beside tree_build_ancestry on the result."""
    import torch
    import workloads as W
    import oracle
    from tree_attention_speculative_gb300 import _build
    _build.build()
    import tree_attention_speculative_gb300 as ts

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shapes = {"c1": (1, 2, 2, 5), "c2": (1, 6, 8, 64), "c4": (args.batch or 64, 8, 8, 64), "c5": (4, 10, 10, 192)}
    if args.workload not in shapes:
        raise SystemExit("--part dynamic takes c1, c2, c4 or c5")
    B, depth, topk, N = shapes[args.workload]
    pool = W.candidate_pool(W.SEEDS[args.workload], B, depth, topk, W.VOCAB[args.workload])
    M = pool.parent.shape[1]
    plen = np.full(B, 8192, np.int32)

    def i32(x):
        return torch.from_numpy(np.ascontiguousarray(x, np.int32)).to(dev)

    pp, lp, tk, pl = i32(pool.parent), torch.from_numpy(pool.logp).to(dev), i32(pool.token), i32(plen)
    Wd = (N + 63) // 64
    out = dict(parent=torch.empty((B, N), dtype=torch.int32, device=dev),
               tokens=torch.empty((B, N), dtype=torch.int32, device=dev),
               sel=torch.empty((B, N), dtype=torch.int32, device=dev),
               anc=torch.empty((B, N, Wd), dtype=torch.int64, device=dev),
               depth=torch.empty((B, N), dtype=torch.int32, device=dev),
               pos=torch.empty((B, N), dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))

    def dyn():
        ts.tree_build_dynamic(pp, lp, tk, pl, out["parent"], out["tokens"], out["sel"], out["anc"], out["depth"],
                              out["pos"], out["status"])

    def anc_only():
        ts.tree_build_ancestry(out["parent"], pl, out["anc"], out["depth"], out["pos"], out["status"])

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        stream = torch.cuda.Stream(device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(steps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    w0 = time.time()
    ms = timed(dyn, args.steps)
    w1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(w0, w1)
    assert (out["status"].cpu().numpy() == 0).all()
    ms_anc = timed(anc_only, args.steps)
    nbytes = B * M * 12 + B * N * (4 * 5 + 8 * Wd)   # pool in; tree, tokens, indices, depths, positions, masks out
    pk = peaks()
    cpu = None
    if not args.no_cpu_baseline:
        c0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - c0 < 3.0 or reps < 1:
            oracle.dynamic.build_dynamic(pool.parent, pool.logp, pool.token, plen, N)
            reps += 1
        t_cpu = (time.perf_counter() - c0) / reps
        cpu = {"value": B * N / t_cpu, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"the whole batch of this workload, {reps} repeats"}
    line = {
        "metric": "dynamic tree construction: tree tokens built/s", "value": B * N / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}-shaped pools: B{B}, {depth} levels, top-{topk} expansion "
                               f"(M={M} candidates) -> N={N}",
                   "part": "dynamic", "ancestry_only_ms": ms_anc,
                   "timing": "CUDA graph of the call alone, CUDA events; inputs stay in L2 (they are small)"},
        "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "traffic": None,
                     "kernel": "tree_build_dynamic", "algorithmic_bytes": nbytes,
                     "note": "latency-bound: one CTA per sequence, a few KB each"},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_reference(args, world, rank):
    """The oracle as the reference arm: rank 0 alone, on the host cores.  Each
    step is one real, bounded piece of the workload, timed as run (no
    extrapolation): one whole sequence (its ancestry, attention over every kv
    head, argmax of its rows and its walk), or on c5, where a sequence takes
    minutes, one (sequence, kv-head) unit plus that sequence's verification,
    credited as N / Hkv tokens."""
    if rank != 0:
        return
    import workloads as W
    case = W.make(args.workload, **workload_overrides(args))
    B, N, Hkv = case.B, case.N, case.Hkv
    per_unit = args.workload == "c5"

    def step(k):
        if per_unit:
            b, g = divmod(k % (B * Hkv), Hkv)
            return oracle_part(case, [b], [(b, g)]), N / Hkv
        b = k % B
        return oracle_part(case, [b], [(b, g) for g in range(Hkv)]), float(N)

    for k in range(args.warmup):
        step(k)
    w0 = time.time()
    ts, toks = [], 0.0
    for k in range(args.steps):
        t, n = step(args.warmup + k)
        ts.append(t)
        toks += n
    wall = time.time() - w0
    ms = 1e3 * sum(ts) / len(ts)
    v = toks / sum(ts)
    desc = ("one (sequence, kv-head) unit of attention plus its sequence's ancestry, argmax rows and walk per "
            f"step, credited as N/Hkv = {N / Hkv:g} tokens" if per_unit else
            f"one whole sequence per step ({N} tree tokens: ancestry, attention over all {Hkv} kv heads, argmax of "
            "its rows, walk)")
    line = {
        "metric": "tree-verify step: tree tokens verified/s", "value": v, "unit": "tree tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": f"{args.workload}: " + WORKLOAD_DESC[args.workload]},
        "cpu_baseline": {"kind": "oracle", "cores": blas_threads(), "value": v,
                         "sample": f"{desc}; {args.steps} steps in {wall:.1f} s wall, no extrapolation"},
        "e2e": {"value": v, "unit": "tree tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_overrides(args) -> dict:
    kw = {}
    if args.batch:
        if args.workload != "c4":
            raise SystemExit("--batch applies to c4 only")
        kw["batch"] = args.batch
    if args.prefix:
        if args.workload != "c5":
            raise SystemExit("--prefix applies to c5 only")
        kw["prefix"] = args.prefix
    if getattr(args, "forest", 0):
        if args.workload not in ("c2", "c4", "c5"):
            raise SystemExit("--forest applies to c2, c4 and c5")
        kw["forest_roots"] = args.forest
    return kw


def default_steps(workload: str) -> int:
    return {"c1": 20000, "c2": 20000, "c3": 2000, "c4": 200, "c5": 200}[workload]


DEFAULT_WORKLOAD = "c4"


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_DESC), default=DEFAULT_WORKLOAD,
                    help="the headline workload (default c4, the largest; the 70B-shaped layer)")
    ap.add_argument("--sub", default=None,
                    help="comma-separated workloads measured as sub-records of the same line "
                         "(default with c4: c3,c5,c2,c1; otherwise none; 'none' for none)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="override the batch of c4 (smaller profiling case)")
    ap.add_argument("--prefix", type=int, default=0, help="override the prefix length of c5")
    ap.add_argument("--part", choices=["step", "commit", "stochastic", "dynamic"], default="step",
                    help="step: the verification step (default); commit: append accepted paths to the cache; "
                         "stochastic: rejection-sampling verification; dynamic: tree construction from a pool")
    ap.add_argument("--temperature", type=float, default=1.0, help="sampling temperature of --part stochastic")
    ap.add_argument("--forest", type=int, default=0,
                    help="replace each sequence's tree by a forest of this many trees (same nodes and depth)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.sub is None:
        args.sub = "c3,c5,c2,c1" if (args.workload == DEFAULT_WORKLOAD and args.part == "step" and not args.batch
                                     and not args.prefix and not args.forest) else "none"
    args.sub = [] if args.sub in ("", "none") else [w.strip() for w in args.sub.split(",")]
    for w in args.sub:
        if w not in WORKLOAD_DESC:
            raise SystemExit(f"unknown workload in --sub: {w}")
    if args.steps <= 0:
        args.steps = default_steps(args.workload) if args.impl == "ours" else 3
        if args.impl == "ours" and args.part in ("stochastic", "dynamic"):
            args.steps = 3000   # a quarter of a second or more of timed work, long enough for the clock samples
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.part == "commit":
        run_commit(args, world, rank, local)
    elif args.part == "stochastic":
        run_stochastic(args, world, rank, local)
    elif args.part == "dynamic":
        run_dynamic(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
