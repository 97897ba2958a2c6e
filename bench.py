#!/usr/bin/env python3
"""Benchmark of libspecverify on GB300.

A step is one pass of the verification hot path over one batch of the
top-p workload (B=256 requests, k=8 drafts, V=128256, bf16 logits,
temperature 0.7, top-p 0.9): per-row statistics of all 2k+1 rows of every
request, the accept tests with the residual / bonus draw, and the
compaction of the accepted positions' hidden rows (H=7168) for the next
draft step.  The tree path (B=32, 60-node top-4 tree of depth 5) is timed
beside it.  Inputs are synthetic (seeded) and larger than L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank verifies its own
batch (requests are independent: weak scaling, no collective on the data
path); the step time is the max over ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "linear-b256-k8-v128256-t0.7-p0.9"
TREE_WORKLOAD = "tree-b32-n60-k4-d5-v128256"
HIDDEN = 7168
METRIC = "verified logit rows/s at V=128256 bf16; achieved HBM GB/s vs GB300 peak"
UNIT = "rows/s"
PROFILE = os.path.join(ROOT, "profiles", "k_rows_topp_onepass_linear-b256-k8-v128256-t0.7-p0.9.txt")
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # default: 500 steps for the GPU arm (about 0.26 s timed, several clock
    # samples), 20 for the reference arm (one oracle request per step)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-requests", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling runs on a smaller batch)")
    ap.add_argument("--no-tree", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 500
    return args


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def shard(rank: int, B: int, data_seed: int) -> dict:
    """Rank `rank`'s share of the job: B requests with their own ids and data
    seeds (requests are independent; no rank reads another's rows)."""
    return {"first_request": rank * B, "data_seed": data_seed + 97 * rank, "draft_seed": 11 + rank,
            "hidden_seed": data_seed + 1 + rank}


def max_over_ranks(values, world: int, device):
    """Element-wise max of per-rank timings (identity on one rank)."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_value(rows_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: the rows of every rank over the slowest rank's step time."""
    return rows_per_rank * world / (ms / 1e3)


def source_sha() -> str:
    """Hash of the dominant kernel's sources (rows_topp.cu, the one-read
    top-p row statistics, and every kernel header it includes,
    transitively), to tell whether recorded counters still apply."""
    csrc = os.path.join(ROOT, "speculative_decoding_verification_60_gb300", "csrc")
    seen, todo = set(), ["rows_topp.cu"]
    while todo:
        f = todo.pop()
        if f in seen or not os.path.exists(os.path.join(csrc, f)):
            continue
        seen.add(f)
        for line in open(os.path.join(csrc, f)):
            line = line.strip()
            if line.startswith("#include \"") and "/" not in line:
                todo.append(line.split('"')[1])
    h = hashlib.sha256()
    for f in sorted(seen):
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the one-read row-statistics kernel from the
    committed ncu summary, or None when that summary is missing or was taken
    on other kernel sources."""
    if not os.path.exists(PROFILE):
        return None
    kv = {}
    for line in open(PROFILE):
        if ":" in line and line.strip().startswith("- "):
            key, _, val = line.strip()[2:].partition(":")
            val = val.strip()
            if val.startswith("`") and "`" in val[1:]:
                val = val[1:val.index("`", 1)]  # the value quoted in backticks; a comment may follow
            kv[key.strip()] = val
    if kv.get("source_sha") != source_sha():
        return None
    try:
        return float(kv["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def draft_tokens_torch(drf, T: float, top_p: float, seed: int, chunk: int = 256):
    """Synthetic draft tokens: one draw per draft row from its filtered
    softmax (the draft model's own sampling; input generation only)."""
    import torch

    B, k, V = drf.shape
    flat = drf.reshape(B * k, V)
    g = torch.Generator(device=drf.device)
    g.manual_seed(seed)
    out = torch.empty(B * k, dtype=torch.int64, device=drf.device)
    for r0 in range(0, B * k, chunk):
        x = flat[r0:r0 + chunk].float() / T
        p = torch.softmax(x, dim=-1)
        if top_p < 1.0:
            ps, idx = torch.sort(p, dim=-1, descending=True, stable=True)
            keep = (torch.cumsum(ps, dim=-1) - ps) < top_p
            ps = ps * keep
            p = torch.zeros_like(p).scatter_(1, idx, ps)
        out[r0:r0 + chunk] = torch.multinomial(p, 1, generator=g).squeeze(1)
    return out.reshape(B, k).to(torch.int32)


class LinearStep:
    """Device-resident inputs, outputs and workspace of one rank's batch,
    and the raw C-ABI calls of one step."""

    def __init__(self, rank: int, device, batch=None, workload: str = WORKLOAD, temperature=None):
        import torch

        import speculative_decoding_verification_60_gb300 as svp
        import synth

        self.torch = torch
        self.svp = svp
        self.lib = svp.load()
        w = synth.WORKLOADS[workload]
        self.workload = workload
        self.B, self.k, self.V = (batch or w["B"]), w["k"], w["V"]
        self.T = w["T"] if temperature is None else temperature
        self.top_p, self.seed = w["top_p"], w["seed"]
        self.H = w.get("H", HIDDEN)
        B, k, V = self.B, self.k, self.V
        self.dev = device
        sh = shard(rank, B, w["data_seed"])
        self.tgt, self.drf = synth.linear_logits(B, k, V, "bf16", sh["data_seed"], device=device)
        # drafts: the draft model's own samples (greedy: its argmax)
        self.d = (draft_tokens_torch(self.drf, self.T, self.top_p, seed=sh["draft_seed"]) if self.T > 0
                  else self.drf.argmax(dim=-1).to(torch.int32))
        self.req = (torch.arange(B, dtype=torch.int64, device=device) + sh["first_request"])
        self.pos = torch.full((B,), 1000, dtype=torch.int64, device=device)
        self.hidden = synth.hidden_states(B, k + 1, self.H, seed=sh["hidden_seed"], device=device)
        ws = svp.workspace_size(svp.SPEC_OP_LINEAR, B, k, V)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        i32, f32 = torch.int32, torch.float32
        self.acc = torch.empty(B, dtype=i32, device=device)
        self.toks = torch.empty(B, k + 1, dtype=i32, device=device)
        self.aprob = torch.empty(B, k, dtype=f32, device=device)
        self.tprob = torch.empty(B, k, 2, dtype=f32, device=device)
        self.hist = torch.empty(k + 1, dtype=i32, device=device)
        self.err = torch.empty(1, dtype=i32, device=device)
        self.ohid = torch.empty(B * (k + 1), self.H, dtype=torch.bfloat16, device=device)
        self.offs = torch.empty(B + 1, dtype=i32, device=device)
        self.ntok = torch.empty(B * (k + 1), dtype=i32, device=device)
        self.sp = svp.SamplingParams(self.T, self.top_p, self.seed, 0)
        # one read of every target and draft row (greedy: target rows only)
        self.algo_bytes = B * ((2 * k + 1) if self.T > 0 else (k + 1)) * V * 2
        self.mode = 0 if self.T == 0 else (2 if self.top_p < 1.0 else 1)
        # launches of one step: the counters zeroed; the row statistics (the
        # one-read top-p pass, or the two-pass kernel); the finishing launch
        # (rows the one-read pass left, the decisions, the offsets); the draw
        # with the compaction
        self.launches_per_step = 4

    @staticmethod
    def P(t):
        return ctypes.c_void_p(t.data_ptr())

    def stats(self, stream):
        """Row statistics with every request's accept decisions and packed offsets."""
        P = self.P
        st = self.lib.spec_linear_stats_decide(P(self.tgt), P(self.drf), 0, P(self.d), self.B, self.k, self.V,
                                               P(self.req), P(self.pos), ctypes.byref(self.sp), P(self.acc),
                                               P(self.aprob), P(self.tprob), P(self.hist), P(self.err), P(self.ws),
                                               self.ws.numel(), ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, self.svp.status_string(st)

    def draw_compact(self, stream):
        """The residual / bonus draw, with the accepted hidden rows and next
        tokens packed for the next draft step in the same launch."""
        P = self.P
        st = self.lib.spec_linear_draw(P(self.tgt), P(self.drf), 0, P(self.d), self.B, self.k, self.V, P(self.req),
                                       P(self.pos), ctypes.byref(self.sp), P(self.hidden), self.H, P(self.toks),
                                       P(self.ohid), P(self.offs), P(self.ntok), P(self.ws), self.ws.numel(),
                                       ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, self.svp.status_string(st)


def time_linear(step: LinearStep, K: int, W: int, barrier):
    """K timed steps after W warm-up steps, on one stream; returns
    (ms per step, mean ms of the row-statistics launch, launches)."""
    torch = step.torch
    s = torch.cuda.current_stream()
    for _ in range(W):
        step.stats(s)
        step.draw_compact(s)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(K):
        step.stats(s)
        step.draw_compact(s)
    e1.record(s)
    torch.cuda.synchronize()
    barrier()
    ms = e0.elapsed_time(e1) / K
    # the row-statistics call timed on its own, in steps of the same kind
    # (outside the timed steps: an event between two launches keeps the
    # second from starting while the first ends)
    K2 = min(K, 100)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K2)]
    for i in range(K2):
        ev[i][0].record(s)
        step.stats(s)
        ev[i][1].record(s)
        step.draw_compact(s)
    torch.cuda.synchronize()
    stats_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return ms, stats_ms, step.launches_per_step * K


def time_e2e(step: LinearStep, K: int, chunks: int = 4):
    """The same step through the public calls with host buffers: per step the
    inputs are copied from pinned host memory, verified, compacted, and the
    accepted lengths and tokens copied back.  The batch is cut into `chunks`
    request groups so that the copy of group i+1 (a copy stream) overlaps the
    verification of group i; results depend only on request ids and
    positions, so the outputs are those of one call over the whole batch."""
    torch = step.torch
    P = step.P
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    B, k, V = step.B, step.k, step.V
    Bc = (B + chunks - 1) // chunks
    hosts = [step.tgt.cpu().pin_memory(), step.drf.cpu().pin_memory(), step.d.cpu().pin_memory(),
             step.hidden.cpu().pin_memory()]
    devs = [step.tgt, step.drf, step.d, step.hidden]
    outs = [step.acc, step.toks]
    outs_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h2d = sum(h.numel() * h.element_size() for h in hosts)
    d2h = sum(o.numel() * o.element_size() for o in outs)
    ws = torch.empty(step.svp.workspace_size(step.svp.SPEC_OP_LINEAR, Bc, k, V), dtype=torch.uint8,
                     device=step.dev)
    hist = torch.empty(chunks, k + 1, dtype=torch.int32, device=step.dev)
    offs = torch.empty(chunks, Bc + 1, dtype=torch.int32, device=step.dev)
    errs = torch.zeros(chunks, dtype=torch.int32, device=step.dev)  # one slot per group: each call zeroes its own

    def one():
        ready = []
        for c in range(chunks):
            lo, hi = c * Bc, min(B, (c + 1) * Bc)
            with torch.cuda.stream(copy):
                for h, d in zip(hosts, devs):
                    d[lo:hi].copy_(h[lo:hi], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy)
            ready.append(ev)
        for c in range(chunks):
            lo, hi = c * Bc, min(B, (c + 1) * Bc)
            n = hi - lo
            comp.wait_event(ready[c])
            st = step.lib.spec_verify_linear_compact(
                P(step.tgt[lo:hi]), P(step.drf[lo:hi]), 0, P(step.d[lo:hi]), n, k, V, P(step.req[lo:hi]),
                P(step.pos[lo:hi]), ctypes.byref(step.sp), P(step.hidden[lo:hi]), step.H, P(step.acc[lo:hi]),
                P(step.toks[lo:hi]), P(step.aprob[lo:hi]), P(step.tprob[lo:hi]), P(hist[c]),
                P(step.ohid[lo * (k + 1):]), P(offs[c]), P(step.ntok[lo * (k + 1):]), P(errs[c:c + 1]), P(ws),
                ws.numel(), ctypes.c_void_p(comp.cuda_stream))
            assert st == 0, step.svp.status_string(st)
            for o, oh in zip(outs, outs_h):
                oh[lo:hi].copy_(o[lo:hi], non_blocking=True)
        copy.wait_stream(comp)  # the next step's copies overwrite inputs this step still reads

    one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for _ in range(K):
        one()
    comp.wait_stream(copy)
    e1.record(comp)
    torch.cuda.synchronize()
    err = 0
    for v in errs.tolist():  # device errors of the last step, every group
        err |= int(v)
    return e0.elapsed_time(e1) / K, h2d, d2h, chunks, err


def time_sampler(step: LinearStep, K: int, W: int, peak: float):
    """Draft-side sampling (spec_sample_rows) of one token per request: the
    first B draft rows of the batch, V = 128256 bf16, the workload's T and
    top-p.  The 64 MB of rows fit in L2, so L2 is flushed (a 256 MB write)
    before every timed launch, each launch timed alone with CUDA events."""
    torch = step.torch
    B, V = step.B, step.V
    rows = step.drf.reshape(-1, V)[:B]
    req = torch.arange(B, dtype=torch.int64, device=step.dev)
    pos = torch.full((B,), 1001, dtype=torch.int64, device=step.dev)
    out = dict(out_tokens=torch.empty(B, dtype=torch.int32, device=step.dev),
               dev_error=torch.empty(1, dtype=torch.int32, device=step.dev))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=step.dev)
    s = torch.cuda.current_stream()
    for _ in range(W):
        step.svp.sample_rows(rows, step.T, step.top_p, step.seed, req, pos, out=out, stream=s)
    ts = []
    for _ in range(K):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        step.svp.sample_rows(rows, step.T, step.top_p, step.seed, req, pos, out=out, stream=s)
        e1.record(s)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = statistics.mean(ts)
    gbps = B * V * 2 / (ms / 1e3) / 1e9
    return {"workload": f"{B} rows of V={V} bf16, T={step.T}, top-p {step.top_p}", "ms": round(ms, 4),
            "rows_per_s": round(B / (ms / 1e3), 1), "gbps": round(gbps, 1), "frac": round(gbps / peak, 4),
            "launches": K * (2 if step.mode == 2 else 1), "l2": "flushed before every launch"}


def time_tree(device, K: int, W: int, peak: float):
    """The tree workload (B=32, 60-node top-4 tree of depth 5): each node's
    children are distinct tokens drawn without replacement from the
    parent's draft row (input generation only), verified in WOR mode."""
    import numpy as np
    import torch

    import speculative_decoding_verification_60_gb300 as svp
    import synth

    w = synth.WORKLOADS[TREE_WORKLOAD]
    B, N, V = w["B"], w["N"], w["V"]
    parent = synth.pruned_tree(w["K"], w["depth"], N)
    tgt, drf = synth.tree_logits(B, N, V, w["data_seed"], device=device)
    tok = torch.zeros(B, N, dtype=torch.int32, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(w["data_seed"] + 5)
    for n in range(N):
        kids = [i for i in range(1, N) if parent[i] == n]
        if kids:
            p = torch.softmax(drf[:, n].float() / w["T"], -1)
            tok[:, kids] = torch.multinomial(p, len(kids), replacement=False, generator=g).to(torch.int32)
    parent_d = torch.as_tensor(parent, dtype=torch.int32, device=device)
    out = None
    for _ in range(W):
        out = svp.verify_tree(tgt, drf, tok, parent_d, w["depth"], w["T"], w["top_p"], w["seed"], svp.CHILD_WOR)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        out = svp.verify_tree(tgt, drf, tok, parent_d, w["depth"], w["T"], w["top_p"], w["seed"], svp.CHILD_WOR)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    acc = out["accepted_len"].cpu().numpy()
    visited = int(np.sum(acc + 1))                # nodes on the accepted paths (each a target and a draft row)
    path_bytes = visited * 2 * V * 2
    all_bytes = B * N * 2 * V * 2
    gbps = path_bytes / (ms / 1e3) / 1e9
    res = {"workload": TREE_WORKLOAD, "ms_per_step": round(ms, 4), "requests": B, "child_mode": "wor",
           "children": "distinct tokens drawn without replacement from the parent's draft row",
           "visited_nodes": visited, "visited_nodes_per_s": round(visited / (ms / 1e3), 1),
           "mean_accepted_depth": float(np.mean(acc)), "path_bytes": path_bytes, "all_nodes_bytes": all_bytes,
           "path_gbps": round(gbps, 1), "frac": round(gbps / peak, 4)}

    # a tree per request (spec_verify_tree_dynamic): request b keeps the
    # n_b best nodes of the same top-4, depth-5 tree, n_b from 20 to 60
    counts = np.array([20 + (b * 7) % 41 for b in range(B)], dtype=np.int32)
    parents = np.zeros((B, N), dtype=np.int32)
    tok_d = torch.zeros(B, N, dtype=torch.int32, device=device)
    for b in range(B):
        pb = synth.pruned_tree(w["K"], w["depth"], int(counts[b]))
        parents[b, :len(pb)] = pb
        for n in range(len(pb)):
            kids = [i for i in range(1, len(pb)) if pb[i] == n]
            if kids:
                p = torch.softmax(drf[b, n].float() / w["T"], -1)
                tok_d[b, kids] = torch.multinomial(p, len(kids), replacement=False, generator=g).to(torch.int32)
    parents_d = torch.as_tensor(parents, device=device)
    counts_d = torch.as_tensor(counts, device=device)
    for _ in range(W):
        out = svp.verify_tree_dynamic(tgt, drf, tok_d, parents_d, counts_d, w["depth"], w["T"], w["top_p"],
                                      w["seed"], svp.CHILD_WOR)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(K):
        out = svp.verify_tree_dynamic(tgt, drf, tok_d, parents_d, counts_d, w["depth"], w["T"], w["top_p"],
                                      w["seed"], svp.CHILD_WOR)
    e1.record()
    torch.cuda.synchronize()
    ms_d = e0.elapsed_time(e1) / K
    acc_d = out["accepted_len"].cpu().numpy()
    visited_d = int(np.sum(acc_d + 1))
    gbps_d = visited_d * 2 * V * 2 / (ms_d / 1e3) / 1e9
    res["dynamic"] = {"nodes_per_request": f"{int(counts.min())}..{int(counts.max())} (mean {float(counts.mean()):.1f})",
                      "ms_per_step": round(ms_d, 4), "visited_nodes": visited_d,
                      "mean_accepted_depth": float(np.mean(acc_d)), "path_gbps": round(gbps_d, 1),
                      "frac": round(gbps_d / peak, 4), "dev_error": int(out["dev_error"].cpu()[0])}
    return res


# The other workloads the method's pages describe, timed beside the headline
# one: a Llama-1B draft for a 70B-class target (B=64, k=4, T=1) and
# DeepSeek-scale MTP verification with the 7168-wide hidden-state gather
# (B=1024, k=3, V=129280), sampled and greedy.
EXTRA_WORKLOADS = (("linear-b64-k4-v128256", None), ("linear-b1024-k3-v129280-h7168", None),
                   ("linear-b1024-k3-v129280-h7168", 0.0))


def time_workload(name: str, temperature, rank: int, world: int, device, K: int, W: int, peak: float, barrier):
    """One extra workload: the same step (row statistics, decisions,
    compaction) timed on its own inputs (larger than L2), with the row
    statistics launch timed alone and the compaction's gather bytes."""
    import torch

    step = LinearStep(rank, device, workload=name, temperature=temperature)
    ms, stats_ms, launches = time_linear(step, K, W, barrier)
    ms, stats_ms = max_over_ranks([ms, stats_ms], world, device)
    acc = step.acc.to(torch.int64)
    gather = int(((acc + 1) * step.H * 2 * 2).sum())  # accepted hidden rows read and written
    stats_gbps = step.algo_bytes / (stats_ms / 1e3) / 1e9
    out = {"workload": name, "temperature": step.T, "top_p": step.top_p, "B": step.B, "k": step.k, "V": step.V,
           "ms_per_step": round(ms, 4), "rows_per_s": round(job_value(step.B * (step.k + 1), world, ms), 1),
           "stats_ms": round(stats_ms, 4), "stats_gbps": round(stats_gbps, 1), "frac": round(stats_gbps / peak, 4),
           "step_bytes": step.algo_bytes + gather,
           "step_gbps": round((step.algo_bytes + gather) / (ms / 1e3) / 1e9, 1),
           "mean_accepted_len": round(float(acc.float().mean()), 4), "launches_per_step": launches // K,
           "steps": K}
    del step
    torch.cuda.empty_cache()
    return out


def _oracle_request(job):
    """One request through the oracle (a worker process of the all-cores
    timing): returns its wall time."""
    import oracle

    tgt, drf, d, T, top_p, seed, req, pos = job
    t0 = time.perf_counter()
    oracle.verify_linear(tgt, drf, d, T, top_p, seed, req_ids=req, positions=pos)
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(step: LinearStep, n_req: int) -> dict:
    """The oracle, as it stands, on bounded samples of the same batch: n_req
    requests single-threaded (its results compared with the GPU's for the
    same requests), then 2 requests per host core spread over every core
    (one process per core)."""
    import multiprocessing
    from concurrent.futures import ProcessPoolExecutor

    import numpy as np

    import oracle

    sel = list(range(min(n_req, step.B)))
    tgt = step.tgt[sel].cpu()
    drf = step.drf[sel].cpu()
    d = step.d[sel].cpu().numpy()
    req = step.req[sel].cpu().numpy()
    pos = step.pos[sel].cpu().numpy()
    g_acc = step.acc[sel].cpu().numpy()
    g_tok = step.toks[sel].cpu().numpy()
    g_tp = step.tprob[sel].cpu().numpy().astype(np.float64)
    mism = excused = 0
    perr = 0.0
    t0 = time.perf_counter()
    for j, b in enumerate(sel):  # one request at a time, as the method defines it
        r = oracle.verify_linear(tgt[j:j + 1], drf[j:j + 1], d[j:j + 1], step.T, step.top_p, step.seed,
                                 req_ids=req[j:j + 1], positions=pos[j:j + 1])
        if int(r["accepted_len"][0]) != int(g_acc[j]) or not np.array_equal(r["out_tokens"][0], g_tok[j]):
            if r["margin"][0] < 1e-6:
                excused += 1
            else:
                mism += 1
        perr = max(perr, float(np.max(np.abs(g_tp[j] - r["tok_p"][0]))))
    dt = time.perf_counter() - t0
    single = {"value": round(len(sel) * (step.k + 1) / dt, 3), "cores": 1,
              "sample": f"{len(sel)} of {step.B} requests of {step.workload} ({len(sel) * (2 * step.k + 1)} rows), "
                        f"fp64 C oracle, {dt:.1f} s"}
    cores = host_cores()
    n_all = min(step.B, 2 * cores)
    tf = step.tgt[:n_all].float().cpu().numpy()
    qf = step.drf[:n_all].float().cpu().numpy()
    dd = step.d[:n_all].cpu().numpy()
    rq = step.req[:n_all].cpu().numpy()
    ps = step.pos[:n_all].cpu().numpy()
    jobs = [(tf[b:b + 1], qf[b:b + 1], dd[b:b + 1], step.T, step.top_p, step.seed, rq[b:b + 1], ps[b:b + 1])
            for b in range(n_all)]
    # spawn: this process already holds a CUDA context
    with ProcessPoolExecutor(max_workers=cores, mp_context=multiprocessing.get_context("spawn")) as ex:
        list(ex.map(_oracle_request, jobs[:cores]))  # start every worker (imports, library load)
        t1 = time.perf_counter()
        list(ex.map(_oracle_request, jobs))
        wall = time.perf_counter() - t1
    return {"value": round(n_all * (step.k + 1) / wall, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_all} of {step.B} requests of {step.workload}, one process per host core "
                      f"({cores}), fp64 C oracle, {wall:.1f} s wall",
            "single_core": single,
            "parity": {"requests": len(sel), "mismatches": mism, "margin_excused": excused,
                       "max_token_prob_err": perr, "bar": "identical a and tokens unless the oracle's decision "
                                                         "margin is < 1e-6; token probabilities within 1e-5"}}


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if world > 1:
            dist.barrier()

    step = LinearStep(rank, device, args.batch)
    clocks = Clocks(local_rank)
    clocks.start()
    ms, stats_ms, launches = time_linear(step, args.steps, args.warmup, barrier)
    clk = clocks.stop()
    ms, stats_ms = max_over_ranks([ms, stats_ms], world, device)
    rows = step.B * (step.k + 1)
    value = job_value(rows, world, ms)
    e2e_ms, h2d, d2h, chunks, e2e_err = (ms, 0, 0, 1, 0) if args.no_e2e else time_e2e(step, args.e2e_steps)
    e2e_ms = max_over_ranks([e2e_ms], world, device)[0]
    peak0, _ = hbm_peak()
    tree = None if args.no_tree else time_tree(device, max(3, args.steps // 2), 2, peak0)
    extra = [] if args.no_extra else [
        time_workload(name, temp, rank, world, device, max(10, min(100, args.steps // 5)), 3, peak0, barrier)
        for name, temp in EXTRA_WORKLOADS]
    sampler = time_sampler(step, max(3, min(50, args.steps)), 3, peak0)
    peak, peak_kind = hbm_peak()
    achieved = step.algo_bytes / (stats_ms / 1e3) / 1e9
    acc = step.acc.cpu()
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if args.batch is None else f"{WORKLOAD} (B={step.B})", "B": step.B, "k": step.k, "V": step.V, "temperature": step.T,
                   "top_p": step.top_p, "hidden": HIDDEN, "rows_per_step": step.B * (2 * step.k + 1),
                   "l2": "inputs larger than L2 (1116 MB of logits per step, L2 129 MB)",
                   "parallelism": f"dp{world} (independent request shards)" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "kernel": "k_rows_topp_onepass",
                     "timed": "the row-statistics call: the one-read pass and the finishing launch (decisions, "
                              "offsets), events on its stream", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind, "traffic": recorded_traffic(),
                     "algorithmic_bytes_per_launch": step.algo_bytes, "launch_ms": round(stats_ms, 4)},
        "e2e": None if args.no_e2e else {
            "value": round(job_value(rows, world, e2e_ms), 1), "unit": UNIT, "ms_per_step": round(e2e_ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": f"{chunks} request groups, copy of group i+1 overlapping verification of group i",
            "dev_error": e2e_err},
        "gpu_launches": launches,
        "clocks": clk,
        "mean_accepted_len": round(float(acc.float().mean()), 4),
        "tree": tree,
        "draft_sampler": sampler,
        "workloads": extra,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(step, args.cpu_requests)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The reference arm: the oracle, as it stands, on the host cores; each
    step is one request of the same workload."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    import synth

    w = synth.WORKLOADS[WORKLOAD]
    k, V, T, top_p = w["k"], w["V"], w["T"], w["top_p"]
    n = args.warmup + args.steps
    pool = min(n, 32)  # requests generated; step b verifies request b % pool
    tgt, drf = synth.linear_logits(pool, k, V, "bf16", w["data_seed"])
    d = np.zeros((pool, k), dtype=np.int32)
    for b in range(pool):
        d[b] = oracle.sample_rows(drf[b], T, top_p, seed=11, req=np.full(k, b), pos=np.arange(k))
    times = []
    for b in range(n):
        r = b % pool
        t0 = time.perf_counter()
        oracle.verify_linear(tgt[r:r + 1], drf[r:r + 1], d[r:r + 1], T, top_p, w["seed"],
                             req_ids=np.array([r]), positions=np.array([1000]))
        if b >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = (k + 1) / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": 1, "k": k, "V": V, "temperature": T, "top_p": top_p,
                   "note": "each step one request of the workload"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} requests of {WORKLOAD} (a pool of {pool}), one per step, fp64 C oracle"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
