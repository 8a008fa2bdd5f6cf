#!/usr/bin/env python
"""Benchmark of the verify step: verify rows/s and logits HBM GB/s.

Workload (default): 128 requests x 8-token blocks = 1,024 target rows (+ 896
draft rows) x 248,320 vocab, bf16, T = 0.6, top-k 20, top-p 0.95 -- the shape
the pages quote for GB300.  One step = one sv_verify_chain call over the whole
batch with inputs resident in HBM (target-distribution build, draft
distribution, chain test, residual / bonus resample).

Prints one JSON line.  --impl reference times the CPU oracle instead (the
reference arm of this repository: a plain single-threaded C definition),
on a bounded sample of the same workload per step.

Multi-GPU (torchrun): every rank runs its own independent batch on its own
GPU (the requests of a verify step are independent: weak scaling, no
collective on the data path); a barrier brackets the timed region and the
slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "verify rows/s and logits HBM GB/s (% of peak), 1024 rows x 248k vocab bf16"
UNIT = "rows/s"
L2_BYTES = 129 * 1024 * 1024
DESCRIPTIONS = {
    "large": "128 requests x 8-token blocks (1024 target rows + 896 draft rows) x 248,320 vocab bf16; "
             "T=0.6, top-k 20, top-p 0.95",
    "medium": "32 requests x (5+1) rows x 151,936 vocab bf16; T=1.0, top-p 0.95",
    "greedy_wide": "512 requests x 8-token blocks (4096 rows) x 129,280 vocab bf16; greedy",
    "ragged": "256 requests x 16 drafted, budget 2048 tokens, bucket 2048, 248,320 vocab bf16; "
              "half greedy, half T~U[0.3,1.2] top-p 0.9; planner + ragged verify",
    "tiny": "4 requests x (4+1) rows x 1024 vocab fp32",
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="large", choices=sorted(DESCRIPTIONS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline")
    p.add_argument("--quick", action="store_true",
                   help="profiling runs: no settle loop, no end-to-end pass, no CPU baseline")
    p.add_argument("--requests", type=int, default=0, help="scale the batch to this many requests (profiling)")
    p.add_argument("--method", choices=["chain", "block"], default="chain",
                   help="token-by-token chain test, or block verification (uniform layout only)")
    p.add_argument("--estimator", action="store_true",
                   help="uniform layout: each step also predicts acceptance from the draft rows and observes the result")
    p.add_argument("--cost-table", action="store_true",
                   help="ragged workload: choose the budget from a synthetic step-cost table on the device")
    p.add_argument("--no-graph", action="store_true",
                   help="launch each timed step on the stream instead of replaying it as one captured CUDA graph")
    p.add_argument("--shards", type=int, default=0,
                   help="uniform layout: verify over N vocabulary shards (N record passes on this GPU, one merge; "
                        "no exchange, one GPU holds every shard)")
    p.add_argument("--no-promise", action="store_true",
                   help="never pass the small-top-k sampling promise (the full launch sequence of every call)")
    p.add_argument("--fp32", action="store_true",
                   help="the workload's logits in fp32 instead of bf16 (the same values, twice the bytes)")
    return p.parse_args()


def make_workload(args, dev, scale=None):
    """The named workload, its logits in fp32 when --fp32 asks for it."""
    from speculative_decoding_verification_rows_gb300 import workloads
    w = workloads.make(args.workload, device=dev, scale=scale)
    if getattr(args, "fp32", False) and w.dtype != torch.float32:
        w = dataclasses.replace(w, dtype=torch.float32, target=w.target.float().contiguous(),
                                draft=None if w.draft is None else w.draft.float().contiguous())
    return w


# ----------------------------------------------------------------------------
# distributed plumbing (barrier and max over ranks only)
# ----------------------------------------------------------------------------
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks during the load window
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), sm_max=float(f[2]), hw=f[5], hw_thermal=f[6],
                                 sw_thermal=f[7], sw_power=f[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["sm_max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "window": "warm-up + timed region + end-to-end pass (continuous load)"}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# The two row-transform paths: their kernels, the sources that define them,
# and the timing hook of each.
ROW_PATHS = {
    "fast": dict(kernel="fast_rows_kernel (one-pass top-k / argmax row select)", sources=("sv_fast.cu",)),
    "hist": dict(kernel="wide_rows_kernel + hist_rows_kernel (exact per-value histogram, top-p over the vocabulary)",
                 sources=("sv_hist.cu",)),
}


def kernel_source_hash(path_name: str = "fast"):
    h = hashlib.sha256()
    for name in ROW_PATHS[path_name]["sources"] + ("sv_internal.cuh",):
        with open(os.path.join(ROOT, "speculative_decoding_verification_rows_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, path_name: str = "fast"):
    """DRAM bytes per launch of the workload's dominant row kernel from a
    committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("path", "fast") != path_name or rec.get("kernel_source") != kernel_source_hash(path_name):
        return None
    return rec.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# the workload
# ----------------------------------------------------------------------------
def algorithmic_bytes(w) -> tuple[int, int]:
    """(bytes the row kernel must read, target rows) for one step: every target
    row, plus the draft rows of sampling requests, read once."""
    esz = 2 if w.dtype == torch.bfloat16 else 4
    sampling = int((w.temperature > 0).sum())
    if w.layout == "ragged":
        rows_t = w.budget
        rows_d = None   # depends on the plan; filled in by the caller
        return rows_t * w.V * esz, rows_t
    rows_t = w.n * (w.K + 1)
    rows_d = sampling * w.K
    return (rows_t + rows_d) * w.V * esz, rows_t


def path_bytes(w, verify_len=None, method="chain", promise=False) -> tuple[int, int]:
    """Bytes of the rows read by the one-pass kernel (greedy, top-k <= 32) and
    by the histogram kernels (the other sampling rows) in one step: a request
    with window v reads v + 1 target rows, and v draft rows if it samples.
    In chain verification of bf16 rows without the small-top-k promise, the
    library sends greedy rows to the histogram kernel too (as argmax scans)
    whenever some request's kept set takes that path."""
    esz = 2 if w.dtype == torch.bfloat16 else 4
    T = w.temperature.detach().cpu()
    tk = w.top_k.detach().cpu() if w.top_k is not None else torch.zeros_like(T, dtype=torch.int32)
    greedy = T == 0
    k_eff = torch.where(greedy, torch.ones_like(tk), torch.where((tk > 0) & (tk < w.V), tk, torch.full_like(tk, w.V)))
    fast = greedy | (k_eff <= 32)
    if method == "chain" and not promise and w.dtype == torch.bfloat16 and bool((~fast).any()):
        fast = (~greedy) & (k_eff <= 32)
    v = torch.full_like(tk, w.K) if verify_len is None else verify_len.detach().cpu().to(tk.dtype)
    rows = (v + 1) + torch.where(greedy, torch.zeros_like(v), v)
    return int(rows[fast].sum()) * w.V * esz, int(rows[~fast].sum()) * w.V * esz


def small_topk(w) -> bool:
    """Whether every request is greedy or keeps at most 32 tokens by top-k: the
    host-side promise (SAMPLING_SMALL_TOPK) a serving engine can give from the
    batch's sampling settings, which it holds on the host.  Taken once, before
    any timing."""
    T = w.temperature.detach().cpu()
    tk = w.top_k.detach().cpu() if w.top_k is not None else torch.zeros_like(T, dtype=torch.int32)
    return bool(((T == 0) | ((tk >= 1) & (tk <= 32))).all())


def synthetic_cost_table(w, dev):
    """A step-cost table shaped like profiled CUDA-graph buckets: shelves every
    256 submitted tokens up to the bucket, cost rising with the tokens and a
    jump at every 1024 (a larger graph), plus a fixed per-step overhead."""
    toks = list(range(256, w.bucket + 1, 256))
    costs = [1.0 + 0.0006 * t + 0.35 * (t // 1024) for t in toks]
    return (torch.tensor(toks, dtype=torch.int32, device=dev), torch.tensor(costs, dtype=torch.float32, device=dev),
            0.8)


def make_step(w, sv, dev, method="chain", cost_table=False, estimator=False, promise=True, shards=0):
    """A closure running one verify step with preallocated outputs/workspace."""
    ws = sv.Workspace(dev)
    if shards:
        if w.layout != "chain" or method != "chain":
            raise SystemExit("--shards: the uniform layout and the chain method only")
        from speculative_decoding_verification_rows_gb300 import shard
        n, K = w.n, w.K
        bounds = [shard.shard_bounds(w.V, shards, r) for r in range(shards)]
        tgt = [w.target[..., a:b].contiguous() for a, b in bounds]
        drf = [None if w.draft is None else w.draft[..., a:b].contiguous() for a, b in bounds]
        rec = torch.empty((shards, n * (2 * K + 1) * sv.shard_record_bytes()), dtype=torch.uint8, device=dev)
        ws_s = [sv.Workspace(dev) for _ in range(shards)]
        out = sv.VerifyOut(torch.empty(n, dtype=torch.int32, device=dev),
                           torch.empty((n, K + 1), dtype=torch.int32, device=dev),
                           torch.empty(n, dtype=torch.int32, device=dev),
                           torch.empty((n, K + 1), dtype=torch.int32, device=dev))

        def step():
            for r, (a, _) in enumerate(bounds):
                sv.verify_chain_shard_rows(tgt[r], drf[r], w.draft_tokens, w.temperature, w.top_k, w.top_p, a, w.V,
                                           ws=ws_s[r], records=rec[r])
            return sv.verify_chain_shard_merge(rec, shards, w.draft_tokens, w.temperature, w.top_k, w.top_p, w.V,
                                               seed=w.seed, ws=ws, out=out)
        return step, out, None
    n, K = w.n, w.K
    out = sv.VerifyOut(torch.empty(n, dtype=torch.int32, device=dev), torch.empty((n, K + 1), dtype=torch.int32,
                                                                                 device=dev),
                       torch.empty(n, dtype=torch.int32, device=dev), torch.empty((n, K + 1), dtype=torch.int32,
                                                                                 device=dev))
    small = promise and small_topk(w) and method == "chain"
    if w.layout == "chain":
        block = method == "block"
        est = sv.Estimator(w.K, dev) if estimator else None

        q_buf = (torch.empty(int(sv.load().sv_q_rows_bytes(w.n, w.K)), dtype=torch.uint8, device=dev)
                 if estimator and not block else None)

        def step(tgt=w.target, drf=w.draft, toks=w.draft_tokens, T=w.temperature, tk=w.top_k, tp=w.top_p):
            if est is not None and not block:
                # the estimator's pass over the draft rows also serves the verify's q
                x, _, q = est.predict_q(drf, toks, T, tk, tp, q_rows=q_buf)
                o = sv.verify_chain_q(tgt, drf, toks, T, tk, tp, q, seed=w.seed, ws=ws, out=out, small_topk=small)
                est.observe(x, o.accept_len, o.num_emitted)
                return o
            if est is not None:
                x, _ = est.predict(drf, T, tk, tp)
            o = sv.verify_chain(tgt, drf, toks, T, tk, tp, seed=w.seed, ws=ws, out=out, block=block,
                                small_topk=small)
            if est is not None:
                est.observe(x, o.accept_len, o.num_emitted)
            return o
        return step, out, None
    if method != "chain":
        raise SystemExit("block verification is built for the uniform layout only")
    # ragged: planner then verify over target rows packed by the plan
    from speculative_decoding_verification_rows_gb300 import workloads
    ws_p = sv.Workspace(dev)
    table = synthetic_cost_table(w, dev) if cost_table else None

    def plan():
        if table is None:
            return sv.plan_budget(w.conf, w.budget, w.bucket, ws=ws_p)
        _, _, vl_, qo_, tot_, st_ = sv.plan_budget_cost(w.conf, table[0], table[1], w.bucket, table[2], ws=ws_p)
        return vl_, qo_, tot_, st_

    vl, qo, tot, _ = plan()
    packed = workloads.pack_rows(w.target, qo.cpu(), vl.cpu(), w.bucket)
    extra = dict(packed=packed, draft_rows=int(vl[w.temperature > 0].sum()), rows=int(tot), plan=plan, table=table,
                 path_bytes=path_bytes(w, vl, method))

    def step(tgt=packed, drf=w.draft, toks=w.draft_tokens, T=w.temperature, tk=w.top_k, tp=w.top_p):
        vl_, qo_, _, _ = plan()
        extra["verify_lens"], extra["qo"] = vl_, qo_
        return sv.verify_ragged(tgt, drf, qo_, vl_, toks, T, tk, tp, seed=w.seed, ws=ws, out=out,
                                small_topk=small)
    return step, out, extra


def acceptance_stats(w, sv, out, extra):
    """What one step accepted (taken after the timed region from the outputs
    of a plain step): mean accepted drafts and emitted tokens per request,
    the fraction of requests whose accepted length passes each position, and
    for trimmed windows the trim regret of sv_verify_stats (trimmed requests
    that accepted their whole window, over trimmed requests)."""
    vl = None if extra is None else extra.get("verify_lens")
    st = sv.verify_stats(out.accept_len, out.num_emitted, vl, w.K).cpu().tolist()
    acc = out.accept_len.cpu()
    ok = out.num_emitted.cpu() > 0
    a = acc[ok].float()
    per_pos = [round(float((a > j).float().mean()), 4) if len(a) else None for j in range(w.K)]
    return {"mean_accept_len": round(float(a.mean()), 4) if len(a) else None,
            "tokens_emitted_per_step": int(st[0]), "tokens_submitted_per_step": int(st[1]),
            "accept_rate_by_position": per_pos, "requests_with_errors": int((~ok).sum()),
            "requests_trimmed": int(st[2]),
            "trim_regret_rate": round(st[3] / st[2], 4) if st[2] else None,
            "drafter": "drafts drawn from the draft distribution q (greedy requests: softmax at T = 1)"
                       if w.name != "greedy_wide" else "per-position match probabilities of the workload"}


def run_ours(args, rank, world, local):
    from speculative_decoding_verification_rows_gb300 import build as sv_build
    from speculative_decoding_verification_rows_gb300 import sv, workloads
    sv_build.build()
    sv.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = make_workload(args, dev, scale=dict(n=args.requests) if args.requests else None)
    step, out, extra = make_step(w, sv, dev, args.method, args.cost_table, args.estimator, not args.no_promise,
                                 args.shards)
    alg_bytes, rows_t = algorithmic_bytes(w)
    fast_bytes, hist_bytes = path_bytes(w, None, args.method, not args.no_promise and small_topk(w))
    if extra is not None:
        rows_t = extra["rows"]
        alg_bytes = (rows_t + extra["draft_rows"]) * w.V * (2 if w.dtype == torch.bfloat16 else 4)
        fast_bytes, hist_bytes = extra["path_bytes"]
    # the roofline is taken on the path that reads more of the logits (with
    # vocabulary shards: over the whole step)
    roof_path = "hist" if hist_bytes > fast_bytes else "fast"
    roof_bytes = hist_bytes if roof_path == "hist" else fast_bytes

    # prep, row select (with finalisation and the chains of its requests),
    # one-CTA histogram, cluster histogram (rows handed on), chain (the other
    # requests), resample (+ block decision and draw for block verification;
    # + the planner for ragged batches, + the budget choice with a cost
    # table).  Under the small-top-k promise: prep and row select.
    small = small_topk(w) and args.method == "chain" and not args.no_promise
    if small:
        launches_per_step = 2
    elif w.dtype != torch.bfloat16:
        launches_per_step = 3
    else:
        launches_per_step = 6 + (2 if args.method == "block" else 0)
    launches_per_step += (1 if w.layout == "ragged" else 0) + (1 if args.cost_table else 0)
    if args.estimator:   # prep, row select, two histogram kernels, features for the draft rows; observe
        launches_per_step += 6 if args.method == "block" else 6 - (1 if small else 0)
    if args.shards:      # per shard: prep, row select; then prep, merge, chain
        launches_per_step = 2 * args.shards + 3

    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    if not args.quick:
        clocks.start()
        time.sleep(0.3)
        # settle: about a second of steps before the warm-up (untimed)
        t_end = time.time() + 1.0
        while time.time() < t_end:
            step()
        torch.cuda.synchronize()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # One step captured as a CUDA graph and replayed, as a serving engine runs
    # it (the calls do no host synchronisation and allocate nothing).  If the
    # capture fails, the steps are launched on the stream and the reason kept.
    graph, graph_note = None, "stream launches (--no-graph)" if args.no_graph else None
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            torch.cuda.synchronize()
            for _ in range(max(args.warmup, 3)):
                g.replay()
            torch.cuda.synchronize()
            graph, graph_note = g, "one CUDA graph per step (captured once, replayed)"
        except Exception as e:   # keep the stream launches
            graph_note = f"stream launches (graph capture failed: {type(e).__name__}: {str(e)[:160]})"
    run_step = graph.replay if graph is not None else step

    # The same step without the small-top-k promise (the full launch sequence), timed the same way,
    # so the line reports the headline both ways.
    no_promise_ms = None
    if small and not args.quick:
        step_np, _, _ = make_step(w, sv, dev, args.method, args.cost_table, args.estimator, False, args.shards)
        for _ in range(max(args.warmup, 3)):
            step_np()
        g_np = None
        try:
            g_np = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_np):
                step_np()
            torch.cuda.synchronize()
        except Exception:
            g_np = None
        run_np = g_np.replay if g_np is not None else step_np
        for _ in range(3):
            run_np()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            run_np()
        e1.record()
        torch.cuda.synchronize()
        no_promise_ms = e0.elapsed_time(e1) / args.steps

    stream = torch.cuda.current_stream(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        starts[i].record(stream)
        run_step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # The dominant row kernel(s) alone, for the roofline: events recorded by
    # the library on its stream right around those launches (a separate pass,
    # because events between kernels stop the launches from overlapping).
    n_k = max(3, min(args.steps, 20))
    k0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_k)]
    k1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_k)]
    for ev in k0 + k1:      # torch creates the CUDA event on its first record
        ev.record(stream)
    torch.cuda.synchronize()
    set_events = sv.set_hist_timing_events if roof_path == "hist" else sv.set_timing_events
    for i in range(n_k):
        set_events(k0[i], k1[i])
        step()
    set_events(None, None)
    torch.cuda.synchronize()
    kern_ms = [a.elapsed_time(b) for a, b in zip(k0, k1)]
    step()
    torch.cuda.synchronize()
    accept = acceptance_stats(w, sv, out, extra)
    ms_per_step = sum(step_ms) / len(step_ms)
    ms_worst = max_over_ranks(ms_per_step, world)

    # end to end through the public API: pinned host inputs in, results out, every step
    e2e = None if (args.quick or args.shards) else run_e2e(w, sv, dev, extra, max(3, min(args.steps, 10)),
                                                            args.method, not args.no_promise)
    torch.cuda.synchronize()
    clk = clocks.stop()

    value = world * rows_t / (ms_worst / 1e3)
    kern_avg_s = statistics.mean(kern_ms) / 1e3
    if args.shards:   # the records of N shards and the merge on one GPU: the rate over the whole step
        kern_avg_s, roof_bytes = ms_worst / 1e3, fast_bytes
    elif args.estimator and args.method == "chain" and roof_path == "fast":
        # the timed launch is the verify's row kernel, which streams the target rows only (the
        # estimator's pass over the draft rows made their distributions)
        roof_bytes = w.n * (w.K + 1) * w.V * (2 if w.dtype == torch.bfloat16 else 4)
    peak, peak_kind = measured_peak()
    achieved = roof_bytes / kern_avg_s / 1e9
    logits_gbs_step = alg_bytes / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_worst, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "impl": "ours",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}"
                   + (f" (scaled to {w.n} requests)" if args.requests else "")
                   + (" -- block verification" if args.method == "block" else "")
                   + (" -- with the online acceptance estimator (predict + observe)" if args.estimator else "")
                   + (" -- budget from a synthetic step-cost table" if args.cost_table else "")
                   + (f" -- over {args.shards} vocabulary shards on this GPU (records, merge)" if args.shards else ""),
                   "rows_per_step": rows_t,
                   "sampling_promise": "small_topk (every request greedy or top-k <= 32: the full-vocabulary "
                                       "kernels are not launched)" if small else None,
                   "ms_per_step_without_promise": no_promise_ms,
                   "vocab": w.V, "logits_bytes_per_step": alg_bytes,
                   "logits_gbs_step": round(logits_gbs_step, 1),
                   "logits_frac_of_8tbs_step": round(logits_gbs_step / 8000.0, 4),
                   "l2": f"no flush: inputs of {alg_bytes / 1e6:.1f} MB per step exceed the 129 MB L2",
                   "parallelism": f"replicas x{world} (independent batches, no collective)",
                   "step_ms_median": statistics.median(step_ms), "step_ms_min": min(step_ms),
                   "launch": graph_note},
        "roofline": {"bound": "hbm", "kernel": (f"whole step over {args.shards} vocabulary shards (records + merge)"
                                                if args.shards else
                                                "rows32_kernel (fp32 radix descent, top-p over the vocabulary)"
                                                if roof_path == "hist" and w.dtype == torch.float32 else
                                                ROW_PATHS[roof_path]["kernel"]),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)",
                     "traffic": recorded_traffic(args.workload, roof_path), "kernel_ms_mean": statistics.mean(kern_ms),
                     "algorithmic_bytes_per_launch": roof_bytes,
                     "other_path_bytes_per_step": fast_bytes if roof_path == "hist" else hist_bytes},
        "acceptance": accept,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, extra)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(w, sv, dev, extra, steps, method="chain", promise=True):
    """Same metric through the public API from pinned host buffers: H2D of every
    step's inputs and D2H of its results inside the timed region.  Two device
    input buffers and a copy stream let step i+1's inputs cross the host link
    while step i verifies (each buffer is refilled only after the step that
    read it)."""
    names = ["target", "draft", "draft_tokens", "temperature", "top_k", "top_p"]
    dev_t = {k: (extra["packed"] if (k == "target" and extra) else getattr(w, k)) for k in names}
    if extra is not None:
        dev_t["conf"] = w.conf
    host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in dev_t.items()}
    dbufs = [{k: (torch.empty_like(v) if v is not None else None) for k, v in dev_t.items()} for _ in range(2)]
    res_host = [torch.empty(w.n, dtype=torch.int32).pin_memory(),
                torch.empty((w.n, w.K + 1), dtype=torch.int32).pin_memory(),
                torch.empty(w.n, dtype=torch.int32).pin_memory()]
    ws = sv.Workspace(dev)
    ws_p = sv.Workspace(dev)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = sum(t.numel() * t.element_size() for t in res_host)
    small = promise and small_topk(w) and method == "chain"
    comp = torch.cuda.current_stream(dev)
    copy_s = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    freed = [torch.cuda.Event(), torch.cuda.Event()]

    def load(i):
        b = i % 2
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(freed[b])     # the step that read this buffer is done
            for k, v in host.items():
                if v is not None:
                    dbufs[b][k].copy_(v, non_blocking=True)
            copied[b].record(copy_s)

    def verify(i):
        b = i % 2
        d = dbufs[b]
        comp.wait_event(copied[b])
        if extra is None:
            o = sv.verify_chain(d["target"], d["draft"], d["draft_tokens"], d["temperature"], d["top_k"], d["top_p"],
                                seed=w.seed, ws=ws, block=method == "block", small_topk=small)
        else:
            if extra["table"] is None:
                vl, qo, _, _ = sv.plan_budget(d["conf"], w.budget, w.bucket, ws=ws_p)
            else:
                tb = extra["table"]
                _, _, vl, qo, _, _ = sv.plan_budget_cost(d["conf"], tb[0], tb[1], w.bucket, tb[2], ws=ws_p)
            o = sv.verify_ragged(d["target"], d["draft"], qo, vl, d["draft_tokens"], d["temperature"], d["top_k"],
                                 d["top_p"], seed=w.seed, ws=ws, small_topk=small)
        freed[b].record(comp)
        res_host[0].copy_(o.accept_len, non_blocking=True)
        res_host[1].copy_(o.out_tokens, non_blocking=True)
        res_host[2].copy_(o.num_emitted, non_blocking=True)

    def run(n):
        load(0)
        for i in range(n):
            if i + 1 < n:
                load(i + 1)
            verify(i)

    run(2)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(copy_s)
    comp.wait_stream(copy_s)
    run(steps)
    e.record(comp)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    rows = extra["rows"] if extra is not None else w.n * (w.K + 1)
    return {"value": rows / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "every step's inputs copied from pinned host memory and its results read back inside the "
                    "timed region; the next step's copy overlaps this step's verify (two input buffers)"}


# ----------------------------------------------------------------------------
# the CPU oracle (baseline leg and reference arm)
# ----------------------------------------------------------------------------
def _host_logits(t):
    import numpy as np
    t = t.detach().contiguous().cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class pinned_core:
    """Run the calling thread on one core (the last one it may use), as
    taskset would, and restore its affinity afterwards."""

    def __enter__(self):
        self.saved = None
        try:
            self.saved = os.sched_getaffinity(0)
            self.core = max(self.saved)
            os.sched_setaffinity(0, {self.core})
        except (AttributeError, OSError):
            self.core = None
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)


def ragged_slice(w, extra, r0, r1):
    """Host inputs of requests r0..r1-1 of a ragged workload as the plan laid
    them out: their packed target rows (re-based qo_indptr) and block drafts."""
    vl = extra["verify_lens_host"]
    qo = extra["qo_host"]
    rows = extra["packed"][int(qo[r0]):int(qo[r1])]
    return (_host_logits(rows), None if w.draft is None else _host_logits(w.draft[r0:r1]), qo[r0:r1 + 1] - qo[r0],
            vl[r0:r1])


def oracle_sample(w, r0, r1, extra=None):
    """Run the oracle on requests r0..r1-1 (uniform or ragged layout, keys
    of the full batch); returns (target rows, seconds)."""
    import oracle
    args = (w.draft_tokens[r0:r1].cpu().numpy(), w.temperature[r0:r1].cpu().numpy(), w.top_k[r0:r1].cpu().numpy(),
            w.top_p[r0:r1].cpu().numpy())
    if w.layout == "ragged":
        tgt, drf, qo, vl = ragged_slice(w, extra, r0, r1)
        t0 = time.perf_counter()
        oracle.verify_ragged(tgt, drf, qo, vl, *args, seed=w.seed, first_req=r0)
        return int(qo[-1]), time.perf_counter() - t0
    tgt = _host_logits(w.target[r0:r1])
    drf = None if w.draft is None else _host_logits(w.draft[r0:r1])
    t0 = time.perf_counter()
    oracle.verify_chain(tgt, drf, *args, seed=w.seed, first_req=r0)
    dt = time.perf_counter() - t0
    return (r1 - r0) * (w.K + 1), dt


def ragged_host_plan(w, extra):
    """The plan of a ragged workload on the host (the oracle's planner) and its
    packed rows, for the oracle legs."""
    import oracle
    from speculative_decoding_verification_rows_gb300 import workloads
    if extra is None:
        extra = {}
    if "verify_lens" in extra:   # the plan the timed steps used (cost table or not)
        vl, qo = extra["verify_lens"].cpu().numpy(), extra["qo"].cpu().numpy()
    else:
        vl, qo, _, _ = oracle.plan_budget(w.conf.cpu().numpy(), w.budget, w.bucket)
    extra["verify_lens_host"], extra["qo_host"] = vl, qo
    if "packed" not in extra:
        extra["packed"] = workloads.pack_rows(w.target, qo, vl, w.bucket)
    return extra


def cpu_baseline(w, seconds, extra=None):
    import oracle
    oracle.build()
    if w.layout == "ragged":
        extra = ragged_host_plan(w, dict(extra or {}))
    with pinned_core() as pin:
        # requests in order, one at a time, until about `seconds` of CPU work
        rows, dt, n = 0, 0.0, 0
        while n < w.n and dt < seconds:
            r_rows, r_dt = oracle_sample(w, n, n + 1, extra)
            rows, dt, n = rows + r_rows, dt + r_dt, n + 1
    what = "packed target rows of the plan" if w.layout == "ragged" else "target rows"
    return {"value": rows / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"requests 0..{n - 1} of the same workload ({rows} {what}), single thread, fp64",
            "seconds": dt, "host_cores": os.cpu_count(), "pinned_core": pin.core, "cpu_model": cpu_model()}


def run_reference(args, rank, world, local):
    if rank != 0:
        return
    import oracle
    from speculative_decoding_verification_rows_gb300 import workloads
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = make_workload(args, dev)
    extra = ragged_host_plan(w, None) if w.layout == "ragged" else None
    times, rows = [], 0
    with pinned_core() as pin:
        for i in range(max(args.warmup, 3)):
            oracle_sample(w, i % w.n, i % w.n + 1, extra)
        for i in range(args.steps):
            r = (i * 7) % w.n
            n_rows, dt = oracle_sample(w, r, r + 1, extra)
            times.append(dt)
            rows += n_rows
    ms = 1e3 * sum(times) / len(times)
    value = rows / (sum(times))
    sample = (f"one request of the workload per step ({rows / len(times):.1f} target rows + its draft rows on "
              f"average), single thread pinned to core {pin.core}, fp64")
    print(json.dumps({
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                   "rows_per_step": rows / len(times)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model(), "host_cores": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    rank, world, local = dist_init()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
