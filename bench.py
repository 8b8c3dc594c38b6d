"""Benchmark of the MSA block-sparse prefill path on GB300.

One step = one pass of the whole per-layer path on one batch: msa_plan
(build_k2q_csr + work list), the attention kernel and the log-sum-exp
combine -- the unit the MSA prefill page times per layer (vLLM PR 60684,
Performance: build_k2q_csr + attention + combine).

Workload (default): long_prefill_1m -- one request, 2048 query tokens at the
tail of a 1,048,576-token context (8192 pages of 128 tokens), Hkv = 2,
Hq = 16, head dim 128, E4M3 Q/K/V with per-tensor scales, top-16 pages per
(token, KV head) drawn by the pages' rule (random earlier pages, own page
forced, later pages masked), block_table a random permutation.

Metric: selected-token attention TFLOP/s = 4 * 128 * N_pairs / time, with
N_pairs the (query head, key) pairs the causal page mask leaves, and the
per-layer time in microseconds; plus the roofline fraction of the dominant
kernel.  L2 is flushed (256 MiB written) before every timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (torchrun, one process per GPU) every rank runs its own
independent batch of the same shape (different seed): the path has no
exchange between batches, so scaling is weak and no collective touches the
data path; ranks meet only in a barrier and a max-reduction of the timings.

--impl reference times the FP64 CPU oracle (the test-side checker) on the
host cores on bounded samples of the same workload, as a reported baseline.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

WORKLOAD = "long_prefill_1m"
# the metric both arms print (the oracle arm and ours), so the two lines
# compare directly
METRIC = "selected-token attention TFLOP/s"
# the HBM figure the per-layer target is stated against
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 256 << 20
KERNELS_PER_STEP = 6  # plan: prep, mark, rows, scatter; attention; combine
DECODE_KERNELS_PER_STEP = 7  # msa_decode: seq-lens prefix sums, then the same 6
# one (page, KV head) of an NVFP4 pool: K and V slots of 128 x 64 code
# bytes and 128 x 8 E4M3 block scales
NVFP4_PAGE_HEAD_BYTES = 2 * (128 * 64 + 128 * 8)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attention_kernel_traffic.json")
# the dominant kernel's sources, by query type: a recorded DRAM traffic
# figure stays valid while their code is unchanged
ATTN_SOURCES = {"e4m3": ["attention.cu", "ptx.cuh", "common.cuh", "nvfp4.cuh", "partial.cuh"],
                "bf16": ["attention_bf16q.cu", "ptx.cuh", "common.cuh", "partial.cuh"]}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay timing")
    return ap.parse_args()


# ---------------------------------------------------------------- ranks
# One process per GPU under torchrun; every rank runs its own independent
# batch (its own seed).  Ranks exchange only timings and work counts.

def rank_seed(seed, rank):
    return seed + rank


def reduce_over_ranks(values, world, device, op="max"):
    """Element-wise max (timings) or sum (work) over the ranks."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(
            t, op=torch.distributed.ReduceOp.MAX if op == "max"
            else torch.distributed.ReduceOp.SUM)
    return t.tolist()


def job_tflops(total_pairs, step_ms):
    """Whole-job selected-token TFLOP/s: 4 * 128 FLOPs per attended
    (query head, key) pair, summed over ranks, over the slowest rank's
    time."""
    return 4.0 * 128 * total_pairs / (step_ms / 1e3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]),
                "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained",
                                                     p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------- work counts

def pair_and_page_counts(w):
    """(query-head, key) pairs after the causal page mask, and the unique
    (KV head, physical page) set the batch selects -- measurement
    bookkeeping for the metric and the roofline."""
    tk = w.topk.cpu().numpy()
    bt = w.block_table.cpu().numpy()
    pairs = 0
    pages = set()
    off = 0
    for b in range(w.B):
        ql, sl = w.q_lens[b], w.seq_lens[b]
        npg = (sl + 127) // 128
        t0 = int(w.cu_q[b])
        ids = tk[t0:t0 + ql].astype(np.int64)          # [ql, Hkv, 16]
        pos = np.arange(sl - ql, sl)[:, None, None]
        own = pos // 128
        valid = (ids >= 0) & (ids < npg) & (ids <= own)
        # repeats count once
        srt = np.sort(np.where(valid, ids, -1), axis=-1)
        first = np.ones_like(srt, dtype=bool)
        first[..., 1:] = srt[..., 1:] != srt[..., :-1]
        keep = first & (srt >= 0)
        keys = np.where(srt < own, 128, (pos % 128) + 1)
        pairs += int((keys * keep).sum()) * w.G
        for h in range(w.Hkv):
            sel = np.unique(srt[:, h][keep[:, h]])
            for p in sel.tolist():
                pages.add((h, int(bt[b, p])))
        off += npg
    return pairs, len(pages)


def algorithmic_bytes(w, unique_pages):
    """Bytes the step must move: Q once, each selected (KV head, page) once
    (E4M3: 128 x 256 bytes; NVFP4: two slots of codes and block scales),
    out bf16, the top-k ids."""
    q = w.T * w.Hq * 128 * (2 if is_bf16q(w) else 1)
    kv = unique_pages * (NVFP4_PAGE_HEAD_BYTES if is_nvfp4(w) else 128 * 256)
    out = w.T * w.Hq * 128 * 2
    topk = w.T * w.Hkv * 16 * 4
    return {"attention": q + kv, "prefill": q + kv + out,
            "step": q + kv + out + topk}


def source_hash(names):
    """Hash of the kernel sources without their // comments and blank
    lines: the recorded DRAM traffic stays valid across comment edits and is
    dropped as soon as a line of code changes."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_sparse_attention_prefill_gb300", "csrc")
    for n in names:
        with open(os.path.join(d, n)) as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def is_nvfp4(w):
    return getattr(w, "kv4", None) is not None


def is_bf16q(w):
    return getattr(w, "q16", None) is not None


def measured_traffic(workload, query="e4m3"):
    """dram bytes per attention launch on ``workload`` from the committed
    ncu summaries, or None when there is none for it or the kernel source
    changed since it was captured."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    h = source_hash(ATTN_SOURCES[query])
    for e in t if isinstance(t, list) else [t]:
        if e.get("workload") == workload and e.get("source_hash") == h:
            return e.get("bytes_per_launch")
    return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world):
    import block_sparse_attention_prefill_gb300 as msa

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    msa.load()
    w = workloads.make_config(args.workload, seed=rank_seed(args.seed, rank),
                              device="cpu", kv_device=dev)
    pairs, upages = pair_and_page_counts(w)
    wd = w.to(dev)
    stream = torch.cuda.current_stream(dev)

    ws_plan = torch.empty(msa.plan_workspace_bytes(
        w.B, w.T, w.Hq, w.Hkv, w.total_rows, w.max_seqlen_q), dtype=torch.uint8,
        device=dev)
    ws_pre = torch.empty(msa.prefill_workspace_bytes(w.T, w.Hq),
                         dtype=torch.uint8, device=dev)
    out = torch.empty((w.T, w.Hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.Hq), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    decode = is_decode(w)
    fp4 = is_nvfp4(w)
    bf16q = is_bf16q(w)
    if bf16q and (fp4 or decode):
        raise SystemExit("the BF16-query mode is a prefill over the E4M3 pool")
    kv_dev = wd.kv4 if fp4 else wd.kv
    attention_fn = msa.msa_prefill_attention_nvfp4 if fp4 else msa.msa_prefill_attention
    prefill_fn = msa.msa_prefill_nvfp4 if fp4 else msa.msa_prefill
    decode_fn = msa.msa_decode_nvfp4 if fp4 else msa.msa_decode
    if bf16q:
        attention_fn, prefill_fn = msa.msa_prefill_attention_bf16q, msa.msa_prefill_bf16q
    q_key = "q16" if bf16q else "q"
    q_dev = getattr(wd, q_key)
    kv_key = "kv4" if fp4 else "kv"
    if decode:
        # decode-shaped batches go through msa_decode: n tokens at the tail
        # of every request, one call per step
        n_dec = int(w.q_lens[0])
        seq_lens_d = torch.tensor(w.seq_lens, dtype=torch.int32, device=dev)
        ws_dec = torch.empty(msa.decode_workspace_bytes(
            w.B, n_dec, w.Hq, w.Hkv, w.max_seqlen_k), dtype=torch.uint8,
            device=dev)

    def decode_step(ev=None, st=stream):
        if ev:
            ev[0].record(st)
        _, _, plan = decode_fn(wd.q, kv_dev, w.q_scale, w.k_scale,
                               w.v_scale, w.softmax_scale, wd.topk,
                               wd.block_table, seq_lens_d, n_dec,
                               w.max_seqlen_k, workspace=ws_dec, out=out,
                               lse=lse, stream=st)
        if ev:
            for e in ev[1:]:
                e.record(st)
        return plan

    def step_timed(ev, st=stream):
        """One step with events at its two ends only."""
        ev[0].record(st)
        if decode:
            decode_step(None, st)
        else:
            plan = msa.msa_plan(wd.topk, wd.cu_q, wd.cu_k, wd.block_table,
                                w.num_pages, w.Hq, w.total_rows, w.max_seqlen_q,
                                w.max_seqlen_k, workspace=ws_plan, stream=st)
            prefill_fn(q_dev, kv_dev, w.q_scale, w.k_scale, w.v_scale,
                       w.softmax_scale, wd.block_table, plan, workspace=ws_pre,
                       out=out, lse=lse, stream=st)
        ev[1].record(st)

    def step(ev=None, st=stream):
        if decode:
            return decode_step(ev, st)
        if ev:
            ev[0].record(st)
        plan = msa.msa_plan(wd.topk, wd.cu_q, wd.cu_k, wd.block_table,
                            w.num_pages, w.Hq, w.total_rows, w.max_seqlen_q,
                            w.max_seqlen_k, workspace=ws_plan, stream=st)
        if ev:
            ev[1].record(st)
        attention_fn(q_dev, kv_dev, w.q_scale, w.k_scale, w.v_scale,
                     w.softmax_scale, wd.block_table, plan, ws_pre, stream=st)
        if ev:
            ev[2].record(st)
        msa.msa_prefill_combine(plan, ws_pre, out, lse, stream=st)
        if ev:
            ev[3].record(st)
        return plan

    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        flush.zero_()
        plan = step()
    torch.cuda.synchronize()
    status = plan.status()

    # The timed steps carry events only at their two ends: an event between
    # two of the library's kernels would stop the second one's programmatic
    # dependent launch from overlapping the first one's tail, which the step
    # does not do in use.
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        step_timed(evs[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    steps_ms = np.array([a.elapsed_time(b) for a, b in evs])
    step_ms = float(steps_ms.mean())
    step_med_ms = float(np.median(steps_ms))
    total_ms = float(steps_ms.sum())

    # The breakdown into plan / attention / combine, from separate steps
    # with an event at every boundary (reported beside the step, not as it).
    bevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
            for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        step(bevs[i])
    torch.cuda.synchronize()
    per = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]),
                     e[2].elapsed_time(e[3])] for e in bevs])     # ms
    plan_ms, attn_ms, comb_ms = per.mean(axis=0)

    # ---- the same step captured once in a CUDA graph, replayed with the L2
    # flushed before every replay (reported beside the eager figure)
    graph_ms = None
    if not args.no_graph:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(st=cap)
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in gev:
            flush.zero_()
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        graph_ms = float(np.mean([a.elapsed_time(b) for a, b in gev]))

    # ---- end to end through host buffers (pinned), copies inside the region
    e2e = None
    if not args.no_e2e:
        host = {k: getattr(w, k).cpu().pin_memory() if getattr(w, k).device.type == "cpu"
                else getattr(w, k).cpu().pin_memory()
                for k in (q_key, kv_key, "topk", "block_table", "cu_q", "cu_k")}
        dev_in = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
        out_h = torch.empty((w.T, w.Hq, 128), dtype=torch.bfloat16).pin_memory()
        lse_h = torch.empty((w.T, w.Hq), dtype=torch.float32).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = out_h.numel() * 2 + lse_h.numel() * 4
        e2e_steps = max(3, min(args.steps, 20))

        if decode:
            host["seq_lens"] = seq_lens_d.cpu().pin_memory()
            dev_in["seq_lens"] = torch.empty_like(seq_lens_d)
            h2d = sum(v.numel() * v.element_size() for k, v in host.items()
                      if k not in ("cu_q", "cu_k"))

        def e2e_step():
            for k in host:
                if decode and k in ("cu_q", "cu_k"):
                    continue
                dev_in[k].copy_(host[k], non_blocking=True)
            if decode:
                decode_fn(dev_in["q"], dev_in[kv_key], w.q_scale, w.k_scale,
                          w.v_scale, w.softmax_scale, dev_in["topk"],
                          dev_in["block_table"], dev_in["seq_lens"],
                          n_dec, w.max_seqlen_k, workspace=ws_dec,
                          out=out, lse=lse, stream=stream)
                out_h.copy_(out, non_blocking=True)
                lse_h.copy_(lse, non_blocking=True)
                return
            p = msa.msa_plan(dev_in["topk"], dev_in["cu_q"], dev_in["cu_k"],
                             dev_in["block_table"], w.num_pages, w.Hq,
                             w.total_rows, w.max_seqlen_q, w.max_seqlen_k,
                             workspace=ws_plan, stream=stream)
            prefill_fn(dev_in[q_key], dev_in[kv_key], w.q_scale, w.k_scale,
                       w.v_scale, w.softmax_scale, dev_in["block_table"],
                       p, workspace=ws_pre, out=out, lse=lse,
                       stream=stream)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b) / e2e_steps
        e2e = {"ms": e2e_ms, "h2d": h2d, "d2h": d2h}
    clk = clocks.stop()

    total_ms, attn_ms, comb_ms, plan_ms, step_ms, step_med_ms, e2e_ms = reduce_over_ranks(
        [total_ms, attn_ms, comb_ms, plan_ms, step_ms, step_med_ms,
         e2e["ms"] if e2e else 0.0], world, dev, "max")
    (job_pairs,) = reduce_over_ranks([float(pairs)], world, dev, "sum")
    if graph_ms is not None:
        (graph_ms,) = reduce_over_ranks([graph_ms], world, dev, "max")
    return dict(w=w, decode=decode, pairs=pairs, upages=upages, total_ms=total_ms,
                attn_ms=attn_ms, comb_ms=comb_ms, plan_ms=plan_ms,
                step_ms=step_ms, step_med_ms=step_med_ms, e2e=e2e,
                e2e_ms=e2e_ms, clocks=clk,
                job_pairs=job_pairs, graph_ms=graph_ms,
                status=status, t_wall=t_wall)


# ---------------------------------------------------------------- oracle

def oracle_sample_rate(w, budget_s, nthreads):
    """Time the FP64 oracle on a bounded sample of ``w``: a growing subset
    of query tokens, or repeated passes over all of them once the whole
    workload takes less than the budget; returns (TFLOP/s, seconds,
    description)."""
    import oracle

    n = 8
    rng = np.random.default_rng(0)
    while True:
        toks = np.sort(rng.choice(w.T, size=min(n, w.T), replace=False))
        t0 = time.perf_counter()
        _, _, nk = oracle.attention(w, tokens=toks, nthreads=nthreads)
        dt = time.perf_counter() - t0
        if dt >= budget_s or n >= w.T:
            break
        n = int(min(w.T, max(n * 2, n * budget_s / max(dt, 1e-3) * 1.1)))
    flops = 4.0 * 128 * float(nk.sum()) * w.G
    reps = 1
    if dt < budget_s:
        reps = int(math.ceil(budget_s / max(dt, 1e-3)))
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.attention(w, tokens=toks, nthreads=nthreads)
        dt = time.perf_counter() - t0
    desc = "%d of %d query tokens (all %d heads, all their selected pages)" % (
        len(toks), w.T, w.Hq)
    if reps > 1:
        desc += ", %d passes" % reps
    return flops * reps / dt / 1e12, dt, desc


def run_reference(args, rank, world):
    import oracle

    if rank != 0:
        return None
    w = workloads.make_config(args.workload, seed=args.seed)
    nthreads = os.cpu_count() or 1
    pairs, upages = pair_and_page_counts(w)
    per_step = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    rng = np.random.default_rng(1)
    # size one step's token sample to the per-step budget
    probe = np.sort(rng.choice(w.T, size=min(4, w.T), replace=False))
    t0 = time.perf_counter()
    oracle.attention(w, tokens=probe, nthreads=nthreads)
    t_tok = (time.perf_counter() - t0) / len(probe)
    ntok = int(max(1, min(w.T, per_step / max(t_tok, 1e-6))))
    done_flops, done_t = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        toks = np.sort(rng.choice(w.T, size=ntok, replace=False))
        t0 = time.perf_counter()
        _, _, nk = oracle.attention(w, tokens=toks, nthreads=nthreads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            done_flops += 4.0 * 128 * float(nk.sum()) * w.G
            done_t += dt
    value = done_flops / done_t / 1e12
    full_ms = 4.0 * 128 * pairs / (value * 1e12) * 1e3
    sample = "%d of %d query tokens per step, all heads and selected pages" % (
        ntok, w.T)
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": full_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads,
                         "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "note": "FP64 CPU oracle (the parity checker), not a GPU kernel; "
                "ms_per_step is the whole workload extrapolated from the "
                "sampled rate",
    }
    print(json.dumps(line))
    return line


def cpu_model():
    """The host CPU's model name (for the CPU baseline's record)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip() in ("model name", "Model name", "CPU part"):
                    if v.strip():
                        return v.strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def is_decode(w):
    return w.name.startswith("decode")


def config_of(w, args):
    return {"workload": "%s: %s" % (w.name, w.meta.get("description", "")),
            "T": w.T, "seq_lens": w.seq_lens if w.B <= 8 else "%d requests" % w.B,
            "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": 128, "page": 128, "topk": 16,
            "kv_cache": "nvfp4" if is_nvfp4(w) else "e4m3",
            "query": "bf16" if is_bf16q(w) else "e4m3",
            "l2": "flushed before every timed step (256 MiB write)",
            "parallelism": "independent batch per GPU" if args.gpus > 1
            else "single GPU"}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group(
            backend="nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
            return
        r = run_ours(args, rank, world)
        if rank != 0:
            return
        w = r["w"]
        peaks = load_peaks()
        flops = 4.0 * 128 * r["pairs"]
        step_s = r["step_ms"] / 1e3
        value = job_tflops(r["job_pairs"], r["step_ms"])
        alg = algorithmic_bytes(w, r["upages"])
        if r["decode"]:
            # one msa_decode call per step: its kernels are not timed apart,
            # so the roofline covers the whole call and the step's bytes
            roof_bytes, roof_s, roof_kernel = alg["step"], step_s, "msa_decode (%d kernels)" % DECODE_KERNELS_PER_STEP
            traffic = None
            breakdown = {"decode": r["step_ms"] * 1e3}
            launches = DECODE_KERNELS_PER_STEP * args.steps
        else:
            roof_kernel = "attention_bf16q_kernel" if is_bf16q(w) else "attention_kernel"
            roof_bytes, roof_s = alg["attention"], r["attn_ms"] / 1e3
            traffic = measured_traffic(w.name, "bf16" if is_bf16q(w) else "e4m3")
            breakdown = {"plan": r["plan_ms"] * 1e3, "attention": r["attn_ms"] * 1e3,
                         "combine": r["comb_ms"] * 1e3}
            launches = KERNELS_PER_STEP * args.steps
        achieved = roof_bytes / roof_s / 1e9
        # the MMAs' own dtype: bf16 for the BF16 query, E4M3 (2 x the bf16
        # rate) otherwise
        tc_peak = peaks["bf16_tflops"] * (1.0 if is_bf16q(w) else 2.0)
        t_hbm = alg["step"] / (peaks["hbm_gbs"] * 1e9)
        t_fp8 = flops / (tc_peak * 1e12)
        line = {
            "metric": METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": r["step_ms"], "us_per_layer": r["step_ms"] * 1e3,
            "us_per_layer_median": r["step_med_ms"] * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("nvfp4 K/V dequantised to e4m3, e4m3 Q (fp32 accumulate)"
                      if is_nvfp4(w) else
                      "bf16 Q, e4m3 K/V widened to bf16, bf16 MMAs (fp32 accumulate)"
                      if is_bf16q(w) else "e4m3 (fp32 accumulate)"),
            "data": "synthetic",
            "config": config_of(w, args),
            "breakdown_us": breakdown,
            "roofline": {"bound": "hbm", "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": traffic,
                         "kernel": roof_kernel,
                         "algorithmic_bytes": roof_bytes,
                         "peak_source": peaks["source"] + " (burst hbm_gbs)"},
            "roofline_step": {
                "note": "the whole per-layer step (plan + attention + "
                        "combine) against the slower of the MMA dtype's tensor "
                        "peak and its algorithmic bytes over HBM bandwidth",
                "bound": "hbm" if t_hbm >= t_fp8 else "tensor",
                "roofline_us": max(t_hbm, t_fp8) * 1e6,
                "frac": max(t_hbm, t_fp8) / step_s,
                "hbm_peak_gbs": peaks["hbm_gbs"],
                "frac_vs_nominal_8tbs": max(alg["step"] / (NOMINAL_HBM_GBS * 1e9),
                                            t_fp8) / step_s,
                "algorithmic_bytes": alg["step"], "flops": flops,
                "tensor_peak_tflops": tc_peak,
                "tensor_peak_source": ("measured bf16 burst" if is_bf16q(w)
                                       else "2 x measured bf16 burst (E4M3)")},
            "work": {"pairs": r["pairs"], "unique_kv_pages": r["upages"]},
            "gpu_launches": launches,
            "roofline_prefill": None if r["decode"] else {
                "note": "msa_prefill alone (attention + combine, the plan "
                        "excluded): Q, the selected pages and out",
                "bound": "hbm" if alg["prefill"] / (peaks["hbm_gbs"] * 1e9) >= t_fp8
                         else "tensor",
                "roofline_us": max(alg["prefill"] / (peaks["hbm_gbs"] * 1e9), t_fp8) * 1e6,
                "frac": max(alg["prefill"] / (peaks["hbm_gbs"] * 1e9), t_fp8)
                        / ((r["attn_ms"] + r["comb_ms"]) / 1e3),
                "algorithmic_bytes": alg["prefill"]},
            "graph": None if r["graph_ms"] is None else {
                "us_per_layer": r["graph_ms"] * 1e3,
                "value": job_tflops(r["job_pairs"], r["graph_ms"]),
                "unit": "TFLOP/s", "replays": args.steps,
                "note": "the same step captured once in a CUDA graph; "
                        "replayed after the timed steps, L2 flushed before each"},
            "clocks": r["clocks"], "device_status": r["status"],
        }
        if r["e2e"]:
            line["e2e"] = {"value": job_tflops(r["job_pairs"], r["e2e_ms"]),
                           "unit": "TFLOP/s",
                           "h2d_bytes_per_step": r["e2e"]["h2d"],
                           "d2h_bytes_per_step": r["e2e"]["d2h"],
                           "ms_per_step": r["e2e_ms"]}
        if not args.no_cpu_baseline:
            wc = w.to("cpu")
            nthreads = os.cpu_count() or 1
            rate, dt, desc = oracle_sample_rate(wc, 12.0, nthreads)
            rate1, dt1, desc1 = oracle_sample_rate(wc, 4.0, 1)
            line["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s",
                                    "cores": nthreads, "kind": "oracle",
                                    "cpu_model": cpu_model(),
                                    "sample": desc + ", %.1f s" % dt,
                                    "value_1_thread": rate1,
                                    "sample_1_thread": desc1 + ", %.1f s" % dt1}
        print(json.dumps(line))
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
