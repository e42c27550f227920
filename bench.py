#!/usr/bin/env python
"""Benchmark of the Focus attention hot path on GB300 (one JSON line).

A step is one whole layer of the hot path on one batch of synthetic input:
focus_assign -> focus_build_index -> focus_attention_fwd, all through the C
ABI, for every head of the layer.  The default workload is the 32K-token GQA
layer (B=1, 32 query / 8 KV heads, n=32768, d=128, hidden 4096, K=64, w=512).

value        kept-pair TFLOP/s over the whole layer: 4*d FLOPs per kept
             (query, key) pair per head, kept pairs counted exactly from the
             index, divided by the device time of the step.
e2e          the same metric through focus_layer_fwd_host: host->device copies
             of h, W, C, Q, K, V from pinned memory, the three steps, and the
             device->host copy of O, all inside the timed region.
roofline     the dominant attention kernel's achieved TFLOP/s (its algorithmic
             FLOPs per launch over its CUDA-event duration) against the measured
             burst bf16 tensor peak (the kernel runs for well under a second
             inside a millisecond-scale step); the fraction of the sustained
             peak is given beside it.
cpu_baseline the fp64 oracle timed on the host cores on a bounded row sample.
comparators  plain causal attention (ms_dense_causal) and the pages' own
             two-call strategy with a separate combine (ms_two_call_attention)
             on the same inputs and index.

--topk 2 runs the top-2 membership layer instead (focus_assign_topk ->
focus_build_index_topk -> focus_attention_topk_fwd; each token in its two
best groups, a far pair kept when the tokens' group sets meet), by default
with the pages' K = 4 (--K).  Kept pairs are counted once.

--sinkhorn T times the training-time soft assignment instead: scores
(focus_assign_scores) and T Sinkhorn rounds (focus_sinkhorn_fwd) on the
workload's assignment shape; value = algorithmic GB/s of the Sinkhorn rounds
(for K <= 256, K % 4 == 0: S read once up front and once per round, G
written once).

--backward times focus_attention_bwd (dQ, dK, dV over the kept pairs, after
one untimed forward for O and LSE); value = 10*d FLOPs per kept pair per head
(five d-long products: the recomputed score, dO.v, and the dQ, dK, dV
updates) over the device time; bf16 runs on the tensor cores (roofline against
the measured burst bf16 peak; the dQ and dK/dV kernels each recompute the
score and dO.v, 14*d FLOPs executed per pair), fp32 on the CUDA cores (against
the fp32 peak derived from the SM count and clock: 152 x 128 x 2 x 2.07 GHz).

--impl reference times the oracle alone (the comparison arm of this build).
Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling); there is no data-path collective.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "kept-pair TFLOP/s (% of bf16 TC peak), ms/layer at n=32K, speedup vs dense"
UNIT = "TFLOP/s"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20      # larger than the 129 MB L2
L2_NOTE = ("flushed before every timed step: a 256 MB write, then the same 256 MB read back, so the "
           "flush's own dirty lines are written back before the step; flush not timed")


def flush_l2(buf):
    """Evict the step's data from L2: write a buffer larger than L2, then read
    it, so that L2 holds clean lines and no write-back of the flush lands on
    the first timed kernel."""
    buf.zero_()
    buf.amax()


def index_launches(items: int, K: int) -> int:
    """Kernel launches of one focus_build_index call: two for problems of at
    most 4,096 items and 256 groups (one block per problem, then the work
    list), five otherwise."""
    return 2 if items <= 4096 and K <= 256 else 5


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


def tensor_roofline(kernel: str, achieved: float, traffic=None) -> dict:
    """Roofline record of a tensor-core kernel timed inside a short step: the
    measured burst bf16 peak is the denominator, the sustained one is given
    beside it."""
    peaks, kind = load_peaks()
    burst, sus = float(peaks["bf16_tflops"]), float(peaks["bf16_tflops_sustained"])
    return {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
            "frac": achieved / burst, "traffic": traffic, "peak_source": f"{kind} bf16_tflops (burst)",
            "frac_of_sustained": achieved / sus, "peak_sustained": sus}


def max_over_ranks(vals, dist=None, device="cpu"):
    """Each entry's largest value over the ranks: a replica job takes as long
    as its slowest rank.  With no process group the values come back as is."""
    if dist is None:
        return [float(v) for v in vals]
    import torch
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tflops(world: int, flops_per_rank: float, ms: float) -> float:
    """Whole-job throughput: every rank processes its own replica."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_record(kernel: str, workload: str, path: str | None = None):
    """DRAM bytes per launch from a committed ncu summary, if it was captured
    on this workload and the kernel source is unchanged since; else None."""
    path = path or os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "learned_group_sparse_focus_gb300", "csrc", rec["source"])
    try:
        sha = hashlib.sha1(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return rec if sha == rec.get("source_sha1") else None


# ------------------------------------------------------------ oracle arm ---

def oracle_sample(wl, x, rows_per_head: int, heads, seed: int):
    """Time the oracle on a bounded sample: full assignment and index for the
    batch, attention for `rows_per_head` seeded rows of each head in `heads`.
    Returns (kept-pair FLOPs of the sample, seconds, description)."""
    import oracle.focus_ref as ref
    t0 = time.perf_counter()
    gid, _ = ref.assign(x["h"], x["W"], x["C"])
    idx = ref.build_index(gid, wl.K, max(wl.w, 1))
    t1 = time.perf_counter()
    rng = np.random.default_rng(seed)
    kept = ref.kept_counts(idx, max(wl.w, 1))
    flops = 0
    t_attn = 0.0
    for hq in heads:
        kv = ref.kv_head(hq, wl.H, wl.H_kv)
        a = ref.assignment_of_head(hq, wl.H, wl.H_kv, wl.A)
        rows = np.sort(rng.choice(wl.n, size=min(rows_per_head, wl.n), replace=False))
        s = time.perf_counter()
        ref.attention_rows(x["Q"][:, hq:hq + 1], x["K"][:, kv:kv + 1], x["V"][:, kv:kv + 1],
                           gid[:, a:a + 1], wl.w, wl.scale, rows, 1, row_block=256)
        t_attn += time.perf_counter() - s
        flops += 4 * wl.d * int(kept[:, a, rows].sum())
    frac = len(heads) * rows_per_head / (wl.H * wl.n)
    secs = (t1 - t0) * frac + t_attn
    desc = (f"oracle fp64: assign + index over all {wl.B * wl.n} tokens (time prorated by the "
            f"sampled fraction {frac:.2e}) and attention for {rows_per_head} seeded rows of heads "
            f"{list(heads)}")
    return flops, secs, desc


def oracle_sample_topk(wl, x, rows_per_head: int, heads, seed: int, k: int):
    """oracle_sample for top-k membership (assign_topk, build_index_topk,
    attention_rows_topk).  Returns (kept-pair FLOPs of the sample, seconds,
    description)."""
    import oracle.focus_ref as ref
    t0 = time.perf_counter()
    gid, _ = ref.assign_topk(x["h"], x["W"], x["C"], k)
    ref.build_index_topk(gid, wl.K, max(wl.w, 1))
    t1 = time.perf_counter()
    rng = np.random.default_rng(seed)
    flops = 0
    t_attn = 0.0
    for hq in heads:
        kv = ref.kv_head(hq, wl.H, wl.H_kv)
        a = ref.assignment_of_head(hq, wl.H, wl.H_kv, wl.A)
        rows = np.sort(rng.choice(wl.n, size=min(rows_per_head, wl.n), replace=False))
        s = time.perf_counter()
        ref.attention_rows_topk(x["Q"][:, hq:hq + 1], x["K"][:, kv:kv + 1], x["V"][:, kv:kv + 1],
                                gid[:, a:a + 1], wl.w, wl.scale, rows, 1, row_block=128)
        t_attn += time.perf_counter() - s
        for b in range(wl.B):
            flops += 4 * wl.d * int(ref.keep_mask_rows_topk(gid[b, a], max(wl.w, 1), rows).sum())
    frac = len(heads) * rows_per_head / (wl.H * wl.n)
    secs = (t1 - t0) * frac + t_attn
    desc = (f"oracle fp64, top-{k}: assign + index over all {wl.B * wl.n} tokens (time prorated by the "
            f"sampled fraction {frac:.2e}) and attention for {rows_per_head} seeded rows of heads "
            f"{list(heads)}")
    return flops, secs, desc


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    from learned_group_sparse_focus_gb300 import synth
    x = synth.draw(wl)
    heads = [0, wl.H - 1]
    for s in range(args.warmup):
        oracle_sample(wl, x, 64, heads[:1], seed=s)
    tot_f, tot_s, desc = 0, 0.0, ""
    for s in range(args.steps):
        f, sec, desc = oracle_sample(wl, x, args.ref_rows, heads, seed=1000 + s)
        tot_f += f
        tot_s += sec
    v = tot_f / tot_s / 1e12
    ms = tot_s / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, **{k: getattr(wl, k) for k in ("B", "H", "H_kv", "n", "d", "D", "K", "w", "A")}},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc + f"; per step, {args.steps} steps"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU arm ---

def run_ours(args, wl, world, rank, local):
    import torch
    from learned_group_sparse_focus_gb300 import synth
    from learned_group_sparse_focus_gb300 import focus as fz

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    x = synth.draw(wl)

    def dev(a):
        if wl.dtype == "bf16":
            return torch.from_numpy(synth.bf16_bits(a)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()

    d = {k: dev(x[k]) for k in ("h", "W", "C", "Q", "K", "V")}
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace(p)
    gid = torch.empty((wl.B, wl.A, wl.n), dtype=torch.int32, device="cuda")
    O = torch.empty_like(d["Q"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    # one untimed pass: kept-pair counts come from the index itself
    fz.focus_assign(p, d["h"], d["W"], d["C"], gid, ws)
    idx = fz.focus_build_index(p, gid, ws)
    fz.focus_attention_fwd(p, d["Q"], d["K"], d["V"], idx, O, None, ws)
    st = fz.focus_check_errors(ws)
    if st != 0:
        raise RuntimeError(f"device error status {st}")
    far = fz.index_views(p, idx, ws)["farlen_tok"].to(torch.int64).cpu().numpy()   # [B, A, n]
    n_items = int(fz.index_views(p, idx, ws)["n_items"].item())
    win_per_head = int(np.minimum(np.arange(wl.n) + 1, max(wl.w, 1)).sum())
    far_pairs = 0
    for hq in range(wl.H):
        a = 0 if wl.A == 1 else (hq * wl.H_kv) // wl.H
        far_pairs += int(far[:, a, :].sum())
    win_pairs = win_per_head * wl.B * wl.H
    kept = win_pairs + far_pairs
    f_attn, f_group, f_local = 4 * wl.d * kept, 4 * wl.d * far_pairs, 4 * wl.d * win_pairs

    def step(evs):
        flush_l2(flush)
        evs[0].record()
        fz.focus_assign(p, d["h"], d["W"], d["C"], gid, ws)
        evs[1].record()
        ix = fz.focus_build_index(p, gid, ws)
        evs[2].record()
        fz.focus_attention_fwd_timed(p, d["Q"], d["K"], d["V"], ix, O, None, ws, evs[3:7])

    def new_events(k):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(k)]
        for row in evs:            # events are created lazily: record each once
            for e in row:
                e.record()
        return evs

    warm = new_events(1)[0]
    for _ in range(args.warmup):
        step(warm)
    evs = new_events(args.steps)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(int(os.environ.get("FOCUS_NVSMI_INDEX", local))) as clk:
        wall0 = time.perf_counter()
        for s in range(args.steps):
            step(evs[s])
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    st = fz.focus_check_errors(ws)
    if st != 0:
        raise RuntimeError(f"device error status {st}")

    def mean_ms(i, j):
        return statistics.mean(evs[s][i].elapsed_time(evs[s][j]) for s in range(args.steps))

    t_step = mean_ms(0, 6)
    t = {"assign": mean_ms(0, 1), "index": mean_ms(1, 2), "permute_kv": mean_ms(3, 4),
         "group_pass": mean_ms(4, 5), "local_pass": mean_ms(5, 6)}
    t_attn = mean_ms(3, 6)

    # dense causal comparator on the same shape
    for _ in range(3):
        fz.focus_dense_causal_fwd(p, d["Q"], d["K"], d["V"], O, None, ws)
    dn = max(3, min(args.steps, 10))
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(dn)]
    for a0, a1 in dev_ev:
        flush_l2(flush)
        a0.record()
        fz.focus_dense_causal_fwd(p, d["Q"], d["K"], d["V"], O, None, ws)
        a1.record()
    torch.cuda.synchronize()
    t_dense = statistics.mean(a0.elapsed_time(a1) for a0, a1 in dev_ev)

    # two-call comparator (group call, window call, separate combine) on the same index
    for _ in range(3):
        fz.focus_attention_two_call_fwd(p, d["Q"], d["K"], d["V"], idx, O, None, ws)
    tc_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(dn)]
    for a0, a1 in tc_ev:
        flush_l2(flush)
        a0.record()
        fz.focus_attention_two_call_fwd(p, d["Q"], d["K"], d["V"], idx, O, None, ws)
        a1.record()
    torch.cuda.synchronize()
    t_two = statistics.mean(a0.elapsed_time(a1) for a0, a1 in tc_ev)

    # end to end through the host-buffer entry point
    host = {k: d[k].cpu().pin_memory() for k in ("h", "W", "C", "Q", "K", "V")}
    host["O"] = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    dbuf = {k: torch.empty_like(d[k]) for k in ("h", "W", "C", "Q", "K", "V")}
    dbuf["O"] = torch.empty_like(O)
    dbuf["gid"] = torch.empty_like(gid)
    h2d = sum(host[k].numel() * host[k].element_size() for k in ("h", "W", "C", "Q", "K", "V"))
    d2h = host["O"].numel() * host["O"].element_size()
    for _ in range(2):
        fz.focus_layer_fwd_host(p, host, dbuf, ws)
    en = max(3, min(args.steps, 10))
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(en)]
    for a0, a1 in e2e_ev:
        flush_l2(flush)
        a0.record()
        fz.focus_layer_fwd_host(p, host, dbuf, ws)
        a1.record()
    torch.cuda.synchronize()
    t_e2e = statistics.mean(a0.elapsed_time(a1) for a0, a1 in e2e_ev)
    st = fz.focus_check_errors(ws)
    if st != 0:
        raise RuntimeError(f"device error status {st}")
    if not torch.equal(host["O"].cuda(), O):
        # dense comparator overwrote O; recompute the device result for the check
        fz.focus_attention_fwd(p, d["Q"], d["K"], d["V"], fz.focus_build_index(p, gid, ws), O, None, ws)
        torch.cuda.synchronize()
        if not torch.equal(host["O"].cuda(), O):
            raise RuntimeError("host-buffer path and device path disagree")

    names = list(t)
    red = max_over_ranks([t_step, t_attn, t_dense, t_e2e, t_two] + [t[k] for k in names], dist, "cuda")
    t_step, t_attn, t_dense, t_e2e, t_two = red[:5]
    t = dict(zip(names, red[5:]))

    peaks, peak_kind = load_peaks()
    peak_hbm = float(peaks["hbm_gbs"])
    dom = "group_pass" if t["group_pass"] >= t["local_pass"] else "local_pass"
    dom_flops = f_group if dom == "group_pass" else f_local
    achieved = dom_flops / (t[dom] * 1e-3) / 1e12
    tr = traffic_record("attn_tc_" + dom, wl.name)
    value = job_tflops(world, f_attn, t_step)
    es = 2 if wl.dtype == "bf16" else 4
    assign_bytes = (wl.B * wl.n * wl.D + wl.A * wl.d_g * wl.D + wl.A * wl.K * wl.d_g) * es + wl.B * wl.A * wl.n * 4
    kv_bytes = 2 * wl.B * wl.H_kv * wl.n * wl.d * es
    # index: gid read once, perm, rank, farlen per token and per slot written (int32)
    index_bytes = wl.B * wl.A * wl.n * 4 * 5
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded N(0,1) Q/K/V/h, Zipf-planted groups)",
        "config": {"workload": wl.name, **{k: getattr(wl, k) for k in ("B", "H", "H_kv", "n", "d", "D", "d_g", "K", "w", "A")},
                   "kept_pairs": kept, "kept_density_vs_causal": kept / (wl.B * wl.H * wl.n * (wl.n + 1) / 2),
                   "work_items": n_items, "l2": L2_NOTE,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_bf16_peak": 100.0 * (f_attn / (t_step * 1e-3) / 1e12) / float(peaks["bf16_tflops"]),
        "attention_tflops": f_attn / (t_attn * 1e-3) / 1e12,
        "ms_breakdown": t, "ms_attention": t_attn, "ms_dense_causal": t_dense,
        "speedup_vs_dense": t_dense / t_step, "speedup_vs_dense_attention_only": t_dense / t_attn,
        "ms_two_call_attention": t_two, "fused_vs_two_call": t_two / t_attn,
        "roofline": tensor_roofline("attn_tc_" + dom, achieved, tr["bytes_per_launch"] if tr else None),
        "kernels": {
            "assign": {"ms": t["assign"], "GB/s": assign_bytes / (t["assign"] * 1e-3) / 1e9,
                       "hbm_frac": assign_bytes / (t["assign"] * 1e-3) / 1e9 / peak_hbm},
            "permute_kv": {"ms": t["permute_kv"], "GB/s": 2 * kv_bytes / (t["permute_kv"] * 1e-3) / 1e9},
            "group_pass": {"ms": t["group_pass"], "TFLOP/s": f_group / (t["group_pass"] * 1e-3) / 1e12},
            "local_pass": {"ms": t["local_pass"], "TFLOP/s": f_local / (t["local_pass"] * 1e-3) / 1e12},
            "index": {"ms": t["index"], "GB/s": index_bytes / (t["index"] * 1e-3) / 1e9,
                      "hbm_frac": index_bytes / (t["index"] * 1e-3) / 1e9 / peak_hbm},
        },
        "e2e": {"value": job_tflops(world, f_attn, t_e2e), "unit": UNIT, "ms_per_step": t_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "call": "focus_layer_fwd_host (pinned host buffers)"},
        "gpu_launches": (4 + index_launches(wl.n, wl.K)) * args.steps,
        "wall_s_timed_region": wall,
    }
    if rank == 0:
        line["clocks"] = clk.summary()
        if world == 1 and not args.no_cpu_baseline:
            heads = sorted({0, wl.H // 3, (2 * wl.H) // 3, wl.H - 1})
            f, sec, desc = oracle_sample(wl, x, args.cpu_rows, heads, seed=7)
            line["cpu_baseline"] = {"value": f / sec / 1e12, "unit": UNIT, "cores": cpu_cores(),
                                    "kind": "oracle", "sample": desc, "seconds": sec}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_ours_topk(args, wl, world, rank, local):
    """The top-k layer: same timing rules as run_ours (L2 flushed before each
    timed step, CUDA events on the launching stream, clocks sampled)."""
    import torch
    from learned_group_sparse_focus_gb300 import synth
    from learned_group_sparse_focus_gb300 import focus as fz

    k = args.topk
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    x = synth.draw(wl)

    def dev(a):
        if wl.dtype == "bf16":
            return torch.from_numpy(synth.bf16_bits(a)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()

    names = ("h", "W", "C", "Q", "K", "V")
    d = {n_: dev(x[n_]) for n_ in names}
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace_topk(p, k)
    gid = torch.empty((wl.B, wl.A, wl.n, k), dtype=torch.int32, device="cuda")
    O = torch.empty_like(d["Q"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    fz.focus_assign_topk(p, k, d["h"], d["W"], d["C"], gid, ws)
    idx = fz.focus_build_index_topk(p, k, gid, ws)
    fz.focus_attention_topk_fwd(p, d["Q"], d["K"], d["V"], idx, O, None, ws)
    st = fz.focus_check_errors(ws)
    if st != 0:
        raise RuntimeError(f"device error status {st}")
    # far pairs per assignment: entry far keys (a key sharing both groups
    # counted twice) minus pair far keys (those keys once more); the split
    # index (K <= 8) counts every far pair once and has no pair index
    ent = fz.index_views(p, idx.entry, ws, n=wl.n * k, K=wl.K * wl.K if idx.split else wl.K)
    far_e = ent["farlen_tok"].to(torch.int64).sum(dim=2).cpu().numpy()       # [B, A]
    if k == 2 and not idx.split:
        pv = fz.index_views(p, idx.pair, ws, K=wl.K * (wl.K - 1) // 2)
        far_p = pv["farlen_tok"].to(torch.int64).sum(dim=2).cpu().numpy()
    else:
        far_p = np.zeros_like(far_e)
    heads_of = [0 if wl.A == 1 else (hq * wl.H_kv) // wl.H for hq in range(wl.H)]
    far_pairs = sum(int(far_e[:, a].sum() - far_p[:, a].sum()) for a in heads_of)
    ent_pairs = sum(int(far_e[:, a].sum()) for a in heads_of)
    pair_pairs = sum(int(far_p[:, a].sum()) for a in heads_of)
    win_pairs = int(np.minimum(np.arange(wl.n) + 1, max(wl.w, 1)).sum()) * wl.B * wl.H
    kept = win_pairs + far_pairs
    f_attn = 4 * wl.d * kept

    def step(evs):
        flush_l2(flush)
        evs[0].record()
        fz.focus_assign_topk(p, k, d["h"], d["W"], d["C"], gid, ws)
        evs[1].record()
        ix = fz.focus_build_index_topk(p, k, gid, ws)
        evs[2].record()
        fz.focus_attention_topk_fwd_timed(p, d["Q"], d["K"], d["V"], ix, O, None, ws, evs[3:8])

    def new_events(cnt):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(cnt)]
        for row in evs:
            for e in row:
                e.record()
        return evs

    warm = new_events(1)[0]
    for _ in range(args.warmup):
        step(warm)
    evs = new_events(args.steps)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(int(os.environ.get("FOCUS_NVSMI_INDEX", local))) as clk:
        for s_ in range(args.steps):
            step(evs[s_])
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
    st = fz.focus_check_errors(ws)
    if st != 0:
        raise RuntimeError(f"device error status {st}")

    def mean_ms(i, j):
        return statistics.mean(evs[s_][i].elapsed_time(evs[s_][j]) for s_ in range(args.steps))

    t = {"assign": mean_ms(0, 1), "index": mean_ms(1, 2), "permute_kv": mean_ms(3, 4),
         "entry_group_pass": mean_ms(4, 5), "pair_pass_and_merge": mean_ms(5, 6),
         "local_pass": mean_ms(6, 7)}
    t_step = mean_ms(0, 7)

    # dense comparator
    dws = fz.alloc_workspace(p)
    for _ in range(3):
        fz.focus_dense_causal_fwd(p, d["Q"], d["K"], d["V"], O, None, dws)
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
    for a0, a1 in dev_ev:
        flush_l2(flush)
        a0.record()
        fz.focus_dense_causal_fwd(p, d["Q"], d["K"], d["V"], O, None, dws)
        a1.record()
    torch.cuda.synchronize()
    t_dense = statistics.mean(a0.elapsed_time(a1) for a0, a1 in dev_ev)
    del dws

    # end to end: pinned host inputs in, the three calls, O back to pinned host
    host = {n_: d[n_].cpu().pin_memory() for n_ in names}
    hO = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    h2d = sum(host[n_].numel() * host[n_].element_size() for n_ in names)
    d2h = hO.numel() * hO.element_size()

    def e2e_step():
        for n_ in names:
            d[n_].copy_(host[n_], non_blocking=True)
        fz.focus_assign_topk(p, k, d["h"], d["W"], d["C"], gid, ws)
        ix = fz.focus_build_index_topk(p, k, gid, ws)
        fz.focus_attention_topk_fwd(p, d["Q"], d["K"], d["V"], ix, O, None, ws)
        hO.copy_(O, non_blocking=True)

    for _ in range(2):
        e2e_step()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
    for a0, a1 in e2e_ev:
        flush_l2(flush)
        a0.record()
        e2e_step()
        a1.record()
    torch.cuda.synchronize()
    t_e2e = statistics.mean(a0.elapsed_time(a1) for a0, a1 in e2e_ev)

    keys = list(t)
    red = max_over_ranks([t_step, t_dense, t_e2e] + [t[kk] for kk in keys], dist, "cuda")
    t_step, t_dense, t_e2e = red[:3]
    t = dict(zip(keys, red[3:]))
    f_ent = 4 * wl.d * ent_pairs
    achieved = f_ent / (t["entry_group_pass"] * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": job_tflops(world, f_attn, t_step), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": f"synthetic (seeded N(0,1) Q/K/V/h, {wl.groups} hidden states), top-{k} membership",
        "config": {"workload": wl.name, "topk": k,
                   **{kk: getattr(wl, kk) for kk in ("B", "H", "H_kv", "n", "d", "D", "d_g", "K", "w", "A")},
                   "kept_pairs": kept, "kept_density_vs_causal": kept / (wl.B * wl.H * wl.n * (wl.n + 1) / 2),
                   "far_pairs_entry_pass": ent_pairs, "far_pairs_pair_pass": pair_pairs,
                   "topk_index": "split (each far pair once)" if idx.split else "entry + pair",
                   "l2": L2_NOTE,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "ms_breakdown": t, "ms_dense_causal": t_dense, "speedup_vs_dense": t_dense / t_step,
        "roofline": tensor_roofline("attn_tc_group_pass (entries)", achieved),
        "e2e": {"value": job_tflops(world, f_attn, t_e2e), "unit": UNIT, "ms_per_step": t_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "call": "pinned host copies + focus_assign_topk, focus_build_index_topk, focus_attention_topk_fwd"},
        "gpu_launches": (1 + (12 if k == 2 else index_launches(wl.n * k, wl.K)) + (6 if k == 2 else 3)) * args.steps,
    }
    if rank == 0:
        line["clocks"] = clk.summary()
        if world == 1 and not args.no_cpu_baseline:
            heads = sorted({0, wl.H - 1})
            f, sec, desc = oracle_sample_topk(wl, x, max(64, args.cpu_rows // 8), heads, seed=7, k=k)
            line["cpu_baseline"] = {"value": f / sec / 1e12, "unit": UNIT, "cores": cpu_cores(),
                                    "kind": "oracle", "sample": desc, "seconds": sec}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_ours_sinkhorn(args, wl, world, rank, local):
    import torch
    from learned_group_sparse_focus_gb300 import synth
    from learned_group_sparse_focus_gb300 import focus as fz

    T = args.sinkhorn
    torch.cuda.set_device(local)
    x = synth.draw(wl, parts=("assign",))

    def dev(a):
        if wl.dtype == "bf16":
            return torch.from_numpy(synth.bf16_bits(a)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()

    h, W, C = (dev(x[k]) for k in ("h", "W", "C"))
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace_sinkhorn(p)
    S = torch.empty((wl.B, wl.A, wl.n, wl.K), dtype=torch.float32, device="cuda")
    G = torch.empty_like(S)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        fz.focus_assign_scores(p, h, W, C, S, ws)
        fz.focus_sinkhorn_fwd(p, T, 1.0, S, G, ws)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(int(os.environ.get("FOCUS_NVSMI_INDEX", local))) as clk:
        for e in ev:
            flush_l2(flush)
            e[0].record()
            fz.focus_assign_scores(p, h, W, C, S, ws)
            e[1].record()
            fz.focus_sinkhorn_fwd(p, T, 1.0, S, G, ws)
            e[2].record()
        torch.cuda.synchronize()
    if fz.focus_check_errors(ws) != 0:
        raise RuntimeError("device error")
    t_sc = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    t_sk = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    sbytes = S.numel() * 4
    # K <= 256: S once up front and once per round, G once; larger K: S twice
    # per round, G once, u per round
    fused = wl.K <= 256 and wl.K % 4 == 0
    alg = (T + 2) * sbytes if fused else (2 * T + 1) * sbytes + 4 * wl.B * wl.A * wl.n * T
    peaks, peak_kind = load_peaks()
    gbs = alg / (t_sk * 1e-3) / 1e9
    line = {
        "metric": "Sinkhorn forward algorithmic GB/s", "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_sc + t_sk, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "rounds": T, "tau": 1.0,
                   **{k: getattr(wl, k) for k in ("B", "n", "D", "d_g", "K", "A")},
                   "S_bytes": sbytes, "l2": L2_NOTE},
        "ms_breakdown": {"scores": t_sc, "sinkhorn": t_sk, "per_round": t_sk / T},
        "roofline": {"bound": "hbm", "kernel": "sinkhorn rounds", "achieved": gbs,
                     "peak": float(peaks["hbm_gbs"]), "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]),
                     "traffic": None, "peak_source": f"{peak_kind} hbm_gbs",
                     "note": "S is L2-resident when smaller than ~100 MB, so frac can exceed 1"},
        "gpu_launches": ((2 + T) if fused else (1 + 3 * T)) * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle.focus_ref as ref
        rows = min(wl.n, 8192)
        t0 = time.perf_counter()
        Sref = ref.scores(x["h"][:, :rows], x["W"], x["C"])
        ref.sinkhorn(Sref, T, 1.0)
        sec = time.perf_counter() - t0
        ab = ((T + 2) * Sref.size * 4 if fused
              else (2 * T + 1) * Sref.size * 4 + 4 * Sref.shape[0] * Sref.shape[1] * rows * T)
        line["cpu_baseline"] = {"value": ab / sec / 1e9, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": f"oracle fp64 scores + {T} Sinkhorn rounds on the first {rows} tokens "
                                          f"(the same bytes-per-round accounting)", "seconds": sec}
    if rank == 0:       # one replica per process; rank 0 reports its own
        print(json.dumps(line), flush=True)


FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12     # CUDA-core fp32 FMA peak


def run_ours_backward(args, wl, world, rank, local):
    import torch
    from learned_group_sparse_focus_gb300 import synth
    from learned_group_sparse_focus_gb300 import focus as fz

    torch.cuda.set_device(local)
    x = synth.draw(wl, parts=("attn",))
    rng = np.random.default_rng(wl.seed + 17)
    dO_np = synth.round_bf16(rng.standard_normal(x["Q"].shape).astype(np.float32)) if wl.dtype == "bf16" \
        else rng.standard_normal(x["Q"].shape).astype(np.float32)

    def dev(a):
        if wl.dtype == "bf16":
            return torch.from_numpy(synth.bf16_bits(a)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()

    Q, K, V, dO = dev(x["Q"]), dev(x["K"]), dev(x["V"]), dev(dO_np)
    g = torch.from_numpy(synth.draw_group_ids(wl.seed, wl.B, wl.A, wl.n, wl.K, wl.groups)).cuda()
    p = fz.params_from_workload(wl)
    ws = fz.alloc_workspace(p)
    wsb = fz.alloc_workspace_backward(p)
    idx = fz.focus_build_index(p, g, ws)
    O = torch.empty_like(Q)
    lse = torch.empty((wl.B, wl.H, wl.n), dtype=torch.float32, device="cuda")
    fz.focus_attention_fwd(p, Q, K, V, idx, O, lse, ws)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    far = fz.index_views(p, idx, ws)["farlen_tok"].to(torch.int64).cpu().numpy()
    win = int(np.minimum(np.arange(wl.n) + 1, max(wl.w, 1)).sum()) * wl.B * wl.H
    far_pairs = sum(int(far[:, 0 if wl.A == 1 else (h * wl.H_kv) // wl.H, :].sum()) for h in range(wl.H))
    kept = win + far_pairs
    flops = 10 * wl.d * kept
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        fz.focus_attention_bwd(p, Q, K, V, O, dO, lse, idx, dQ, dK, dV, wsb)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(int(os.environ.get("FOCUS_NVSMI_INDEX", local))) as clk:
        for a0, a1 in ev:
            flush_l2(flush)
            a0.record()
            fz.focus_attention_bwd(p, Q, K, V, O, dO, lse, idx, dQ, dK, dV, wsb)
            a1.record()
        torch.cuda.synchronize()
    if fz.focus_check_errors(ws) != 0 or fz.focus_check_errors(wsb) != 0:
        raise RuntimeError("device error")
    t = statistics.mean(a0.elapsed_time(a1) for a0, a1 in ev)
    tf = flops / (t * 1e-3) / 1e12
    line = {
        "metric": "backward kept-pair TFLOP/s (10*d FLOP per kept pair per head)", "value": tf,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, **{k: getattr(wl, k) for k in ("B", "H", "H_kv", "n", "d", "K", "w", "A")},
                   "kept_pairs": kept, "l2": L2_NOTE},
        "roofline": (tensor_roofline("backward (tcgen05 dQ and dK/dV kernels)", tf)
                     if wl.dtype == "bf16" else
                     {"bound": "alu", "kernel": "backward (fp32 CUDA cores)", "achieved": tf,
                      "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s", "frac": tf / FP32_ALU_TFLOPS, "traffic": None,
                      "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz"}),
        "gpu_launches": (7 if wl.dtype == "bf16" else 5) * args.steps,
        "clocks": clk.summary(),
        "ms_note": ("bf16: the index-order copies of Q/dO/LSE with Delta and of K/V, the far dK/dV work order, "
                    "and 4 persistent tcgen05 kernels (dQ far, dQ window, dK/dV far, dK/dV window)"
                    if wl.dtype == "bf16" else
                    "fp32: delta + 4 CUDA-core kernels"),
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle.focus_ref as ref
        nb = min(wl.n, 1024)
        Hs = min(wl.H, 2 * (wl.H // wl.H_kv))
        Hkv_s = max(1, Hs * wl.H_kv // wl.H)
        gs = synth.draw_group_ids(wl.seed, wl.B, wl.A, wl.n, wl.K, wl.groups)[:, :, :nb]
        t0 = time.perf_counter()
        ref.attention_backward(x["Q"][:, :Hs, :nb], x["K"][:, :Hkv_s, :nb], x["V"][:, :Hkv_s, :nb], gs[:, :min(wl.A, Hkv_s)],
                               max(wl.w, 1), wl.scale, min(wl.A, Hkv_s), dO_np[:, :Hs, :nb])
        sec = time.perf_counter() - t0
        kept_s = 0
        for b in range(wl.B):
            for h in range(Hs):
                a = 0 if wl.A == 1 else ref.kv_head(h, Hs, Hkv_s)
                kept_s += int(ref.keep_mask_rows(gs[b, a], max(wl.w, 1), np.arange(nb)).sum())
        line["cpu_baseline"] = {"value": 10 * wl.d * kept_s / sec / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
                                "kind": "oracle",
                                "sample": f"oracle fp64 backward on the first {nb} tokens of {Hs} query heads",
                                "seconds": sec}
    if rank == 0:       # one replica per process; rank 0 reports its own
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_32k")
    ap.add_argument("--cpu-rows", type=int, default=6144)
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--topk", type=int, default=1, choices=[1, 2],
                    help="groups per token; 2 runs the top-2 membership layer")
    ap.add_argument("--K", type=int, default=None, help="centroids (default: 4 with --topk 2)")
    ap.add_argument("--sinkhorn", type=int, default=0, help="time T Sinkhorn rounds instead")
    ap.add_argument("--backward", action="store_true", help="time the backward pass instead")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from learned_group_sparse_focus_gb300 import synth
    K = args.K if args.K is not None else (4 if args.topk == 2 else None)
    wl = synth.WORKLOADS[args.workload] if K is None else synth.workload(args.workload, K=K)
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, wl, world, rank)
    elif args.backward:
        run_ours_backward(args, wl, world, rank, local)
    elif args.sinkhorn > 0:
        run_ours_sinkhorn(args, wl, world, rank, local)
    elif args.topk > 1:
        run_ours_topk(args, wl, world, rank, local)
    else:
        run_ours(args, wl, world, rank, local)


if __name__ == "__main__":
    main()
