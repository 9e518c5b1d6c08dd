"""Benchmark: grouped-attention forward + backward on one GB300 (or N, one process per GPU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole hot path over one batch: packing is done once (it is input
construction), then every step runs pg_grouped_attn_fwd (RoPE + attention) and
pg_grouped_attn_bwd (RoPE, preprocess, dK/dV with the cross-response prefix reduction, dQ,
inverse RoPE) through the C ABI, on inputs already resident in HBM.  The metric is counted
grouped-attention TFLOP/s (14 * d * visible pairs * Hq per step), with tokens/s and the fraction of
the BF16 tensor peak beside it.  With N > 1 every rank runs its own independent batch (groups are
independent problems: weak scaling, no collective on the data path).

--impl reference times the CPU oracle (the repeated-prefix baseline, fp64) on bounded samples of
the same workload on the host cores; it prints one line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from shared_prefix_grouped_gb300 import _lib, api, flops, workloads  # noqa: E402

METRIC = "grouped-attn fwd+bwd TFLOP/s, tokens/s & % BF16 peak vs repeated-prefix (1 GB300)"
# The long-prefix GRPO shape: one group, P=16384, G=16 responses of U[256,1024] tokens, GQA 32/8.
DEFAULT_WORKLOAD = workloads.WORKLOADS[3].name
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_BYTES = 129 * 2 ** 20
# DRAM bytes (read + write) of one launch of the dominant kernel, from the committed ncu capture of
# this kernel on this workload.  Reported only while the kernel source still has the hash it had
# when the counters were taken, and only for that workload.
TRAFFIC = {"file": "shared_prefix_grouped_gb300/csrc/pg_attn_bwd_sm100.cu",
           "sha256": "22dedeb8e037a5aa23de43faf60910665b14d232aab36375afda24a21fe3b070",
           "workload": "bf16_gqa32x8_d128_p16384_g16_r256-1024", "bytes": 3043818496}


def key_major_flops(pairs: int, w, deterministic: bool) -> float:
    """FLOPs the key-major backward kernel executes: its five products (10·d per visible pair and
    query head) when it also forms dQ, four (8·d: S, dP, dV, dK) in the deterministic mode, where
    the query-major kernel forms dQ."""
    per = flops.attn_flops(pairs, w.heads_q, w.head_dim, "fwd")      # 4·d·pairs·Hq
    return 2.0 * per if deterministic else 2.5 * per


def measured_traffic(workload: str):
    import hashlib
    try:
        with open(os.path.join(ROOT, TRAFFIC["file"]), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    if sha != TRAFFIC["sha256"] or workload != TRAFFIC["workload"]:
        return None
    return TRAFFIC["bytes"]


def fp32_ffma_peak(peaks):
    """FP32 FMA peak of one GB300 (TFLOP/s): 152 SMs x 128 FP32 lanes x 2 FLOP per FMA x the
    maximum SM clock (MEASURED_PEAKS.json's sm_max_mhz, else 2070 MHz)."""
    return 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            data = json.load(open(path))
            flat = {}

            def walk(d):
                for k, v in d.items():
                    if isinstance(v, dict):
                        walk(v)
                    elif isinstance(v, (int, float)):
                        flat.setdefault(k, float(v))
            walk(data)
            if "bf16_tflops" in flat:
                return flat, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    QUERY = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        bus = None
        try:
            bus = torch.cuda.get_device_properties(self.device).pci_bus_id
        except Exception:
            pass
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        if bus is not None:
            mine = [r for r in rows if r[1].lower().endswith(str(bus).lower()[-12:])]
            rows = mine or rows
        elif len({r[0] for r in rows}) > 1:
            rows = [r for r in rows if r[0] == str(self.device)] or rows

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world, device):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(w, prob, l2_note):
    return {"workload": w.name, "groups": w.num_groups, "responses_per_group": w.group_size,
            "prefix_len": w.prefix_len, "suffix_lens": "fixed" if w.suffix_lens else
            f"uniform[{w.suffix_range[0]},{w.suffix_range[1]}] seed {w.seed}",
            "total_tokens": prob.total_tokens, "heads_q": w.heads_q, "heads_kv": w.heads_kv,
            "head_dim": w.head_dim, "rope_theta": w.rope_theta, "l2": l2_note}


# ------------------------------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------------

def oracle_sample(prob, head: int, n_resp: int):
    """Run the oracle on q-head `head`, group 0, its prefix and first n_resp responses.
    Returns (seconds, counted FLOPs of that grouped sample)."""
    from oracle import prefix_grouper_oracle as orc
    w = prob.workload
    lp = prob.prefix_lens[0]
    rs = prob.suffix_lens[:prob.group_sizes[0]][:n_resp]
    T = lp + sum(rs)
    # the sample is the group's first T packed rows (prefix, then responses in order)
    lay = orc.pack_layout([lp], [len(rs)], rs)
    sl = slice(0, T)
    kh = head // (w.heads_q // w.heads_kv)
    q = prob.q[sl, head:head + 1]
    k = prob.k[sl, kh:kh + 1]
    v = prob.v[sl, kh:kh + 1]
    do = prob.do[sl, head:head + 1]
    t0 = time.perf_counter()
    orc.repeated_prefix(lay, q, k, v, do, theta=w.rope_theta, check_prefix_copies=False)
    dt = time.perf_counter() - t0
    fl = flops.attn_flops(flops.group_pairs(lp, rs), 1, w.head_dim, "fwdbwd")
    return dt, fl


def cpu_baseline_leg(prob, budget_s=12.0, max_s=30.0):
    """The oracle on a bounded sample: group 0's prefix and its first n responses, one query head
    at a time, n sized from a one-response probe so the whole leg stays within ~10-30 s."""
    w = prob.workload
    G = prob.group_sizes[0]
    dt1, _ = oracle_sample(prob, 0, 1)
    n_resp = G if dt1 * G <= max_s else max(1, int(budget_s / dt1))
    total_t, total_f, heads = 0.0, 0.0, 0
    while True:            # query heads in turn, repeated for small workloads
        dt, fl = oracle_sample(prob, heads % w.heads_q, n_resp)
        total_t += dt
        total_f += fl
        heads += 1
        if total_t >= budget_s or total_t + dt > max_s:
            break
    return {"value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": torch.get_num_threads(),
            "kind": "oracle",
            "sample": f"group 0, prefix + {n_resp} of {G} responses, {heads} single-head runs "
                      f"(query heads in turn, {w.heads_q} in the workload), fp64 repeated-prefix "
                      f"forward+backward, {total_t:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    w = workloads.by_name(args.workload)
    prob = workloads.make_problem(w)
    G = prob.group_sizes[0]
    per_step_budget = max(1.0, 150.0 / (args.steps + args.warmup))
    dt, _ = oracle_sample(prob, 0, 1)
    n_resp = G
    if dt * G > per_step_budget:
        n_resp = max(1, int(per_step_budget / dt))
    times, fls = [], []
    for i in range(args.warmup + args.steps):
        dt, fl = oracle_sample(prob, i % w.heads_q, n_resp)
        if i >= args.warmup:
            times.append(dt)
            fls.append(fl)
    sec = sum(times) / len(times)
    value = sum(fls) / sum(times) / 1e12
    sample = (f"per step: group 0, prefix + {n_resp} of {G} responses, one query head "
              f"(cycling), fp64 repeated-prefix forward+backward")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, prob, "CPU run"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": torch.get_num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------------------------------------
# Our arm
# ------------------------------------------------------------------------------------------------

class Step:
    """Buffers and calls of one fwd+bwd step through the C ABI."""

    def __init__(self, prob, device, flags=0, layout=None):
        w = prob.workload
        self.w, self.flags, self.device = w, flags, device
        self.layout = layout if layout is not None else api.pack(
            prob.prefix_lens, prob.group_sizes, prob.suffix_lens, device)
        self.q, self.k, self.v, self.do = (t.to(device) for t in (prob.q, prob.k, prob.v, prob.do))
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((w.heads_q, prob.total_tokens), dtype=torch.float32, device=device)
        self.dq, self.dk, self.dv = (torch.empty_like(t) for t in (self.q, self.k, self.v))
        # One workspace for the step: the forward leaves the rotated q/k and the cos/sin table
        # in it for the backward (PG_FLAG_KEEP_ROTATED), as a training step saves them.
        self.flags = flags | _lib.PG_FLAG_KEEP_ROTATED
        opts = api.make_opts(w.rope_theta, 0.0, self.flags)
        self.ws = api._workspace(api.workspace_size(self.layout, self.q.dtype, w.heads_q,
                                                    w.heads_kv, w.head_dim, opts, 1), device)

    def __call__(self):
        w = self.w
        api.grouped_attn_fwd(self.layout, self.q, self.k, self.v, rope_theta=w.rope_theta,
                             flags=self.flags, out=self.o, lse=self.lse, workspace=self.ws)
        api.grouped_attn_bwd(self.layout, self.q, self.k, self.v, self.o, self.lse, self.do,
                             rope_theta=w.rope_theta, flags=self.flags, dq=self.dq, dk=self.dk,
                             dv=self.dv, workspace=self.ws)


def time_steps(step, n, device):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    s.record()
    for _ in range(n):
        step()
    e.record()
    torch.cuda.synchronize(device)
    return s.elapsed_time(e) / 1e3 / n


def run_ours(args):
    world, rank, local = dist_setup()
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    w = workloads.by_name(args.workload)
    prob = workloads.make_problem(w, seed=w.seed + rank)   # independent batch per rank
    flags = (_lib.PG_FLAG_SIMT if args.simt else 0) | \
        (_lib.PG_FLAG_DETERMINISTIC if args.deterministic else 0)
    step = Step(prob, device, flags)
    pairs = step.layout.pairs
    step_flops = flops.attn_flops(pairs, w.heads_q, w.head_dim, "fwdbwd")
    in_bytes = sum(t.numel() * t.element_size() for t in (step.q, step.k, step.v, step.do))
    l2_note = (f"inputs larger than L2 (q,k,v,dO = {in_bytes / 2**20:.0f} MiB > 129 MiB L2)"
               if in_bytes > L2_BYTES else "L2 flushed between steps")
    flush = None if in_bytes > L2_BYTES else torch.empty(2 * L2_BYTES, dtype=torch.uint8,
                                                         device=device)

    def one():
        if flush is not None:
            flush.zero_()
        step()

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize(device)

    # ---- timed region: K steps, per-launch events around the dominant kernel -----------------
    L = _lib.lib()
    dom_kernel = _lib.PG_KERNEL_BWD_DKDV
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:       # create the CUDA events
        a.record()
        b.record()
    prof = _lib.PgProfile(dom_kernel, 0, None, None, 0)
    sampler = ClockSampler(device.index)
    sampler.start()
    barrier(world, device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    L.pg_set_profile(prof)
    for i in range(args.steps):
        prof.ev_begin = ev[i][0].cuda_event
        prof.ev_end = ev[i][1].cuda_event
        one()
    L.pg_set_profile(None)
    end.record()
    barrier(world, device)
    clocks = sampler.stop()
    sec = start.elapsed_time(end) / 1e3 / args.steps
    sec = max_over_ranks(sec, world, device)
    dom_sec = sum(a.elapsed_time(b) for a, b in ev) / 1e3 / args.steps
    assert api.device_status() == 0, "a kernel reported an error"

    peaks, peak_src = load_peaks()
    value = step_flops * world / sec / 1e12
    # The fp32 (SIMT) path's key-major kernel forms dK and dV only (dQ is query-major there).
    simt = bool(args.simt) or w.dtype == "f32"
    dom_flops = key_major_flops(pairs, w, bool(args.deterministic) or simt)
    peak = peaks["bf16_tflops"]
    if simt:
        roof = {"bound": "alu", "kernel": "SIMT key-major dK/dV (fp32 FMA)",
                "peak": fp32_ffma_peak(peaks), "unit": "TFLOP/s",
                "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 FLOP x max SM clock"}
    else:
        roof = {"bound": "tensor",
                "kernel": "bwd key-major dK/dV" + ("" if args.deterministic else " + dQ"),
                "peak": peak, "unit": "TFLOP/s",
                "peak_source": f"bf16 dense burst, {peak_src}"}
    roof["achieved"] = dom_flops / dom_sec / 1e12
    roof["frac"] = roof["achieved"] / roof["peak"]
    # the capture is of the dQ-fusing kernel
    roof["traffic"] = None if (args.deterministic or simt) else measured_traffic(w.name)
    roof["traffic_unit"] = "bytes per launch (ncu dram read + write)"
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded N(0,1) Q/K/V/dO; no dataset)",
            "config": dict(workload_config(w, prob, l2_note),
                           deterministic_backward=bool(args.deterministic)),
            "tokens_per_s": prob.total_tokens * world / sec,
            "pct_bf16_peak": 100.0 * value / world / peak,
            "peak_source": peak_src,
            "roofline": roof,
            "clocks": clocks, "gpu_launches": int(prof.launches)}
    if rank == 0 and not args.skip_extras:
        line["e2e"] = e2e_leg(step, prob, device, args, step_flops, world)
        line["repeated_prefix"] = repeated_leg(prob, device, flags, sec, args, grouped=step)
        if world == 1:
            line["cpu_baseline"] = cpu_baseline_leg(prob)
    if rank == 0:
        print(json.dumps(line))


def e2e_leg(step, prob, device, args, step_flops, world):
    """Same metric through the public API with host buffers, every step: pinned H2D of q, k, v, dO,
    fwd+bwd, D2H of o, dq, dk, dv.  Steps are pipelined as a training loop would run them: step
    i+1's inputs go up on one copy stream and step i-1's gradients come down on another while the
    GPU computes step i (two device buffer sets); every step's copies are inside the timed
    region, which ends when the last step's results are on the host."""
    w = step.w
    host_in = [t.pin_memory() for t in (prob.q, prob.k, prob.v, prob.do)]
    host_out = [[torch.empty_like(t, device="cpu").pin_memory()
                 for t in (step.o, step.dq, step.dk, step.dv)] for _ in range(2)]
    sets = []
    for b in range(2):
        din = [step.q, step.k, step.v, step.do] if b == 0 else \
            [torch.empty_like(t) for t in (step.q, step.k, step.v, step.do)]
        dout = [step.o, step.lse, step.dq, step.dk, step.dv] if b == 0 else \
            [torch.empty_like(t) for t in (step.o, step.lse, step.dq, step.dk, step.dv)]
        ws = step.ws if b == 0 else torch.empty_like(step.ws)
        sets.append((din, dout, ws))
    comp = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in comp_done + d2h_done:
        e.record(comp)

    def run(n):
        for i in range(n):
            b = i % 2
            (q, k, v, do), (o, lse, dq, dk, dv), ws = sets[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(comp_done[b])          # step i-2 is done reading these inputs
                for d, h in zip((q, k, v, do), host_in):
                    d.copy_(h, non_blocking=True)
                h2d_done[b].record(s_in)
            comp.wait_event(h2d_done[b])
            comp.wait_event(d2h_done[b])               # step i-2's results have left these buffers
            api.grouped_attn_fwd(step.layout, q, k, v, rope_theta=w.rope_theta, flags=step.flags,
                                 out=o, lse=lse, workspace=ws)
            api.grouped_attn_bwd(step.layout, q, k, v, o, lse, do, rope_theta=w.rope_theta,
                                 flags=step.flags, dq=dq, dk=dk, dv=dv, workspace=ws)
            comp_done[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                for h, d in zip(host_out[b], (o, dq, dk, dv)):
                    h.copy_(d, non_blocking=True)
                d2h_done[b].record(s_out)
        comp.wait_event(d2h_done[0])
        comp.wait_event(d2h_done[1])

    run(max(3, args.warmup))
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    s_in.wait_event(start)
    run(args.steps)
    end.record(comp)
    torch.cuda.synchronize(device)
    sec = start.elapsed_time(end) / 1e3 / args.steps
    sec = max_over_ranks(sec, world, device)
    return {"value": step_flops * world / sec / 1e12, "unit": "TFLOP/s",
            "ms_per_step": sec * 1e3,
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in),
            "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out[0]),
            "pipelining": "H2D of step i+1 and D2H of step i-1 overlap step i (two buffer sets)"}


def repeated_leg(prob, device, flags, grouped_sec, args, grouped=None):
    """The same attention as the repeated-prefix baseline on this GPU: every [P; Ri] materialised
    as its own sequence and run through the same kernels, timed, and (given the grouped step)
    compared with the grouped outputs.

    Upstream gradients at prefix rows go into each group's first copy only (zero in the others),
    so the repeated layout's gradients, summed over copies for prefix rows, are the gradients of
    the packed function.  Mapped back: O / LSE rows from the copy that holds each packed row's
    upstream gradient (prefix rows from copy 0, response rows from their own copy), dQ / dK / dV
    summed over copies.  Errors are normwise (max|grouped - repeated| / max|repeated| per
    tensor)."""
    w = prob.workload
    lps, gss, rss, idx, keep = [], [], [], [], []
    s = 0
    g0 = 0
    for b, (lp, G) in enumerate(zip(prob.prefix_lens, prob.group_sizes)):
        seg0 = g0 + lp
        for i in range(max(G, 1)):
            r = prob.suffix_lens[s + i] if G else 0
            lps.append(lp)
            gss.append(1)
            rss.append(r)
            idx.append(torch.arange(g0, g0 + lp))
            idx.append(torch.arange(seg0, seg0 + r))
            keep.append(torch.full((lp,), i == 0, dtype=torch.bool))
            keep.append(torch.ones(r, dtype=torch.bool))
            seg0 += r
        g0 = seg0
        s += G
    idx, keep = torch.cat(idx), torch.cat(keep)
    do_rep = prob.do[idx] * keep[:, None, None].to(prob.do.dtype)
    rep = workloads.Problem(w, lps, gss, rss, prob.q[idx], prob.k[idx], prob.v[idx], do_rep)
    try:
        rstep = Step(rep, device, flags)
    except torch.cuda.OutOfMemoryError:
        return {"skipped": "out of memory"}
    for _ in range(2):
        rstep()
    n = max(3, min(args.steps, 10))
    sec = time_steps(rstep, n, device)
    rep_pairs = rstep.layout.pairs
    out = {"ms_per_step": sec * 1e3, "tokens": rep.total_tokens,
           # the repeated layout's tokens the grouped step covers per second
           "baseline_equivalent_tokens_per_s": rep.total_tokens / grouped_sec,
           "counted_tflops": flops.attn_flops(rep_pairs, w.heads_q, w.head_dim) / sec / 1e12,
           "speedup_grouped_vs_repeated": sec / grouped_sec,
           "pair_ratio_grouped_over_repeated":
               flops.total_pairs(prob.prefix_lens, prob.group_sizes, prob.suffix_lens) / rep_pairs}
    if grouped is not None:
        grouped()
        rstep()
        torch.cuda.synchronize(device)
        errs = equivalence_errors(grouped, rstep, idx.to(device), keep.to(device))
        out["normwise_err"] = errs
        out["max_normwise_err"] = max(errs.values())
        out["equivalence"] = ("grouped vs repeated-prefix on this GPU: O, LSE from the copy holding "
                              "each row's upstream gradient, dQ/dK/dV summed over copies")
    del rstep
    torch.cuda.empty_cache()
    return out


def equivalence_errors(g, r, idx, keep):
    """Normwise errors of the grouped step's outputs against the repeated step's, mapped back."""
    T = g.q.shape[0]
    sel = idx[keep]
    errs = {}
    for name in ("o", "lse", "dq", "dk", "dv"):
        x, y = getattr(g, name).float(), getattr(r, name).float()
        if name == "lse":
            ref = torch.empty_like(x)
            ref[:, sel] = y[:, keep]
        elif name == "o":
            ref = torch.empty_like(x)
            ref[sel] = y[keep]
        else:
            ref = torch.zeros((T,) + tuple(x.shape[1:]), dtype=torch.float32, device=x.device)
            ref.index_add_(0, idx, y)
        errs[name] = float((x - ref).abs().max() / ref.abs().max())
    return errs


SCORE_METRIC = ("grouped-attn responses-only forward (scoring) TFLOP/s & HBM GB/s "
                "vs the K/V-read roofline (1 GB300)")


def score_counts(prob):
    """Visible pairs of the response rows and the algorithmic bytes of one responses-only call:
    every K/V row a response can see read once per key/value head, the response rows of q read,
    o and lse written."""
    w = prob.workload
    pairs, kv_rows, s = 0, 0, 0
    for lp, G in zip(prob.prefix_lens, prob.group_sizes):
        rs = prob.suffix_lens[s:s + G]
        s += G
        pairs += sum(r * lp + r * (r + 1) // 2 for r in rs)
        kv_rows += (lp + sum(rs)) if sum(rs) else 0
    rows = sum(prob.suffix_lens)
    nbytes = (2 * kv_rows * w.heads_kv * w.head_dim * 2 + 2 * rows * w.heads_q * w.head_dim * 2
              + rows * w.heads_q * 4)
    return pairs, nbytes


def run_score_bench(args):
    """The forward-only scoring workload: response rows only, L2 flushed before every call and
    outside its events."""
    world, rank, local = dist_setup()
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    w = workloads.by_name(args.workload)
    prob = workloads.make_problem(w, seed=w.seed + rank)
    flags = _lib.PG_FLAG_RESPONSES_ONLY | (_lib.PG_FLAG_SIMT if args.simt else 0)
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, device)
    q, k, v = (t.to(device) for t in (prob.q, prob.k, prob.v))
    o = torch.empty_like(q)
    lse = torch.empty((w.heads_q, prob.total_tokens), dtype=torch.float32, device=device)
    opts = api.make_opts(w.rope_theta, 0.0, flags)
    ws = api._workspace(api.workspace_size(lay, q.dtype, w.heads_q, w.heads_kv, w.head_dim, opts,
                                           0), device)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)

    def call():
        api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta, flags=flags, out=o, lse=lse,
                             workspace=ws)

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(device)
    L = _lib.lib()
    n = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    step_ev = [(mk(), mk()) for _ in range(n)]
    kern_ev = [(mk(), mk()) for _ in range(n)]
    for a, b in kern_ev:      # create the CUDA events before their handles are passed on
        a.record()
        b.record()
    prof = _lib.PgProfile(_lib.PG_KERNEL_ATTN_FWD, 0, None, None, 0)
    sampler = ClockSampler(device.index)
    sampler.start()
    barrier(world, device)
    L.pg_set_profile(prof)
    for i in range(n):
        flush.zero_()
        prof.ev_begin = kern_ev[i][0].cuda_event
        prof.ev_end = kern_ev[i][1].cuda_event
        step_ev[i][0].record()
        call()
        step_ev[i][1].record()
    L.pg_set_profile(None)
    barrier(world, device)
    clocks = sampler.stop()
    assert api.device_status() == 0, "a kernel reported an error"
    sec = sum(a.elapsed_time(b) for a, b in step_ev) / 1e3 / n
    sec = max_over_ranks(sec, world, device)
    ksec = sum(a.elapsed_time(b) for a, b in kern_ev) / 1e3 / n
    pairs, nbytes = score_counts(prob)
    fl = flops.attn_flops(pairs, w.heads_q, w.head_dim, "fwd")
    peaks, peak_src = load_peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    value = fl * world / sec / 1e12
    line = {"metric": SCORE_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded N(0,1) Q/K/V; no dataset)",
            "config": dict(workload_config(w, prob, "L2 flushed before every call (outside the "
                                                     "events)"), responses_only=True,
                           response_tokens=sum(prob.suffix_lens)),
            "tokens_per_s": sum(prob.suffix_lens) * world / sec,
            "hbm_gbs_per_call": nbytes / sec / 1e9,
            "roofline": {"bound": "hbm", "kernel": "responses-only forward (key-split, GQA-packed)",
                         "achieved": nbytes / ksec / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": nbytes / ksec / 1e9 / hbm, "traffic": None,
                         "algorithmic_bytes": nbytes, "kernel_ms": ksec * 1e3,
                         "kernel_tflops": fl / ksec / 1e12,
                         "peak_source": f"HBM copy bandwidth, {peak_src}"},
            "clocks": clocks, "gpu_launches": int(prof.launches)}
    if rank == 0:
        print(json.dumps(line))


def run_tree_bench(args):
    """Nested prefixes (a shared context, user turns below it, responses below each turn):
    forward + backward through a pg_pack_tree layout."""
    world, rank, local = dist_setup()
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    w = workloads.tree_by_name(args.workload)
    prob = workloads.make_tree_problem(w, seed=w.seed + rank)
    flags = (_lib.PG_FLAG_SIMT if args.simt else 0) | \
        (_lib.PG_FLAG_DETERMINISTIC if args.deterministic else 0)
    step = Step(prob, device, flags, layout=api.pack_tree(w.parent, w.lens, device))
    pairs = step.layout.pairs
    step_flops = flops.attn_flops(pairs, w.heads_q, w.head_dim, "fwdbwd")
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    L = _lib.lib()
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk()) for _ in range(args.steps)]
    kev = [(mk(), mk()) for _ in range(args.steps)]
    for a, b in kev:
        a.record()
        b.record()
    prof = _lib.PgProfile(_lib.PG_KERNEL_BWD_DKDV, 0, None, None, 0)
    sampler = ClockSampler(device.index)
    sampler.start()
    barrier(world, device)
    L.pg_set_profile(prof)
    for i in range(args.steps):
        flush.zero_()
        prof.ev_begin, prof.ev_end = kev[i][0].cuda_event, kev[i][1].cuda_event
        ev[i][0].record()
        step()
        ev[i][1].record()
    L.pg_set_profile(None)
    barrier(world, device)
    clocks = sampler.stop()
    assert api.device_status() == 0, "a kernel reported an error"
    sec = sum(a.elapsed_time(b) for a, b in ev) / 1e3 / args.steps
    sec = max_over_ranks(sec, world, device)
    ksec = sum(a.elapsed_time(b) for a, b in kev) / 1e3 / args.steps
    peaks, peak_src = load_peaks()
    peak = peaks["bf16_tflops"]
    # repeated-prefix equivalent: every root-to-leaf path as its own sequence
    tl_paths, parent, lens = [], list(w.parent), list(w.lens)
    children = [[] for _ in parent]
    for i, p_ in enumerate(parent):
        if p_ >= 0:
            children[p_].append(i)
    rep_pairs = 0
    for i in range(len(parent)):
        if not children[i]:
            n, a = 0, i
            while a >= 0:
                n += lens[a]
                a = parent[a]
            rep_pairs += n * (n + 1) // 2
    line = {"metric": METRIC, "value": step_flops * world / sec / 1e12, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded N(0,1) Q/K/V/dO; no dataset)",
            "config": {"workload": w.name, "segments": len(parent), "max_depth":
                       int(step.layout.struct.max_depth), "total_tokens": prob.total_tokens,
                       "heads_q": w.heads_q, "heads_kv": w.heads_kv, "head_dim": w.head_dim,
                       "rope_theta": w.rope_theta, "deterministic_backward": bool(args.deterministic),
                       "l2": "L2 flushed before every step (outside the events)"},
            "tokens_per_s": prob.total_tokens * world / sec,
            "pct_bf16_peak": 100.0 * step_flops / sec / 1e12 / peak, "peak_source": peak_src,
            "pair_ratio_grouped_over_paths": pairs / rep_pairs,
            "roofline": {"bound": "tensor",
                         "kernel": "bwd key-major dK/dV" + ("" if args.deterministic else " + dQ"),
                         "achieved": key_major_flops(pairs, w, bool(args.deterministic)) / ksec / 1e12,
                         "peak": peak, "unit": "TFLOP/s", "traffic": None,
                         "peak_source": f"bf16 dense burst, {peak_src}"},
            "clocks": clocks, "gpu_launches": int(prof.launches)}
    line["roofline"]["frac"] = line["roofline"]["achieved"] / peak
    if rank == 0:
        print(json.dumps(line))


def run_layer_bench(args):
    """The decoder-layer workload: forward + backward of one layer over the packed groups."""
    from shared_prefix_grouped_gb300 import layer
    world, rank, local = dist_setup()
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    w = workloads.LayerWorkload()
    prob = workloads.make_layer_problem(w, seed=w.seed + rank)
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, device)
    W = [t.to(device) for t in (prob.w_qkv, prob.w_o, prob.w_gu, prob.w_d, prob.g1, prob.g2)]
    x, dy = prob.x.to(device), prob.dy.to(device)
    kw = dict(heads_q=w.heads_q, heads_kv=w.heads_kv, head_dim=w.head_dim,
              rope_theta=w.rope_theta, eps=w.rms_eps)

    def step():
        y, saved = layer.layer_fwd(lay, x, *W, **kw)
        layer.layer_bwd(lay, x, *W, saved, dy, **kw)

    for _ in range(args.warmup):
        step()
    L = _lib.lib()
    prof = _lib.PgProfile(0, 0, None, None, 0)
    sampler = ClockSampler(device.index)
    sampler.start()
    barrier(world, device)
    L.pg_set_profile(prof)
    sec = time_steps(step, args.steps, device)
    L.pg_set_profile(None)
    barrier(world, device)
    clocks = sampler.stop()
    sec = max_over_ranks(sec, world, device)
    T, H, I = prob.total_tokens, w.hidden, w.mlp
    qkv = (w.heads_q + 2 * w.heads_kv) * w.head_dim
    gemm = 2.0 * T * H * (qkv + w.heads_q * w.head_dim + 3 * I) * 3    # forward + 2x backward
    attn = flops.attn_flops(lay.pairs, w.heads_q, w.head_dim, "fwdbwd")
    peaks, peak_src = load_peaks()
    value = (gemm + attn) * world / sec / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) inputs, N(0,0.02) weights; no checkpoint)",
            "config": {"workload": w.name, "groups": w.num_groups,
                       "responses_per_group": w.group_size, "prefix_len": w.prefix_len,
                       "suffix_len": w.suffix_len, "total_tokens": T, "hidden": H, "mlp": I,
                       "heads_q": w.heads_q, "heads_kv": w.heads_kv, "head_dim": w.head_dim,
                       "rope_theta": w.rope_theta, "l2": "activations far larger than L2"},
            "tokens_per_s": T * world / sec, "pct_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "peak_source": peak_src, "counted_tflop": {"gemm": gemm / 1e12, "attention": attn / 1e12},
            "clocks": clocks, "gpu_launches": int(prof.launches)}
    if rank == 0:
        print(json.dumps(line))


# The decoder layer's GEMM shapes (tokens x out x in, B MN-major where the layer stores the weight
# that way), and a smaller gate/up case that a full ncu capture can hold.
GEMM_WORKLOADS = {
    "gemm_bf16_qkv_m32768_n6144_k4096": (32768, 6144, 4096, False),
    "gemm_bf16_gate_up_m32768_n28672_k4096": (32768, 28672, 4096, False),
    "gemm_bf16_down_m32768_n4096_k14336": (32768, 4096, 14336, False),
    "gemm_bf16_gate_up_m8192_n28672_k4096": (8192, 28672, 4096, False),
}

GEMM_METRIC = "bf16 tensor-core GEMM TFLOP/s (decoder-layer projection shapes, 1 GB300)"


def run_gemm_bench(args):
    """One of the decoder layer's projection GEMMs, C = A B^T in bf16 through pg_gemm_bf16."""
    world, rank, local = dist_setup()
    device = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    M, N, K, b_mn = GEMM_WORKLOADS[args.workload]
    gen = torch.Generator().manual_seed(1007 + rank)
    a = (torch.randn((M, K), generator=gen) * 0.5).to(torch.bfloat16).to(device)
    b = (torch.randn((K, N) if b_mn else (N, K), generator=gen) * 0.02).to(torch.bfloat16).to(device)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    in_bytes = (a.numel() + b.numel()) * 2
    flush = None if in_bytes > L2_BYTES else torch.empty(2 * L2_BYTES, dtype=torch.uint8,
                                                         device=device)

    def call():
        if flush is not None:
            flush.zero_()
        api.gemm_bf16(a, b, b_mn=b_mn, out_dtype=torch.bfloat16, out=c)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(device)
    L = _lib.lib()
    mk = lambda: torch.cuda.Event(enable_timing=True)
    kev = [(mk(), mk()) for _ in range(args.steps)]
    for e0, e1 in kev:
        e0.record()
        e1.record()
    prof = _lib.PgProfile(_lib.PG_KERNEL_GEMM, 0, None, None, 0)
    sampler = ClockSampler(device.index)
    sampler.start()
    barrier(world, device)
    start, end = mk(), mk()
    start.record()
    L.pg_set_profile(prof)
    for i in range(args.steps):
        prof.ev_begin, prof.ev_end = kev[i][0].cuda_event, kev[i][1].cuda_event
        call()
    L.pg_set_profile(None)
    end.record()
    barrier(world, device)
    clocks = sampler.stop()
    assert api.device_status() == 0, "a kernel reported an error"
    sec = start.elapsed_time(end) / 1e3 / args.steps
    sec = max_over_ranks(sec, world, device)
    ksec = sum(e0.elapsed_time(e1) for e0, e1 in kev) / 1e3 / args.steps
    fl = 2.0 * M * N * K
    peaks, peak_src = load_peaks()
    peak = peaks["bf16_tflops"]
    line = {"metric": GEMM_METRIC, "value": fl * world / sec / 1e12, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
            "config": {"workload": args.workload, "M": M, "N": N, "K": K, "b_mn_major": b_mn,
                       "out": "bf16", "l2": "inputs larger than L2" if flush is None else
                       "L2 flushed before every call"},
            "pct_bf16_peak": 100.0 * fl / sec / 1e12 / peak, "peak_source": peak_src,
            "roofline": {"bound": "tensor", "kernel": "pg_gemm_bf16 (tcgen05, 128x256 tiles)",
                         "achieved": fl / ksec / 1e12, "peak": peak, "unit": "TFLOP/s",
                         "frac": fl / ksec / 1e12 / peak, "traffic": None,
                         "peak_source": f"bf16 dense burst, {peak_src}"},
            "clocks": clocks, "gpu_launches": int(prof.launches)}
    if rank == 0:
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[w.name for w in workloads.WORKLOADS] + [workloads.LayerWorkload().name]
                    + [w.name for w in workloads.TREE_WORKLOADS] + list(GEMM_WORKLOADS))
    ap.add_argument("--simt", action="store_true", help="force the fp32 SIMT kernels")
    ap.add_argument("--deterministic", action="store_true",
                    help="bitwise-reproducible backward (query-major dQ kernel)")
    ap.add_argument("--skip-extras", action="store_true",
                    help="skip the e2e, repeated-prefix and CPU legs (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == workloads.LayerWorkload().name:
        run_layer_bench(args)
    elif args.workload in GEMM_WORKLOADS:
        run_gemm_bench(args)
    elif args.workload in [w.name for w in workloads.TREE_WORKLOADS]:
        run_tree_bench(args)
    elif workloads.by_name(args.workload).responses_only:
        run_score_bench(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
