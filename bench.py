#!/usr/bin/env python
"""Throughput of the speculative-decoding verification hot path on GB300.

One step is one pass of the whole hot path over one batch of the chain-b64
workload (B=64 sequences, gamma=7 drafts, V=151936, bf16 logits, T=0.6,
draft noise sigma in {0.25, 1, 4}): stochastic verification (row statistics,
accept decisions, residual/bonus sample), greedy verification of the same
drafts, and greedy tree verification of the same drafts laid out as a
chain-shaped tree.  The metric is verified rows per second, rows being
(sequence, position) pairs: 3 * B * (gamma+1) per step.

Own arm (default): inputs resident in HBM, CUDA-event timing of exactly K
steps after W warm-up steps, 4 rotating input copies (1.17 GB, > 4x the
129 MB L2) so every call reads cold logits.  Also reported: the end-to-end
rate through the public calls with host buffers (pinned H2D of every step's
inputs and D2H of its outputs inside the timed region, the next step's copy
double-buffered against the current step's kernels), the roofline of the dominant
kernel (the streaming row-statistics pass), clocks during the timed region and the
fp64 CPU oracle timed on the host cores.

Reference arm (--impl reference): the fp64 CPU oracle, as it stands, on a
bounded slice of the same workload per step, timed on the host cores.

Multi-GPU (torchrun, one process per GPU): every rank verifies its own
batch (weak scaling, no collective on the data path); the slowest rank's
time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verified rows/s & achieved HBM GB/s (fraction of GB300 roofline) at V=151936"
UNIT = "rows/s"
ROTATE = 4
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def rank_seed(workload_seed, rank):
    """Each replica verifies its own batch: rank r draws from seed + 1000 r."""
    return workload_seed + 1000 * rank


def max_over_ranks(v, world, device=None):
    """The largest per-rank value (the slowest replica's time) over the group."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_step, steps, ms_max):
    """Whole-job throughput: the units all replicas processed over the slowest
    replica's time (every replica runs the same number of steps)."""
    return world * units_per_step * steps / (ms_max * 1e-3)


def chain_tree(x):
    """The batch's drafts as a chain-shaped draft tree: node 0 is the root,
    node i+1 carries draft x_i and hangs under node i."""
    B, g = x.draft_tokens.shape
    par = np.tile(np.arange(-1, g, dtype=np.int32), (B, 1))
    tok = np.concatenate([np.full((B, 1), -1, np.int32), x.draft_tokens], axis=1)
    return np.ascontiguousarray(tok), np.ascontiguousarray(par)


def step_accounting(x):
    elt = 2 if x.dtype == "bf16" else 4
    rows_chain = x.B * (x.gamma + 1)
    bytes_stats = x.B * (2 * x.gamma + 1) * x.V * elt
    bytes_greedy = x.B * (x.gamma + 1) * x.V * elt
    return {
        "rows": 3 * rows_chain,
        "bytes_stats": bytes_stats,
        "bytes_step": bytes_stats + 2 * bytes_greedy,
    }


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = ("sv_common.cuh", "sv_internal.h", "sv_tma.cuh", "sv_decide.cuh", "sv_stream.cuh")


def kernel_source_hash(csrc=None):
    """Hash of the code that defines the row-statistics stream kernel (its sources with
    comments and blank lines removed, so that an edit of comments alone keeps it); ncu
    traffic figures recorded under profiles/ are only reported while it matches."""
    h = hashlib.sha256()
    if csrc is None:
        csrc = os.path.join(ROOT, "speculative_decoding_verification_59_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """dram bytes per launch of the row-statistics stream kernel from the committed ncu
    summary (profiles/stats_traffic.txt: key=value lines), or None."""
    p = os.path.join(ROOT, "profiles", "stats_traffic.txt")
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if "=" in line and not line.lstrip().startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_hash") != kernel_source_hash() or kv.get("workload") != workload:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the benchmark runs."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                self.samples.append((time.time(), parts))

    def wait_first(self, timeout_s=5.0):
        """Blocks (at most timeout_s) until nvidia-smi has delivered a sample, so
        that even a timed region of a few milliseconds falls inside the record."""
        t_end = time.time() + timeout_s
        while self.proc is not None and not self.samples and time.time() < t_end:
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1, run=None):
        """Clocks over the timed region [t0, t1] (with 0.15 s of slack).  A
        region shorter than the 100 ms sampling period may hold no sample; the
        samples of the whole GPU run `run` = (start, end) then stand in."""
        win = [p for (t, p) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        window = "timed region"
        if not win and run is not None:
            win = [p for (t, p) in self.samples if run[0] <= t <= run[1]]
            window = "whole GPU run (the timed region is shorter than the sampling period)"
        if not win and self.samples:                       # nearest sample
            mid = 0.5 * (t0 + t1)
            win = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
            window = "nearest sample"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(win[0][3]), "reasons": reasons, "samples": len(win),
                "window": window}


# ------------------------------------------------------------------ own arm
def run_own(args):
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_59_gb300 as sv
    from speculative_decoding_verification_59_gb300 import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    x = W.make_chain(args.workload, seed=rank_seed(W.WORKLOADS[args.workload].seed, rank))
    ttok, tpar = chain_tree(x)
    acct = step_accounting(x)
    B, g, V = x.B, x.gamma, x.V
    tdt = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    dcode = sv.SPEC_DTYPE_BF16 if x.dtype == "bf16" else sv.SPEC_DTYPE_F32

    host = {
        "zt": torch.from_numpy(x.target).to(tdt).pin_memory(),
        "zd": torch.from_numpy(x.draft).to(tdt).pin_memory(),
        "x": torch.from_numpy(x.draft_tokens).pin_memory(),
        "u": torch.from_numpy(x.uniforms).pin_memory(),
        "tt": torch.from_numpy(ttok).pin_memory(),
        "tp": torch.from_numpy(tpar).pin_memory(),
    }
    rot = args.rotate
    copies = [{k: v.to(dev) for k, v in host.items()} for _ in range(rot)]
    out = {
        "s_tok": torch.empty((B, g + 1), dtype=torch.int32, device=dev),
        "s_acc": torch.empty((B,), dtype=torch.int32, device=dev),
        "g_tok": torch.empty((B, g + 1), dtype=torch.int32, device=dev),
        "g_acc": torch.empty((B,), dtype=torch.int32, device=dev),
        "t_nodes": torch.empty((B, g + 1), dtype=torch.int32, device=dev),
        "t_tok": torch.empty((B, g + 1), dtype=torch.int32, device=dev),
        "t_acc": torch.empty((B,), dtype=torch.int32, device=dev),
    }
    ws = sv.Workspace(dev)
    wp, wb = ws.get(B, g + 1, V)       # the chain-shaped tree has g+1 nodes
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    P = lambda t: t.data_ptr()  # noqa: E731

    def check(st, what):
        if st != sv.SPEC_OK:
            raise sv.SpecVerifyError(st, what)

    def calls(s, ev=None):
        c0, c1, c2 = copies[s % rot], copies[(s + 1) % rot], copies[(s + 2) % rot]
        if ev is None:
            check(sv.spec_verify_sample(P(c0["zt"]), P(c0["zd"]), dcode, P(c0["x"]), P(c0["u"]),
                                        x.T, B, g, V, P(out["s_tok"]), P(out["s_acc"]), None, wp,
                                        wb, sh), "sample")
        else:
            # the same work as its two halves, with events around the stats stream
            ev[0].record(stream)
            check(sv.spec_verify_sample_stats(P(c0["zt"]), P(c0["zd"]), dcode, x.T, B, g, V, wp,
                                              wb, sh), "stats")
            ev[1].record(stream)
            check(sv.spec_verify_sample_finish(P(c0["zt"]), P(c0["zd"]), dcode, P(c0["x"]),
                                               P(c0["u"]), x.T, B, g, V, P(out["s_tok"]),
                                               P(out["s_acc"]), None, wp, wb, sh), "finish")
        check(sv.spec_verify_greedy(P(c1["zt"]), dcode, P(c1["x"]), B, g, V, P(out["g_tok"]),
                                    P(out["g_acc"]), wp, wb, sh), "greedy")
        check(sv.spec_verify_tree_greedy(P(c2["zt"]), dcode, P(c2["tt"]), P(c2["tp"]), B, g + 1, V,
                                         P(out["t_nodes"]), P(out["t_tok"]), P(out["t_acc"]), wp,
                                         wb, sh), "tree")

    def barrier():
        if world > 1:
            dist.barrier(device_ids=[local])
        torch.cuda.synchronize(dev)

    gpu_id = local
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    clocks = ClockSampler(gpu_id)
    clocks.wait_first()
    t_run0 = time.time()

    # warm-up (also settles clocks)
    for s in range(args.warmup):
        calls(s)
    barrier()

    # ---- device-resident timed region: K steps back to back with no event
    # between the calls (an event recorded between two kernels ends the
    # programmatic overlap of the second with the first, ~8 us per step here)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_wall0 = time.time()
    e0.record(stream)
    for s in range(K):
        calls(s)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world, dev)
    barrier()
    # ---- the same K steps once more, with CUDA events on the launching
    # stream around every launch of the dominant kernel (the stats stream):
    # its mean launch duration for the roofline
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for s in range(K):
        calls(s, evs[s])
    torch.cuda.synchronize(dev)
    t_wall2 = time.time()
    stats_ms = [a.elapsed_time(b) for a, b in evs]
    # ---- context: the stats kernel alone, K back-to-back launches between two
    # events (no event between launches, so each overlaps the previous one's tail)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for s in range(K):
        c0 = copies[s % rot]
        check(sv.spec_verify_sample_stats(P(c0["zt"]), P(c0["zd"]), dcode, x.T, B, g, V, wp, wb,
                                          sh), "stats")
    a1.record(stream)
    torch.cuda.synchronize(dev)
    stats_alone_ms = a0.elapsed_time(a1) / K
    barrier()
    # ---- each call of the step on its own
    n_call = max(50, min(K, 500))
    per_call = time_per_call(sv, torch, copies, x, stream, sh, dev, n_call, world, max_over_ranks)

    # outputs of the last step, for tau
    s_acc = out["s_acc"].cpu().numpy()
    g_acc = out["g_acc"].cpu().numpy()
    tau_sample = float((s_acc + 1).mean())
    tau_greedy = float((g_acc + 1).mean())

    # ---- end-to-end through the public calls with host buffers.  Every step
    # copies its inputs from pinned host memory and reads its outputs back;
    # two staging buffers let step i+1's copy (on a copy stream) overlap step
    # i's kernels.
    Ke = args.steps if args.e2e_steps is None else args.e2e_steps
    stages = [copies[0], copies[1] if len(copies) > 1 else
              {k: torch.empty_like(v) for k, v in copies[0].items()}]
    copy_stream = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    h_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items()}
    lp = torch.empty((B, g, 2), dtype=torch.float32, device=dev)
    h_lp = torch.empty((B, g, 2), dtype=torch.float32).pin_memory()
    bi = sum(v.numel() * v.element_size() for v in host.values())
    bo = sum(v.numel() * v.element_size() for v in out.values()) + lp.numel() * 4

    def e2e_step(i, start=None):
        stage = stages[i % 2]
        with torch.cuda.stream(copy_stream):
            if start is not None:
                copy_stream.wait_event(start)
            copy_stream.wait_event(ev_free[i % 2])        # the step that last read this buffer
            for k, v in host.items():
                stage[k].copy_(v, non_blocking=True)
            ev_in[i % 2].record(copy_stream)
        stream.wait_event(ev_in[i % 2])
        check(sv.spec_verify_sample(P(stage["zt"]), P(stage["zd"]), dcode, P(stage["x"]),
                                    P(stage["u"]), x.T, B, g, V, P(out["s_tok"]), P(out["s_acc"]),
                                    P(lp), wp, wb, sh), "sample")
        check(sv.spec_verify_greedy(P(stage["zt"]), dcode, P(stage["x"]), B, g, V, P(out["g_tok"]),
                                    P(out["g_acc"]), wp, wb, sh), "greedy")
        check(sv.spec_verify_tree_greedy(P(stage["zt"]), dcode, P(stage["tt"]), P(stage["tp"]), B,
                                         g + 1, V, P(out["t_nodes"]), P(out["t_tok"]),
                                         P(out["t_acc"]), wp, wb, sh), "tree")
        ev_free[i % 2].record(stream)
        for k, v in out.items():
            h_out[k].copy_(v, non_blocking=True)
        h_lp.copy_(lp, non_blocking=True)

    for i in range(min(3, Ke)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(Ke):
        e2e_step(i, f0 if i == 0 else None)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev)
    # the box's own pinned host-to-device rate for the same input set, one
    # cudaMemcpyAsync per tensor on the copy stream, for reading e2e against
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nrep = 5
    with torch.cuda.stream(copy_stream):
        h0.record(copy_stream)
        for _ in range(nrep):
            for k, v in host.items():
                stages[0][k].copy_(v, non_blocking=True)
        h1.record(copy_stream)
    torch.cuda.synchronize(dev)
    h2d_ref_gbs = nrep * bi / (h0.elapsed_time(h1) * 1e-3) / 1e9
    # ---- next-step paths, timed on their own (not part of the step above)
    nx = max(50, min(K, 500))
    extra = {"topk_k4": time_topk(sv, torch, copies, x, stream, sh, nx, max_over_ranks, world, dev),
             "lazy_sample": time_lazy(sv, torch, copies, x, stream, sh, nx, max_over_ranks, world,
                                      dev, acct),
             "ngram_b64": time_ngram(sv, torch, W, stream, sh, nx, max_over_ranks, world, dev,
                                     rank),
             "cosine_b64": time_cosine(sv, torch, W, stream, sh, nx, max_over_ranks, world, dev,
                                       rank),
             "tree_b32": time_tree(sv, torch, W, stream, sh, nx, max_over_ranks, world, dev, rank)}
    # ---- the other chain workloads, sample and greedy calls on their own
    configs = {}
    if not args.no_configs:
        for name in ("chain-small", "chain-b8", "chain-b256"):
            if name != args.workload:
                configs[name] = time_config(sv, torch, W, name, stream, sh, dev, nx, world,
                                            max_over_ranks, rank)
    t_run1 = time.time()
    clk = clocks.summary(t_wall0, t_wall2, run=(t_run0, t_run1))
    clocks.stop()

    # ---- CPU baseline: the fp64 oracle on host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_timing(x, ttok, tpar, budget_s=args.cpu_budget)
        one = oracle_timing(x, ttok, tpar, budget_s=0.5 * args.cpu_budget, threads=1)
        cpu["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}

    if rank == 0:
        peak, peak_src = measured_peaks()
        stats_mean_ms = statistics.mean(stats_ms)
        achieved = acct["bytes_stats"] / (stats_mean_ms * 1e-3) / 1e9
        traffic = recorded_traffic(args.workload)
        value = job_rate(world, acct["rows"], K, ms_max)
        line = {
            "metric": METRIC,
            "value": value,
            "unit": UNIT,
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": ms_max / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded generator, chain-b64 recipe)",
            "config": {
                "workload": args.workload,
                "B": B, "gamma": g, "V": V, "logits": x.dtype, "temperature": x.T,
                "step": "spec_verify_sample + spec_verify_greedy + spec_verify_tree_greedy "
                        "(chain-shaped tree), each on its own rotating input copy; value counts "
                        "the rows of all three modes, 3 B (gamma+1) per step (per_call has each "
                        "mode on its own)",
                "l2": f"{rot} rotating input copies of {acct['bytes_stats'] / 1e6:.1f} MB "
                      f"({rot * acct['bytes_stats'] / 129e6:.1f}x the 129 MB L2 in all)",
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            },
            "hbm_gbs_step": job_rate(world, acct["bytes_step"], K, ms_max) / 1e9,
            "rounds_per_s": job_rate(world, x.B, K, ms_max),
            "tau": {"sample": tau_sample, "greedy": tau_greedy},
            "roofline": {
                "kernel": "ring_sample_kernel<bf16> (spec_verify_sample_stats)",
                "bound": "hbm",
                "achieved": achieved,
                "peak": peak,
                "peak_source": f"{peak_src} hbm copy rate",
                "unit": "GB/s",
                "frac": achieved / peak,
                "frac_of_8tbs_nominal": achieved / 8000.0,
                "traffic": traffic,
                "algorithmic_bytes_per_launch": acct["bytes_stats"],
                "launch_ms_mean": stats_mean_ms,
                "timing": "CUDA events around each of the K stats launches of a second pass "
                          "over the timed steps (the first pass, which gives value, records "
                          "no events between calls)",
                "alone": {"launch_ms_mean": stats_alone_ms,
                          "frac": acct["bytes_stats"] / (stats_alone_ms * 1e-3) / 1e9 / peak,
                          "how": "K back-to-back stats launches between two events"},
            },
            "e2e": {
                "value": job_rate(world, acct["rows"], Ke, e2e_ms),
                "unit": UNIT,
                "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo,
                "steps": Ke,
                "pipelining": "double-buffered: step i+1's host-to-device copy runs on a copy "
                              "stream while step i's kernels run",
                "h2d_reference_gbs": h2d_ref_gbs,
                "h2d_reference": "the same pinned input set copied alone, one cudaMemcpyAsync "
                                 "per tensor, 5 repetitions between CUDA events",
                "h2d_gbs_implied": bi * Ke / (e2e_ms * 1e-3) / 1e9,
            },
            "gpu_launches": (sample_launches(x) + 4) * K,
            "clocks": clk,
            "cpu_baseline": cpu,
            "per_call": per_call,
            "configs": configs,
            "extra_paths": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def time_loop(torch, stream, dev, call, n, warm=3):
    """Mean milliseconds per call of n back-to-back calls call(0..n-1) between
    two CUDA events on the launching stream (no event between the calls),
    after `warm` untimed calls."""
    for s in range(warm):
        call(s)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(n):
        call(s)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / n


def call_entry(ms, rows, nbytes, peak, peak_src, launches, roofline=True):
    d = {"us_per_call": 1e3 * ms, "rows_per_s": rows / (ms * 1e-3),
         "algorithmic_bytes_per_call": nbytes, "gpu_launches_per_call": launches}
    if roofline:
        gbs = nbytes / (ms * 1e-3) / 1e9
        d["hbm"] = {"achieved_gbs": gbs, "peak_gbs": peak, "peak_source": peak_src,
                    "frac": gbs / peak, "frac_of_8tbs_nominal": gbs / 8000.0}
    else:
        d["hbm"] = None
        d["note"] = "latency-bound (tens of KB per call): no roofline claim"
    return d


def sample_launches(x):
    """Kernel launches of one spec_verify_sample call: the statistics stream,
    the decisions and the final pass (with the search)."""
    return 3


def time_per_call(sv, torch, copies, x, stream, sh, dev, n, world, max_over_ranks):
    """Each of the step's three calls on its own: n back-to-back calls over the
    rotating input copies, CUDA events on the launching stream."""
    B, g, V = x.B, x.gamma, x.V
    dcode = sv.SPEC_DTYPE_BF16 if x.dtype == "bf16" else sv.SPEC_DTYPE_F32
    elt = 2 if x.dtype == "bf16" else 4
    rot = len(copies)
    ws = sv.Workspace(dev)
    wp, wb = ws.get(B, g + 1, V)
    tok = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    nodes = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    P = lambda t: t.data_ptr()  # noqa: E731

    def check(st, what):
        if st != sv.SPEC_OK:
            raise sv.SpecVerifyError(st, what)

    def sample(s):
        c = copies[s % rot]
        check(sv.spec_verify_sample(P(c["zt"]), P(c["zd"]), dcode, P(c["x"]), P(c["u"]), x.T, B,
                                    g, V, P(tok), P(acc), None, wp, wb, sh), "sample")

    def greedy(s):
        c = copies[s % rot]
        check(sv.spec_verify_greedy(P(c["zt"]), dcode, P(c["x"]), B, g, V, P(tok), P(acc), wp, wb,
                                    sh), "greedy")

    def tree(s):
        c = copies[s % rot]
        check(sv.spec_verify_tree_greedy(P(c["zt"]), dcode, P(c["tt"]), P(c["tp"]), B, g + 1, V,
                                         P(nodes), P(tok), P(acc), wp, wb, sh), "tree")

    peak, src = measured_peaks()
    rows = world * B * (g + 1)
    b_s = B * (2 * g + 1) * V * elt
    b_g = B * (g + 1) * V * elt
    out = {}
    for name, fn, nb, launches in (("sample", sample, b_s, sample_launches(x)),
                                   ("greedy", greedy, b_g, 2), ("tree", tree, b_g, 2)):
        ms = max_over_ranks(time_loop(torch, stream, dev, fn, n), world, dev)
        out[name] = call_entry(ms, rows, world * nb, peak, src, launches)
    out["how"] = (f"{n} back-to-back calls of each entry point over {rot} rotating input copies, "
                  "CUDA events on the launching stream; rows = B (gamma+1) per call")
    return out


def time_config(sv, torch, W, name, stream, sh, dev, n, world, max_over_ranks, rank):
    """spec_verify_sample and spec_verify_greedy on another chain workload, each
    timed on its own over rotating input copies (together more than 4x the
    129 MB L2 where the copies fit in a few GB; chain-small's 36 KB stay in L2)."""
    x = W.make_chain(name, seed=rank_seed(W.WORKLOADS[name].seed, rank))
    B, g, V = x.B, x.gamma, x.V
    tdt = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    dcode = sv.SPEC_DTYPE_BF16 if x.dtype == "bf16" else sv.SPEC_DTYPE_F32
    elt = 2 if x.dtype == "bf16" else 4
    b_s = B * (2 * g + 1) * V * elt
    b_g = B * (g + 1) * V * elt
    rot = max(1, min(8, -(-4 * 129_000_000 // b_s))) if b_s > 1_000_000 else 1
    zt = torch.from_numpy(x.target).to(tdt)
    zd = torch.from_numpy(x.draft).to(tdt)
    copies = [{"zt": zt.to(dev), "zd": zd.to(dev)} for _ in range(rot)]
    xd = torch.from_numpy(x.draft_tokens).to(dev)
    ud = torch.from_numpy(x.uniforms).to(dev)
    tok = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sv.Workspace(dev)
    wp, wb = ws.get(B, g, V)

    def check(st, what):
        if st != sv.SPEC_OK:
            raise sv.SpecVerifyError(st, what)

    def sample(s):
        c = copies[s % rot]
        check(sv.spec_verify_sample(c["zt"].data_ptr(), c["zd"].data_ptr(), dcode, xd.data_ptr(),
                                    ud.data_ptr(), x.T, B, g, V, tok.data_ptr(), acc.data_ptr(),
                                    None, wp, wb, sh), "sample")

    def greedy(s):
        c = copies[s % rot]
        check(sv.spec_verify_greedy(c["zt"].data_ptr(), dcode, xd.data_ptr(), B, g, V,
                                    tok.data_ptr(), acc.data_ptr(), wp, wb, sh), "greedy")

    peak, src = measured_peaks()
    big = b_s > 1_000_000
    rows = world * B * (g + 1)
    res = {"B": B, "gamma": g, "V": V, "logits": x.dtype, "temperature": x.T}
    for mode, fn, nb, launches in (("sample", sample, b_s, sample_launches(x)),
                                   ("greedy", greedy, b_g, 2)):
        ms = max_over_ranks(time_loop(torch, stream, dev, fn, n), world, dev)
        res[mode] = call_entry(ms, rows, world * nb, peak, src, launches, roofline=big)
    res["l2"] = (f"{rot} rotating input copies of {b_s / 1e6:.1f} MB" if big else
                 "one input copy (L2-resident: the workload is smaller than the L2)")
    res["calls"] = n
    del copies
    torch.cuda.empty_cache()
    return res


def time_topk(sv, torch, copies, x, stream, sh, steps, max_over_ranks, world, dev):
    """Top-4 branch tokens (AdaPLD's TopKNextTokens minus the main path's first
    token) over every target row of the batch, each row excluding the draft
    token drafted at its position (the bonus row excludes nothing); one call
    per step on rotating input copies, CUDA events on the launching stream."""
    B, g, V = x.B, x.gamma, x.V
    rows = B * (g + 1)
    dcode = sv.SPEC_DTYPE_BF16 if x.dtype == "bf16" else sv.SPEC_DTYPE_F32
    ex = np.concatenate([x.draft_tokens, np.full((B, 1), -1, np.int32)], axis=1)
    exd = torch.from_numpy(np.ascontiguousarray(ex)).to(dev)
    idx = torch.empty((rows, 4), dtype=torch.int32, device=dev)
    ws = sv.Workspace(dev)
    wp, wb = ws.get_bytes(sv.spec_topk_workspace_size(rows, V, 4))

    def call(c):
        st = sv.spec_topk_exclude(c["zt"].data_ptr(), dcode, rows, V, 4, exd.data_ptr(),
                                  idx.data_ptr(), None, wp, wb, sh)
        if st != sv.SPEC_OK:
            raise sv.SpecVerifyError(st, "topk")

    for s in range(5):
        call(copies[s % len(copies)])
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(steps):
        call(copies[s % len(copies)])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
    elt = 2 if x.dtype == "bf16" else 4
    nbytes = rows * V * elt
    peak, src = measured_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"what": "top-4 of every target row, excluding the row's draft token",
            "rows": rows, "V": V, "calls": steps, "ms_per_call": ms,
            "rows_per_s": world * rows / (ms * 1e-3),
            "hbm": {"achieved_gbs": gbs, "peak_gbs": peak, "peak_source": src,
                    "frac": gbs / peak, "algorithmic_bytes_per_call": nbytes},
            "gpu_launches_per_call": 2}


def time_ngram(sv, torch, W, stream, sh, steps, max_over_ranks, world, dev, rank):
    """Lexical (n-gram) retrieval over the ngram-b64 token streams (64
    contexts of 32K..64K tokens, query w=3, draft L=7): every token is read
    once, 4 bytes each.  Eight input copies of 16.8 MB rotate (134 MB, more
    than the 129 MB L2)."""
    g = W.make_ngram("ngram-b64", seed=W.WORKLOADS["ngram-b64"].seed + 1000 * rank)
    B, n_max = g.tokens.shape
    toks = [torch.from_numpy(g.tokens).to(dev) for _ in range(8)]
    lens = torch.from_numpy(g.lengths).to(dev)
    cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    mat = torch.empty((B, g.max_matches), dtype=torch.int32, device=dev)
    dr = torch.empty((B, g.L), dtype=torch.int32, device=dev)
    ws = sv.Workspace(dev)
    wp, wb = ws.get_bytes(sv.spec_ngram_workspace_size(B, n_max, g.max_matches))

    def call(t):
        st = sv.spec_ngram_retrieve(t.data_ptr(), lens.data_ptr(), B, n_max, g.w, g.L,
                                    g.max_matches, cnt.data_ptr(), mat.data_ptr(), dr.data_ptr(),
                                    wp, wb, sh)
        if st != sv.SPEC_OK:
            raise sv.SpecVerifyError(st, "ngram")

    for s in range(5):
        call(toks[s % 8])
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(steps):
        call(toks[s % 8])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
    ntok = int(g.lengths.astype(np.int64).sum())
    peak, src = measured_peaks()
    gbs = 4 * ntok / (ms * 1e-3) / 1e9
    return {"what": "n-gram retrieval, 64 token streams of 32K..64K tokens, w=3, L=7",
            "ms_per_call": ms, "calls": steps, "tokens": ntok,
            "tokens_per_s": world * ntok / (ms * 1e-3),
            "bytes_per_call": 4 * ntok, "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / peak,
            "l2": "8 rotating input copies, 134 MB in all (> L2)", "gpu_launches_per_call": 2}


def time_cosine(sv, torch, W, stream, sh, steps, max_over_ranks, world, dev, rank):
    """Semantic fallback over the cosine-b64 windows (64 sequences x 240
    hidden states x 4096, bf16, delta 4): every window row is read once.
    Two input copies of 126 MB rotate (252 MB, more than the 129 MB L2)."""
    c = W.make_cosine("cosine-b64", seed=W.WORKLOADS["cosine-b64"].seed + 1000 * rank)
    B, Wn, d = c.hidden.shape
    hs = [torch.from_numpy(c.hidden).to(dev).to(torch.bfloat16) for _ in range(2)]
    qs = torch.from_numpy(c.query).to(dev).to(torch.bfloat16)
    pos = torch.from_numpy(c.positions).to(dev)
    idx = torch.empty((B, c.delta), dtype=torch.int32, device=dev)
    out_pos = torch.empty((B, c.delta), dtype=torch.int32, device=dev)
    ws = sv.Workspace(dev)
    wp, wb = ws.get_bytes(sv.spec_cosine_workspace_size(B, Wn))

    def call(h):
        st = sv.spec_cosine_topk(h.data_ptr(), qs.data_ptr(), sv.SPEC_DTYPE_BF16, B, Wn, d, c.delta,
                                 pos.data_ptr(), idx.data_ptr(), out_pos.data_ptr(), None, wp, wb, sh)
        if st != sv.SPEC_OK:
            raise sv.SpecVerifyError(st, "cosine")

    for s in range(5):
        call(hs[s % 2])
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(steps):
        call(hs[s % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
    nbytes = B * Wn * d * 2 + B * d * 2
    peak, src = measured_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    del hs
    return {"what": "cosine top-4 over 64 windows of 240 x 4096 bf16 hidden states",
            "ms_per_call": ms, "calls": steps, "rows_per_s": world * B * Wn / (ms * 1e-3),
            "bytes_per_call": nbytes, "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / peak,
            "peak_source": src, "l2": "2 rotating input copies, 252 MB in all (> L2)",
            "gpu_launches_per_call": 2}


def time_tree(sv, torch, W, stream, sh, steps, max_over_ranks, world, dev, rank):
    """Greedy draft-tree verification on the tree-b32 workload (32 sequences,
    36-node trees: root, a 7-node main chain and 4 single-node branches at
    each of its depths, V = 151936, bf16): every node's target row is read
    once.  Two input copies of 350 MB rotate (700 MB, more than the L2)."""
    t = W.make_tree("tree-b32", seed=W.WORKLOADS["tree-b32"].seed + 1000 * rank)
    B, N, V = t.B, t.N, t.V
    zs = [torch.from_numpy(t.target).to(dev).to(torch.bfloat16) for _ in range(2)]
    tok = torch.from_numpy(t.node_tokens).to(dev)
    par = torch.from_numpy(t.parents).to(dev)
    nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    otok = torch.empty((B, N), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sv.Workspace(dev)
    wp, wb = ws.get(B, N, V)

    def call(z):
        st = sv.spec_verify_tree_greedy(z.data_ptr(), sv.SPEC_DTYPE_BF16, tok.data_ptr(),
                                        par.data_ptr(), B, N, V, nodes.data_ptr(),
                                        otok.data_ptr(), acc.data_ptr(), wp, wb, sh)
        if st != sv.SPEC_OK:
            raise sv.SpecVerifyError(st, "tree")

    for s in range(5):
        call(zs[s % 2])
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(steps):
        call(zs[s % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
    nbytes = B * N * V * 2
    peak, src = measured_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    mean_acc = float(acc.float().mean().item())
    del zs
    return {"what": "greedy tree verification, 32 trees of 36 nodes (main chain of 7, "
                    "4 branches per depth), V = 151936 bf16",
            "ms_per_call": ms, "calls": steps, "rows_per_s": world * B * N / (ms * 1e-3),
            "bytes_per_call": nbytes, "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / peak,
            "peak_source": src, "mean_path_length": mean_acc,
            "l2": "2 rotating input copies, 700 MB in all (> L2)", "gpu_launches_per_call": 2}


def time_lazy(sv, torch, copies, x, stream, sh, steps, max_over_ranks, world, dev, acct):
    """spec_verify_sample_lazy on the step's inputs: the same tokens as the
    full sampling pass, reading only the rows of positions up to the first
    rejection.  Reports the call time and the bytes actually read."""
    B, g, V = x.B, x.gamma, x.V
    dcode = sv.SPEC_DTYPE_BF16 if x.dtype == "bf16" else sv.SPEC_DTYPE_F32
    tok = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    acc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws = sv.Workspace(dev)
    wp, wb = ws.get(B, g, V)

    def call(c):
        st = sv.spec_verify_sample_lazy(c["zt"].data_ptr(), c["zd"].data_ptr(), dcode,
                                        c["x"].data_ptr(), c["u"].data_ptr(), x.T, B, g, V,
                                        tok.data_ptr(), acc.data_ptr(), None, wp, wb, sh)
        if st != sv.SPEC_OK:
            raise sv.SpecVerifyError(st, "lazy")

    for s in range(5):
        call(copies[s % len(copies)])
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(steps):
        call(copies[s % len(copies)])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
    k = acc.cpu().numpy().astype(np.int64)
    elt = 2 if x.dtype == "bf16" else 4
    groups = sv.lazy_groups(B, g, V, dcode)
    rows_read = int(sum(lazy_rows_read(int(kb), groups) for kb in k))
    bytes_read = rows_read * V * elt
    return {"what": "lazy stochastic verification (rows of the position groups after the one "
                    "holding the first rejection not read) + final sample, same inputs as the step",
            "ms_per_call": ms, "calls": steps,
            "rows_per_s": world * B * (g + 1) / (ms * 1e-3),
            "position_groups": [list(t) for t in groups],
            "pass1_rows_read": rows_read, "pass1_rows_full": B * (2 * g + 1),
            "pass1_bytes_read": bytes_read, "pass1_bytes_full": acct["bytes_stats"],
            "gpu_launches_per_call": 2 * len(groups) + 1}


def lazy_rows_read(k, groups):
    """Rows the lazy pass reads for a sequence finished at k (-1: bad input,
    found in the first group): the target and draft rows of every group up
    to the one holding k."""
    g = groups[-1][1] - 1
    rows = 0
    for lo, hi in groups:
        rows += (hi - lo) + (min(hi, g) - lo)
        if k < hi:
            break
    return rows


def oracle_slice(x, n, ttok, tpar, nthreads):
    """The oracle over the first n sequences of the batch: sample, greedy and
    the chain-shaped tree.  Returns verified rows."""
    import oracle
    sl = slice(0, n)
    oracle.verify_sample(x.target[sl], x.draft[sl], x.draft_tokens[sl], x.uniforms[sl], x.T,
                         nthreads=nthreads)
    oracle.verify_greedy(x.target[sl], x.draft_tokens[sl], nthreads=nthreads)
    oracle.verify_tree_greedy(x.target[sl], ttok[sl], tpar[sl], nthreads=nthreads)
    return 3 * n * (x.gamma + 1)


def oracle_timing(x, ttok, tpar, budget_s=10.0, threads=None):
    """The oracle, as it stands, over the first n sequences of the batch,
    repeated until budget_s of wall time: one sequence per thread."""
    cores = threads or os.cpu_count() or 1
    n = min(x.B, max(1, cores))
    rows, t = 0, 0.0
    reps = 0
    while t < budget_s and reps < 64:
        t0 = time.perf_counter()
        rows += oracle_slice(x, n, ttok, tpar, cores)
        t += time.perf_counter() - t0
        reps += 1
    return {"value": rows / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} x the first {n} sequences of the batch (sample + greedy + tree), "
                      f"{t:.1f} s wall on {cores} thread{'s' if cores > 1 else ''}"}


# ------------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_59_gb300 import workloads as W
    x = W.make_chain(args.workload)
    ttok, tpar = chain_tree(x)
    cores = os.cpu_count() or 1
    # each step: one sequence per core, all cores, bounded so K + W steps stay within minutes
    n = min(x.B, cores)
    for _ in range(args.warmup):
        oracle_slice(x, 1, ttok, tpar, 1)
    rows, t = 0, 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        rows += oracle_slice(x, n, ttok, tpar, cores)
        t += time.perf_counter() - t0
    value = rows / t
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded generator, chain-b64 recipe)",
        "config": {"workload": args.workload, "B": x.B, "gamma": x.gamma, "V": x.V,
                   "logits": x.dtype, "temperature": x.T,
                   "step": f"fp64 CPU oracle on {n} of the {x.B} sequences (sample + greedy + "
                           "chain-shaped tree)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps x {n} sequences on {cores} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--workload", default="chain-b64",
                    choices=["chain-small", "chain-b8", "chain-b64", "chain-b256"])
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other chain workloads (chain-small, chain-b8, chain-b256)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--rotate", type=int, default=ROTATE,
                    help="input copies the calls rotate over (1 keeps profiler captures small)")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        args.steps = 10 if args.steps is None else args.steps
        args.warmup = 3 if args.warmup is None else args.warmup
        run_reference(args)
    else:
        args.steps = 2000 if args.steps is None else args.steps
        args.warmup = 50 if args.warmup is None else args.warmup
        if args.warmup < 3:
            raise SystemExit("at least 3 warm-up steps are required")
        run_own(args)


if __name__ == "__main__":
    main()
