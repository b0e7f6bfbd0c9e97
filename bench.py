#!/usr/bin/env python
"""Decode-attention benchmark: ReTopK and Exact Top-K on one synthetic
Qwen2.5-7B-shaped layer (28 query heads over 4 KV heads, d = 128, bf16).

One step = one decode step of one layer: append the token's K/V row, then
retopk_decode_step (recall, path switch, candidate union, rerank, Top-K,
softmax-value aggregation, cache update), replayed as one CUDA graph.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: W untimed steps, then exactly K steps.  Every step is bracketed by its
own CUDA events on the launching stream; between steps the L2 is flushed by
writing a 256 MiB buffer (the flush is outside the events).  value = mean
microseconds per step per layer (lower is better).  The JSON line also holds
the Exact Top-K step time on the same inputs, the path mix, the roofline of
the full-history scan kernel (algorithmic K-row bytes / its CUDA-event time),
the fp64 CPU oracle timed on the host cores on a bounded sample of the same
workload, an end-to-end number through host buffers, and the SM clocks seen
during the timed region.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAK_FALLBACK_GBS = 6800.0
GPU_BUSY_CYCLES = 200_000      # ~0.1 ms spin before each timed step (outside the events)
METRIC = "decode-attn µs/step/layer at 128K, K=512 (ReTopK & Exact); HBM GB/s vs peak"
UNIT = "us/step/layer"


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback"


def workload_desc(w):
    return (f"{w.name}: B={w.B}, Hq={w.Hq}, Hkv={w.Hkv}, d={w.d}, L0={w.L0}, {w.steps} decode steps, "
            f"K={w.K}, C={w.C}, W={w.W}, R={w.R}, tau={w.tau}, T_r={w.T_r}; topic-mixture keys "
            f"({w.n_topics} topics, runs of {w.run}), Markov query topics (stay {w.stay})")


def oracle_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------
class L2Flush:
    """Evicts the 129 MB L2 between timed steps: writes a 256 MiB buffer, then
    reads another one so that no dirty line is left to be written back while
    the next step runs (both outside the timed events)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(64 << 20, dtype=torch.int32, device=dev)
        self.r = torch.zeros(64 << 20, dtype=torch.int32, device=dev)
        self.sink = torch.empty((), dtype=torch.int32, device=dev)

    def __call__(self):
        import torch
        self.w.fill_(1)
        torch.amax(self.r, dim=0, out=self.sink)


# ------------------------------------------------------------------------------
def run_oracle_steps(w, arrays, state, steps, budget_s=None, b=0):
    """Times oracle.decode_step for `steps` consecutive steps of sequence b from `state`."""
    import oracle
    k, v, qp, qd = arrays
    done, t0 = 0, time.perf_counter()
    for t in steps:
        oracle.decode_step(state, qd[t, b], k[b], v[b], w.L0 + t + 1, w.Hkv, w.W, w.R, w.T_r, w.tau)
        done += 1
        if budget_s is not None and time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0


def reference_arm(args, w, rank, world):
    """The fp64 CPU oracle as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return 0
    from top_sparse_attention_exact_gb300 import synth
    import oracle
    oracle.build()
    oracle.set_threads(oracle_threads())
    w1 = synth.scaled(w, B=1, seeds=w.seeds[:1])
    arrays = synth.generate(w1)
    k, v, qp, qd = arrays
    # cache initialisation (set-up, untimed)
    st = oracle.init_cache(qp[0], k[0], w1.L0, w1.Hq, w1.Hkv, w1.K, w1.C)
    W_, K_ = min(args.warmup, w1.steps - 1), None
    K_ = max(1, min(args.steps, w1.steps - W_))
    run_oracle_steps(w1, arrays, st, range(0, W_))
    n, secs = run_oracle_steps(w1, arrays, st, range(W_, W_ + K_))
    us = secs / n * 1e6
    cores = oracle.get_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world,
        "steps": n, "warmup": W_, "ms_per_step": us / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w1), "sequences_timed": 1},
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"decode steps {W_ + 1}..{W_ + n} of sequence 0 after {W_} warm-up steps"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------
def our_arm(args, w, rank, world, dist):
    import torch
    from top_sparse_attention_exact_gb300 import synth
    from top_sparse_attention_exact_gb300 import retopk
    from top_sparse_attention_exact_gb300.runner import DecodeRun, ExactRun, to_dev

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    # each rank runs its own independent replica (different sequences)
    wr = synth.scaled(w, seeds=tuple(s + 1000 * rank for s in w.seeds)) if rank else w
    arrays = synth.generate(wr)
    Wm = max(3, args.warmup)
    Kt = args.steps
    if Wm + Kt > wr.steps:
        raise SystemExit(f"--warmup + --steps must be <= {wr.steps} decode steps of {wr.name}")

    dr = DecodeRun(wr, arrays=arrays, device=dev)
    init_state = dr.ctx.retopk_export_state() if rank == 0 else None
    dr.capture()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    for t in range(Wm):
        dr.replay(t)
    c0 = dr.ctx.retopk_get_counters()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kt)]
    step_paths = []
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for i in range(Kt):
            t = Wm + i
            flush()
            torch.cuda._sleep(GPU_BUSY_CYCLES)   # keeps the GPU busy while the host enqueues
            dr.stage(t)
            ev[i][0].record(stream)
            dr.graph.replay()
            ev[i][1].record(stream)
            dr.t = t + 1
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    step_ms = np.array([a.elapsed_time(b) for a, b in ev])
    c1 = dr.ctx.retopk_get_counters()
    if dist:
        dist.barrier()
    total_ms = float(step_ms.sum())
    if dist:
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    us_step = total_ms / Kt * 1000.0

    # per-step path mix (eager re-run of the same timed steps on a fresh context,
    # with the same inputs, to classify each step; timing is not taken here)
    mix = {k2: c1[k2] - c0[k2] for k2 in ("reuse", "fallback", "refresh")}
    head_steps = max(1, sum(mix.values()))

    # ---- Exact Top-K on the same inputs (graph replay, same flush) ----------
    ex = ExactRun(dr)
    sl_ex = dr.seqlens                                # the cache already holds every timed row
    L_save = sl_ex.clone()
    q_buf = torch.empty_like(dr.q_dec[0])
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            retopk.exact_topk_attention_step(q_buf, dr.k_cache, dr.v_cache, sl_ex, wr.K, ex.out, ex.idx, ex.ws, s)
    stream.wait_stream(s)
    torch.cuda.synchronize()
    ex_ms = []
    for i in range(Kt):
        t = Wm + i
        flush()
        torch.cuda._sleep(GPU_BUSY_CYCLES)
        sl_ex.fill_(wr.L0 + t + 1)
        q_buf.copy_(dr.q_dec[t])
        a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b2.record(stream)
        ex_ms.append((a, b2))
    torch.cuda.synchronize()
    ex_ms = np.array([a.elapsed_time(b2) for a, b2 in ex_ms])
    us_exact = float(ex_ms.mean() * 1000.0)

    # ---- scan kernel roofline: eager exact steps with CUDA events around the
    #      scan launch (library-side timing), same flush between steps -------
    retopk.profile_enable(True)
    retopk.profile_read()
    n_prof = min(Kt, 64)
    for i in range(n_prof):
        t = Wm + i
        flush()
        torch.cuda._sleep(GPU_BUSY_CYCLES)
        sl_ex.fill_(wr.L0 + t + 1)
        retopk.exact_topk_attention_step(dr.q_dec[t], dr.k_cache, dr.v_cache, sl_ex, wr.K, ex.out, ex.idx, ex.ws)
    torch.cuda.synchronize()
    n_scan, scan_ms = retopk.profile_read()
    retopk.profile_enable(False)
    sl_ex.copy_(L_save)
    mean_L = np.mean([wr.L0 + Wm + i + 1 for i in range(n_prof)])
    scan_bytes = wr.B * wr.Hkv * mean_L * wr.d * 2          # every K row once per GQA group
    scan_us = scan_ms / max(n_scan, 1) * 1000.0
    peak, peak_kind = measured_peak()
    achieved = scan_bytes / (scan_us * 1e-6) / 1e9
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "scan_traffic.json")) as f:
            tr = json.load(f)
        if tr.get("kernel_hash") == kernel_hash():
            traffic = float(tr["bytes_per_launch_at_128k"]) * (mean_L / 131073.0)
    except Exception:
        traffic = None

    # ---- end to end through the public API with host buffers --------------
    e2e = None
    if not args.no_e2e:
        de = DecodeRun(wr, arrays=arrays, device=dev)
        qh = torch.from_numpy(np.ascontiguousarray(arrays[3]).view(np.int16)).pin_memory()   # [steps,B,Hq,d]
        kn = torch.from_numpy(np.ascontiguousarray(arrays[0][:, :, wr.L0:].transpose(2, 0, 1, 3)).view(np.int16)).pin_memory()
        vn = torch.from_numpy(np.ascontiguousarray(arrays[1][:, :, wr.L0:].transpose(2, 0, 1, 3)).view(np.int16)).pin_memory()
        out_h = torch.empty((Kt + Wm, wr.B, wr.Hq, wr.d), dtype=torch.int16).pin_memory()
        qd_, kd_, vd_ = (torch.empty_like(qh[0], device=dev), torch.empty_like(kn[0], device=dev),
                         torch.empty_like(vn[0], device=dev))

        def e2e_step(t):
            qd_.copy_(qh[t], non_blocking=True)
            kd_.copy_(kn[t], non_blocking=True)
            vd_.copy_(vn[t], non_blocking=True)
            de.ctx.retopk_append_kv(kd_, vd_, de.k_cache, de.v_cache, de.seqlens)
            de.ctx.retopk_decode_step(qd_, de.k_cache, de.v_cache, de.seqlens, de.out)
            out_h[t].copy_(de.out, non_blocking=True)

        for t in range(Wm):
            e2e_step(t)
        torch.cuda.synchronize()
        e_ev = []
        for i in range(Kt):
            t = Wm + i
            flush()
            a, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step(t)
            b2.record(stream)
            e_ev.append((a, b2))
        torch.cuda.synchronize()
        e_us = float(np.mean([a.elapsed_time(b2) for a, b2 in e_ev]) * 1000.0)
        e2e = {"value": e_us, "unit": UNIT,
               "h2d_bytes_per_step": int(qh[0].numel() * 2 + kn[0].numel() * 2 + vn[0].numel() * 2),
               "d2h_bytes_per_step": int(out_h[0].numel() * 2)}
        del de

    # ---- CPU oracle baseline on a bounded sample (rank 0 only) -------------
    cpu = None
    if rank == 0 and not args.no_cpu:
        import oracle
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        from parity import oracle_state_from_gpu
        oracle.build()
        oracle.set_threads(oracle_threads())
        st = oracle_state_from_gpu(init_state, 0, wr.K)
        n, secs = run_oracle_steps(wr, arrays, st, range(0, wr.steps), budget_s=args.cpu_budget)
        cpu = {"value": secs / n * 1e6, "unit": UNIT, "cores": oracle.get_threads(), "kind": "oracle",
               "sample": f"decode steps 1..{n} of sequence 0 from the GPU's initialised cache "
                         f"(free-running, ~{args.cpu_budget:.0f} s budget)"}

    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": world, "steps": Kt, "warmup": Wm,
        "ms_per_step": us_step / 1000.0, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(wr), "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (256 MiB write, then 256 MiB read), outside the timed events",
                   "exact_topk_us_per_step": us_exact, "speedup_vs_exact": us_exact / us_step,
                   "reuse_share": mix["reuse"] / head_steps, "fallback_share": mix["fallback"] / head_steps,
                   "refresh_share": mix["refresh"] / head_steps,
                   "mean_candidates": (c1["sum_M"] - c0["sum_M"]) / max(1, mix["reuse"]),
                   "step_us_p50": float(np.median(step_ms) * 1000), "step_us_p90": float(np.percentile(step_ms, 90) * 1000),
                   "wall_s_timed_loop": wall},
        "roofline": {"kernel": "scan_kernel (full-history QK + first radix digit)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic, "scan_us": scan_us,
                     "algorithmic_bytes": scan_bytes, "launches_timed": n_scan},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 6 * Kt,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def kernel_hash():
    import hashlib
    p = os.path.join(ROOT, "top_sparse_attention_exact_gb300", "csrc", "scan.cu")
    return hashlib.sha1(open(p, "rb").read()).hexdigest()[:12]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=496)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--workload", default="qwen7b_128k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()

    from top_sparse_attention_exact_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            dist_mod.init_process_group("nccl")
            dist = dist_mod
    if args.impl == "reference":
        return reference_arm(args, w, rank, world)
    from top_sparse_attention_exact_gb300 import _build
    _build.build()
    rc = our_arm(args, w, rank, world, dist)
    if dist:
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
