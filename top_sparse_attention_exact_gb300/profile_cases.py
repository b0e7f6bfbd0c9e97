"""Small, self-contained GPU runs for profiler captures (ncu).

    python -m top_sparse_attention_exact_gb300.profile_cases exact  [--workload W] [--reps N]
    python -m top_sparse_attention_exact_gb300.profile_cases decode [--workload W] [--steps N]

`exact` runs N stateless Exact Top-K steps on one synthetic workload (the
scan kernel of the 128K case streams 134 MB of K rows, more than the 129 MB
L2); `decode` initialises a ReTopK context and runs N eager decode steps
followed by 4 exact steps.  Both print a one-line summary and exit 0 on
success, so they can be run plainly before being run under a profiler.
"""
from __future__ import annotations

import argparse

import torch

from . import retopk, synth
from .runner import DecodeRun, ExactRun, to_dev


def run_exact(name: str, reps: int) -> None:
    w = synth.scaled(synth.WORKLOADS[name], steps=1)
    k, v, qp, qd = synth.generate(w)
    kc, vc, q = to_dev(k, "cuda"), to_dev(v, "cuda"), to_dev(qd[0], "cuda")
    sl = torch.full((w.B,), w.L0 + 1, dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
    idx = torch.empty((w.B, w.Hq, w.K), dtype=torch.int32, device="cuda")
    ws = torch.empty(retopk.exact_topk_workspace_bytes(w.B, w.Hq, w.Hkv, w.d, k.shape[2], w.K) + 256,
                     dtype=torch.uint8, device="cuda")
    for _ in range(reps):
        retopk.exact_topk_attention_step(q, kc, vc, sl, w.K, out, idx, ws)
    torch.cuda.synchronize()
    print(f"exact {name}: {reps} steps, L={w.L0 + 1}, first support entries {idx[0, 0, :3].tolist()}")


def run_decode(name: str, steps: int) -> None:
    w = synth.scaled(synth.WORKLOADS[name], steps=max(steps, 1))
    dr = DecodeRun(w)
    ex = ExactRun(dr)
    for t in range(steps):
        dr.step(t)
    for t in range(4):
        ex.step(dr.q_dec[t])
    torch.cuda.synchronize()
    print(f"decode {name}: {steps} steps, counters {dr.ctx.retopk_get_counters()}, "
          f"status {dr.ctx.retopk_get_status()}")


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["exact", "decode"])
    ap.add_argument("--workload", default="qwen7b_128k")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--steps", type=int, default=24)
    a = ap.parse_args()
    if a.case == "exact":
        run_exact(a.workload, a.reps)
    else:
        run_decode(a.workload, a.steps)


if __name__ == "__main__":
    main()
