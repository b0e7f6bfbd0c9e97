"""Device-resident decode loop over a synthetic workload (used by the tests,
the smoke check and bench.py).

Holds the KV caches, the per-step inputs and a ReTopK context on one GPU, and
runs each decode step as `append the new token's K/V row, then
retopk_decode_step` -- eagerly or as one replayed CUDA graph.  Only the
library's kernels touch the data; torch provides memory and streams.
"""
from __future__ import annotations

import numpy as np
import torch

from . import synth
from .retopk import ReTopK, exact_topk_attention_step, exact_topk_workspace_bytes, profile_enable


def to_dev(a: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bits -> int16 CUDA tensor holding the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


class DecodeRun:
    """`fused` runs each step through retopk_decode_step_kv (append folded into
    the decision kernel); otherwise retopk_append_kv then retopk_decode_step.
    `scratch` (a uint8 CUDA tensor) makes the context share its per-step
    scratch with other contexts (retopk_create_shared)."""

    def __init__(self, w: synth.Workload, arrays=None, device="cuda", max_len=None, fused: bool = True,
                 scratch=None, cluster: int = 0):
        self.w = w
        self.fused = fused
        self.device = torch.device(device)
        k, v, qp, qd = arrays if arrays is not None else synth.generate(w)
        self.k_host, self.v_host, self.qp_host, self.qd_host = k, v, qp, qd
        B, Hkv, d, L0 = w.B, w.Hkv, w.d, w.L0
        self.max_len = max_len or w.max_len
        dev = self.device
        self.k_cache = torch.zeros((B, Hkv, self.max_len, d), dtype=torch.int16, device=dev)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.k_cache[:, :, :L0] = to_dev(k[:, :, :L0], dev)
        self.v_cache[:, :, :L0] = to_dev(v[:, :, :L0], dev)
        self.seqlens = torch.full((B,), L0, dtype=torch.int32, device=dev)
        self.q_prompt = to_dev(qp, dev)
        self.q_dec = to_dev(qd, dev)                                        # [steps,B,Hq,d]
        self.k_new = to_dev(np.ascontiguousarray(k[:, :, L0:].transpose(2, 0, 1, 3)), dev)  # [steps,B,Hkv,d]
        self.v_new = to_dev(np.ascontiguousarray(v[:, :, L0:].transpose(2, 0, 1, 3)), dev)
        self.out = torch.zeros((B, w.Hq, d), dtype=torch.int16, device=dev)
        self.ctx = ReTopK(B, w.Hq, Hkv, self.max_len, K=w.K, C=w.C, W=w.W, R=w.R, T_r=w.T_r,
                          tau=w.tau, d=d, device=dev, recent=w.recent, scratch=scratch, cluster=cluster)
        self.ctx.retopk_init_cache(self.q_prompt, self.k_cache, self.seqlens)
        self.t = 0
        self.graph = None

    # ---- eager -----------------------------------------------------------
    def step(self, t: int | None = None, stream=None):
        t = self.t if t is None else t
        self._one(self.k_new[t], self.v_new[t], self.q_dec[t], stream)
        self.t = t + 1
        return self.out

    def _one(self, k_new, v_new, q, stream):
        if self.fused:
            self.ctx.retopk_decode_step_kv(k_new, v_new, q, self.k_cache, self.v_cache, self.seqlens, self.out,
                                           stream)
        else:
            self.ctx.retopk_append_kv(k_new, v_new, self.k_cache, self.v_cache, self.seqlens, stream)
            self.ctx.retopk_decode_step(q, self.k_cache, self.v_cache, self.seqlens, self.out, stream)

    # ---- CUDA graph: one capture, replayed with per-step staging copies ----
    def capture(self, profiled: bool = False):
        """Capture one decode step (append included) as a graph; `profiled` embeds the library's
        per-kernel timing events in it (read them with retopk.profile_read)."""
        w = self.w
        self.q_buf = torch.empty((w.B, w.Hq, w.d), dtype=torch.int16, device=self.device)
        self.k_buf = torch.empty((w.B, w.Hkv, w.d), dtype=torch.int16, device=self.device)
        self.v_buf = torch.empty_like(self.k_buf)
        # capture records the launches without running them
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        if profiled:
            profile_enable(True)
        try:
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    self._one(self.k_buf, self.v_buf, self.q_buf, s)
        finally:
            if profiled:
                profile_enable(False)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = g
        return g

    def stage(self, t: int):
        self.q_buf.copy_(self.q_dec[t])
        self.k_buf.copy_(self.k_new[t])
        self.v_buf.copy_(self.v_new[t])

    def replay(self, t: int | None = None):
        t = self.t if t is None else t
        self.stage(t)
        self.graph.replay()
        self.t = t + 1
        return self.out


class ExactRun:
    """Stateless Exact Top-K steps over the same inputs (the comparison path)."""

    def __init__(self, dr: DecodeRun, workspace=None):
        w = dr.w
        self.dr = dr
        self.idx = torch.empty((w.B, w.Hq, w.K), dtype=torch.int32, device=dr.device)
        self.out = torch.empty((w.B, w.Hq, w.d), dtype=torch.int16, device=dr.device)
        nb = exact_topk_workspace_bytes(w.B, w.Hq, w.Hkv, w.d, dr.max_len, w.K)
        self.ws = workspace if workspace is not None else torch.empty(nb + 256, dtype=torch.uint8, device=dr.device)

    def step(self, q, stream=None, seqlens=None):
        dr = self.dr
        sl = dr.seqlens if seqlens is None else seqlens
        exact_topk_attention_step(q, dr.k_cache, dr.v_cache, sl, dr.w.K, self.out, self.idx, self.ws, stream)
        return self.out

    def capture(self, profiled: bool = False):
        """One exact step on staging buffers (q_buf, seqlens_buf) as a graph."""
        dr = self.dr
        self.q_buf = torch.empty_like(dr.q_dec[0])
        self.sl_buf = dr.seqlens.clone()
        s = torch.cuda.Stream(device=dr.device)
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        if profiled:
            profile_enable(True)
        try:
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    self.step(self.q_buf, s, self.sl_buf)
        finally:
            if profiled:
                profile_enable(False)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = g
        return g

    def stage(self, t: int):
        """Stages decode step t's query and length L0 + t + 1 for the graph."""
        self.q_buf.copy_(self.dr.q_dec[t])
        self.sl_buf.fill_(self.dr.w.L0 + t + 1)

    def replay(self, t: int):
        """Exact step for decode step t's query over the first L0 + t + 1 keys."""
        self.stage(t)
        self.graph.replay()
        return self.out
