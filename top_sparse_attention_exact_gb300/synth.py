"""Seeded synthetic decode workloads (inputs only; no attention arithmetic here).

The ReTopK paper ("Recall Before You Rank: Similarity-Guided Top-K Reuse for
Efficient Long-Context Attention", §Experimental Setup) measures Qwen2.5-7B
on PG19 text.  Neither the model nor the dataset is available, so this module
builds stand-in tensors with the same shapes (28 query heads in GQA over 4 KV
heads, head dimension 128, bf16) and with the structure that makes support
reuse meaningful: keys come in topical runs, and each query head wanders
between topics as a Markov chain, so consecutive queries are often similar.

Recipe (per sequence, numpy ``default_rng(seed)``; draws happen in this order):
  1. topic centres  mu[h_kv, n_topics, d] ~ N(0, I)
  2. key topics     one uniform topic per run of ``run`` positions
  3. keys           k_i = mu[z_i] + 0.5 * eps
  4. values         v_i ~ N(0, I)
  5. query topics   per query head, a chain over its KV head's topics that
                    stays with probability ``stay`` and otherwise jumps to a
                    uniform topic; C prompt queries then ``steps`` decode queries
  6. queries        q_t = 2 * mu[g_t] + 0.3 * eps
Every tensor is rounded to bf16 (round to nearest even) before any consumer
sees it; both the CUDA library and the CPU oracle read the same bf16 bits.

Layout of the returned arrays (all uint16 bf16 bit patterns):
  k, v      [B, H_kv, T, d]   T = L0 + steps; position L0 + t - 1 is the key or
                              value appended before decode step t (t >= 1)
  q_prompt  [B, H_q, C, d]    queries of prompt positions L0-C .. L0-1
  q_dec     [steps, B, H_q, d]
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    nan = np.isnan(x)
    rounding = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + rounding) >> 16).astype(np.uint16)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Workload:
    """One synthetic decode workload and the ReTopK hyper-parameters it runs with."""
    name: str
    B: int
    Hq: int
    Hkv: int
    L0: int
    steps: int
    K: int
    C: int
    W: int
    R: int
    tau: float
    T_r: int
    n_topics: int
    run: int
    stay: float
    seeds: tuple = field(default_factory=tuple)
    d: int = 128
    recent: bool = False   # the "recent-R retrieval" ablation instead of Eq. (7)

    @property
    def max_len(self) -> int:
        return self.L0 + self.steps


# Workloads of the pages' evaluation grid (K=512, C=W=32, R=4, tau=0.85,
# T_r=128 at 16K-128K; a tiny single-head case for exhaustive checking; and a
# batched sweep with a high fallback rate).
WORKLOADS = {
    "tiny_1h_2k": Workload("tiny_1h_2k", 1, 1, 1, 2048, 64, 128, 32, 32, 4, 0.85, 16,
                           16, 128, 0.90, (0,)),
    "qwen7b_16k": Workload("qwen7b_16k", 1, 28, 4, 16384, 256, 512, 32, 32, 4, 0.85, 128,
                           64, 256, 0.95, (1,)),
    "qwen7b_32k": Workload("qwen7b_32k", 1, 28, 4, 32768, 256, 512, 32, 32, 4, 0.85, 128,
                           64, 256, 0.95, (2,)),
    "qwen7b_64k": Workload("qwen7b_64k", 1, 28, 4, 65536, 256, 512, 32, 32, 4, 0.85, 128,
                           64, 256, 0.95, (3,)),
    "qwen7b_128k": Workload("qwen7b_128k", 1, 28, 4, 131072, 512, 512, 32, 32, 4, 0.85, 128,
                            64, 256, 0.95, (4,)),
    # the long-context scaling lengths (1M and 5M keys, 2^20 and 5 * 2^20)
    "qwen7b_1m": Workload("qwen7b_1m", 1, 28, 4, 1048576 - 256, 256, 512, 32, 32, 4, 0.85, 128,
                          64, 256, 0.95, (5,)),
    "qwen7b_5m": Workload("qwen7b_5m", 1, 28, 4, 5242880 - 256, 256, 512, 32, 32, 4, 0.85, 128,
                          64, 256, 0.95, (6,)),
}


def batched_sweep(K: int, tau: float, steps: int = 256) -> Workload:
    """Batch of 16 independent 64K sequences with a high fallback rate."""
    return Workload(f"qwen7b_64k_b16_K{K}_tau{tau}", 16, 28, 4, 65536, steps, K, 32, 32, 4,
                    tau, 128, 64, 256, 0.80, tuple(range(100, 116)))


# the batch-16 64K sweep: K in {256, 1024, 2048} x tau in {0.70, 0.95}
for _K in (256, 1024, 2048):
    for _tau in (0.70, 0.95):
        _w = batched_sweep(_K, _tau)
        WORKLOADS[_w.name] = _w


def scaled(w: Workload, **kw) -> Workload:
    """Same recipe with some fields replaced (smaller parity cases)."""
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


def generate_sequence(w: Workload, seed: int):
    """Draw one sequence; returns k, v [Hkv,T,d], q_prompt [Hq,C,d], q_dec [steps,Hq,d]."""
    rng = np.random.default_rng(seed)
    T = w.L0 + w.steps
    d = w.d
    G = w.Hq // w.Hkv
    mu = rng.standard_normal((w.Hkv, w.n_topics, d), dtype=np.float32)
    n_runs = (T + w.run - 1) // w.run
    run_topic = rng.integers(0, w.n_topics, size=(w.Hkv, n_runs))
    z = np.repeat(run_topic, w.run, axis=1)[:, :T]
    k = np.empty((w.Hkv, T, d), dtype=np.uint16)
    v = np.empty((w.Hkv, T, d), dtype=np.uint16)
    for h in range(w.Hkv):
        eps = rng.standard_normal((T, d), dtype=np.float32)
        eps *= np.float32(0.5)
        eps += mu[h][z[h]]
        k[h] = f32_to_bf16_bits(eps)
    for h in range(w.Hkv):
        v[h] = f32_to_bf16_bits(rng.standard_normal((T, d), dtype=np.float32))
    nq = w.C + w.steps
    g = np.empty((w.Hq, nq), dtype=np.int64)
    g[:, 0] = rng.integers(0, w.n_topics, size=w.Hq)
    stay = rng.random((w.Hq, nq)) < w.stay
    jump = rng.integers(0, w.n_topics, size=(w.Hq, nq))
    for t in range(1, nq):
        g[:, t] = np.where(stay[:, t], g[:, t - 1], jump[:, t])
    eq = rng.standard_normal((w.Hq, nq, d), dtype=np.float32)
    q = np.empty((w.Hq, nq, d), dtype=np.float32)
    for h in range(w.Hq):
        q[h] = np.float32(2.0) * mu[h // G][g[h]] + np.float32(0.3) * eq[h]
    qb = f32_to_bf16_bits(q)
    q_prompt = np.ascontiguousarray(qb[:, :w.C])
    q_dec = np.ascontiguousarray(qb[:, w.C:].transpose(1, 0, 2))
    return k, v, q_prompt, q_dec


def generate(w: Workload):
    """Draw every sequence of a workload; shapes as in the module docstring."""
    seeds = w.seeds if w.seeds else tuple(range(w.B))
    assert len(seeds) == w.B
    T = w.L0 + w.steps
    k = np.empty((w.B, w.Hkv, T, w.d), dtype=np.uint16)
    v = np.empty_like(k)
    q_prompt = np.empty((w.B, w.Hq, w.C, w.d), dtype=np.uint16)
    q_dec = np.empty((w.steps, w.B, w.Hq, w.d), dtype=np.uint16)
    for b, s in enumerate(seeds):
        kb, vb, qp, qd = generate_sequence(w, s)
        k[b], v[b], q_prompt[b], q_dec[:, b] = kb, vb, qp, qd
    return k, v, q_prompt, q_dec


def random_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """Gaussian bf16 bits, for small unit cases."""
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))
