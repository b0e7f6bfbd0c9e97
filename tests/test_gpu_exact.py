"""Exact Top-K attention through the C ABI against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_exact, out_close
from top_sparse_attention_exact_gb300 import retopk, synth
from top_sparse_attention_exact_gb300.runner import to_dev

pytestmark = pytest.mark.gpu


def run_exact(q, k, v, L, K, max_len=None):
    """q [B,Hq,d], k/v [B,Hkv,T,d] uint16 bits; returns (idx [B,Hq,K], out f32)."""
    B, Hq, d = q.shape
    Hkv, T = k.shape[1], k.shape[2]
    max_len = max_len or T
    kc = torch.zeros((B, Hkv, max_len, d), dtype=torch.int16, device="cuda")
    vc = torch.zeros_like(kc)
    kc[:, :, :T] = to_dev(k, "cuda")
    vc[:, :, :T] = to_dev(v, "cuda")
    qd = to_dev(q, "cuda")
    sl = torch.tensor(np.asarray(L, np.int32), device="cuda")
    out = torch.empty((B, Hq, d), dtype=torch.int16, device="cuda")
    idx = torch.empty((B, Hq, K), dtype=torch.int32, device="cuda")
    retopk.exact_topk_attention_step(qd, kc, vc, sl, K, out, idx)
    torch.cuda.synchronize()
    o = out.cpu().numpy().view(np.uint16)
    return idx.cpu().numpy(), synth.bf16_bits_to_f32(o)


def gauss(seed, B, Hq, Hkv, T, d=128):
    rng = np.random.default_rng(seed)
    return (synth.random_bf16(rng, (B, Hq, d), 1.0), synth.random_bf16(rng, (B, Hkv, T, d)),
            synth.random_bf16(rng, (B, Hkv, T, d)))


@pytest.mark.parametrize("B,Hq,Hkv,L,K", [
    (2, 4, 2, [1000, 333], 64),          # ragged lengths, several tiles and a tail
    (1, 1, 1, [1], 8),                   # a single key
    (1, 1, 1, [15], 16),                 # fewer keys than K
    (3, 2, 1, [16, 17, 300], 16),        # tile-edge lengths
    (2, 4, 2, [50, 17], 64),             # K > L everywhere: dense attention
    (1, 16, 1, [2049], 100),             # 16 query heads per KV head (two n-tiles)
    (1, 7, 1, [4099], 4096),             # the largest K
])
def test_exact_random(B, Hq, Hkv, L, K):
    q, k, v = gauss(B * 1000 + Hq + K, B, Hq, Hkv, max(L) + 5)
    idx, out = run_exact(q, k, v, L, K, max_len=max(L) + 37)
    errs = compare_exact(q, k, v, L, K, idx, out, "random")
    assert not errs, "\n".join(errs[:20])


def test_exact_K_ge_L_is_dense_attention():
    q, k, v = gauss(7, 1, 4, 2, 200)
    idx, out = run_exact(q, k, v, [200], 256)
    for h in range(4):
        assert idx[0, h, :200].tolist() == list(range(200)) and (idx[0, h, 200:] == -1).all()
        ref = oracle.dense_attention(q[0, h], k[0, h // 2], v[0, h // 2], 200)
        ok, mx, rel = out_close(out[0, h], ref)
        assert ok, (mx, rel)


def test_exact_all_ties_take_lowest_indices():
    rng = np.random.default_rng(3)
    d = 128
    row = synth.random_bf16(rng, (d,))
    k = np.broadcast_to(row, (1, 1, 5000, d)).copy()       # every score equal
    v = synth.random_bf16(rng, (1, 1, 5000, d))
    q = synth.random_bf16(rng, (1, 3, d))
    idx, out = run_exact(q, k, v, [5000], 300)
    for h in range(3):
        assert idx[0, h].tolist() == list(range(300))
        ok, mx, rel = out_close(out[0, h], synth.bf16_bits_to_f32(v[0, 0, :300]).astype(np.float64).mean(0))
        assert ok, (mx, rel)


def test_exact_many_score_ties():
    # keys drawn from 3 distinct rows: scores take 3 values, heavy ties at the K-th
    rng = np.random.default_rng(4)
    rows = synth.random_bf16(rng, (3, 128))
    pick = rng.integers(0, 3, size=3000)
    k = rows[pick][None, None]
    v = synth.random_bf16(rng, (1, 1, 3000, 128))
    q = synth.random_bf16(rng, (1, 2, 128))
    idx, out = run_exact(q, k, v, [3000], 1111)
    errs = compare_exact(q, k, v, [3000], 1111, idx, out, "ties")
    assert not errs, "\n".join(errs[:10])
    for h in range(2):
        sup, _, _ = oracle.exact_one(q[0, h], k[0, 0], v[0, 0], 3000, 1111)
        assert idx[0, h].tolist() == sup.tolist()        # exact ties are resolved identically


def test_exact_ties_beyond_shared_staging():
    # 20000 equal scores: every key is a candidate, more than one CTA stages in
    # shared memory, so the selection runs over the global candidate segments
    rng = np.random.default_rng(5)
    row = synth.random_bf16(rng, (128,))
    k = np.broadcast_to(row, (1, 1, 20000, 128)).copy()
    v = synth.random_bf16(rng, (1, 1, 20000, 128))
    q = synth.random_bf16(rng, (1, 2, 128))
    idx, out = run_exact(q, k, v, [20000], 300)
    for h in range(2):
        assert idx[0, h].tolist() == list(range(300))
        ok, mx, rel = out_close(out[0, h], synth.bf16_bits_to_f32(v[0, 0, :300]).astype(np.float64).mean(0))
        assert ok, (mx, rel)


def test_exact_one_segment_holds_most_candidates():
    # 1500 tied top scores inside the first of 8 candidate segments (more than
    # a segment keeps in shared memory), the other 14884 keys far below
    rng = np.random.default_rng(6)
    q = synth.random_bf16(rng, (1, 1, 128), 1.0)
    qf = synth.bf16_bits_to_f32(q[0, 0]).astype(np.float64)
    k = synth.random_bf16(rng, (1, 1, 16384, 128), 0.05)
    top = synth.f32_to_bf16_bits((2.0 * qf / np.linalg.norm(qf)).astype(np.float32))
    k[0, 0, :1500] = top
    v = synth.random_bf16(rng, (1, 1, 16384, 128))
    idx, out = run_exact(q, k, v, [16384], 512)
    errs = compare_exact(q, k, v, [16384], 512, idx, out, "segment")
    assert not errs, "\n".join(errs[:10])
    assert idx[0, 0].tolist() == list(range(512))


def test_exact_long_sequence_several_slices_per_segment():
    # 150001 keys: each of the 8 segments spans more than one shared-memory slice
    q, k, v = gauss(8, 1, 2, 1, 150001)
    idx, out = run_exact(q, k, v, [150001], 512)
    errs = compare_exact(q, k, v, [150001], 512, idx, out, "long")
    assert not errs, "\n".join(errs[:10])


@pytest.mark.parametrize("name", ["qwen7b_16k"])
def test_exact_qwen_shape_all_heads(name):
    w = synth.scaled(synth.WORKLOADS[name], steps=1)
    k, v, qp, qd = synth.generate(w)
    L = [w.L0 + 1]
    idx, out = run_exact(qd[0], k, v, L, w.K)
    errs = compare_exact(qd[0], k, v, L, w.K, idx, out, name)
    assert not errs, "\n".join(errs[:20])


@pytest.mark.parametrize("L,max_len", [((1 << 20) - 1, 1 << 20),
                                       (5 * (1 << 20) + 3, 1 << 23)])   # the largest cache
def test_exact_longest_history(L, max_len):
    # 1M and 5M keys (the long-context lengths): 8 segments of ~131K / ~655K
    # scores, each copied in many shared-memory slices; the second case in a
    # cache of the largest supported max_len
    q, k, v = gauss(9, 1, 2, 1, L)
    idx, out = run_exact(q, k, v, [L], 512, max_len=max_len)
    from parity import support_ok
    for h in range(2):
        sup, kth, ref = oracle.exact_one(q[0, h], k[0, 0], v[0, 0], L, 512)
        ok, msg = support_ok(q[0, h], k[0, 0], idx[0, h], sup, kth)
        assert ok, msg
        ok, mx, rel = out_close(out[0, h], ref)
        assert ok, (h, mx, rel)


def test_exact_headline_128k_sampled_heads():
    w = synth.scaled(synth.WORKLOADS["qwen7b_128k"], steps=1)
    k, v, qp, qd = synth.generate(w)
    L = w.L0 + 1
    idx, out = run_exact(qd[0], k, v, [L], w.K, max_len=w.L0 + 512)
    for h in (0, 6, 13, 20, 27):
        sup, kth, ref = oracle.exact_one(qd[0, 0, h], k[0, h // 7], v[0, h // 7], L, w.K)
        from parity import support_ok
        ok, msg = support_ok(qd[0, 0, h], k[0, h // 7], idx[0, h], sup, kth)
        assert ok, msg
        ok, mx, rel = out_close(out[0, h], ref)
        assert ok, (h, mx, rel)


@pytest.mark.parametrize("B", [2, 5, 16])
def test_exact_batched_cluster_sizes(B):
    # 28 query heads per sequence over 4 KV heads: B = 2, 5 and 16 give the
    # select 4, 2 and 1 CTAs per head (the clusters of one wave), ragged lengths
    rng = np.random.default_rng(100 + B)
    L = [int(x) for x in rng.integers(900, 3100, size=B)]
    q, k, v = gauss(200 + B, B, 28, 4, max(L) + 3)
    idx, out = run_exact(q, k, v, L, 64, max_len=max(L) + 19)
    errs = compare_exact(q, k, v, L, 64, idx, out, f"B{B}")
    assert not errs, "\n".join(errs[:20])
