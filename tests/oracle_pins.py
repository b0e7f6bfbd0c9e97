"""Pins that tie the fp64 oracle to facts fixed outside itself.

Each pin takes the oracle's ctypes handle so that the same checks can be run
against deliberately broken builds of the oracle (tests/test_oracle_mutants.py)
and must catch them.  Sources of truth used here, none of which is the oracle:
  * the hand-worked example in tests/golden/hand_worked.json (derived from the
    ReTopK paper's Eqs. (1), (4), (6)-(13));
  * closed forms (cosine of parallel / orthogonal vectors, softmax of equal or
    two scores, scores against unit vectors);
  * library routines: numpy float64 matmul, torch's scaled_dot_product_attention
    in float64, scipy's cosine distance;
  * brute-force definitions on tiny inputs (rank counting for Top-K, Python
    set union for the candidate set);
  * invariants the paper states: reranking recovers S_t when S_t is a subset
    of the candidates (Eq. (11) remark); the path rule (Eq. (13)); cache
    insertion after either path; K >= L makes Exact Top-K dense attention.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from top_sparse_attention_exact_gb300.synth import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_worked.json")


def _bf(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _f(h):
    return bf16_bits_to_f32(h).astype(np.float64)


def _rank_topk(s, K):
    """Brute force: key i is selected iff fewer than K keys beat it."""
    n = len(s)
    sel = []
    for i in range(n):
        beats = sum(1 for j in range(n) if s[j] > s[i] or (s[j] == s[i] and j < i))
        if beats < K:
            sel.append(i)
    return sel


# ----------------------------------------------------------------------------
def pin_hand_worked_exact(lib):
    g = json.load(open(GOLDEN))
    q, k, v = _bf(g["q"]), _bf(g["k"]), _bf(g["v"])
    s = oracle.scores(q, k, lib=lib)
    assert np.array_equal(s, np.array(g["scores"])), s
    for key, K in (("exact_K2", 2), ("exact_K3", 3)):
        sup, _, out = oracle.exact_one(q, k, v, 5, K, lib=lib)
        assert sup.tolist() == g[key]["support"], (key, sup)
        assert np.allclose(out, g[key]["out"], rtol=0, atol=1e-15), (key, out)


def pin_hand_worked_reuse(lib):
    g = json.load(open(GOLDEN))
    rs = g["reuse_step"]
    q, k, v = _bf(g["q"]), _bf(g["k"]), _bf(g["v"])
    for case in rs["cases"]:
        st = oracle.CacheState(Hq=1, C=2, K=2, d=4)
        st.fq[0] = _bf(rs["cache_q"])
        for c, sup in enumerate(rs["cache_support"]):
            st.fsup[0, c, :len(sup)] = sup
            st.flen[0, c] = len(sup)
        st.seq[:] = [0, 2, 0]
        r = oracle.decode_step(st, q[None], k[None], v[None], 5, 1, case["W"], 1, 0, case["tau"], lib=lib)
        assert np.allclose(r["rho"][0], rs["rho"], atol=0), r["rho"]
        assert r["topR"][0].tolist() == rs["topR"]
        assert int(r["path"][0]) == case["path"], (case, r["path"])
        if case["path"] == 0:
            assert r["cand"][0, :r["M"][0]].tolist() == case["A"], r["cand"]
        assert r["sup"][0, :r["sup_len"][0]].tolist() == case["support"]
        assert np.allclose(r["out"][0], case["out"], rtol=0, atol=1e-15), r["out"]
        after = rs["cache_after"]
        assert st.seq.tolist() == [after["next_slot"], after["count"], after["t_dec"]]
        assert np.array_equal(st.fq[0, after["slot_written"]], q)
        assert st.fsup[0, after["slot_written"], :st.flen[0, 0]].tolist() == case["support"]
        assert np.array_equal(st.fq[0, 1], _bf(rs["cache_q"][1]))


def pin_scores_library_and_closed_form(lib):
    rng = np.random.default_rng(11)
    q = _bf(rng.standard_normal(128))
    k = _bf(rng.standard_normal((300, 128)))
    ref = _f(k) @ _f(q) / math.sqrt(128.0)
    got = oracle.scores(q, k, lib=lib)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)
    idx = np.array([299, 0, 17, 17], dtype=np.int32)
    assert np.allclose(oracle.scores(q, k, idx, lib=lib), ref[idx], rtol=1e-13, atol=1e-13)
    # unit query picks out one coordinate: e_i = k_i[j] / sqrt(d)
    e = np.zeros(128, np.float32)
    e[5] = 1.0
    s = oracle.scores(_bf(e), k, lib=lib)
    assert np.allclose(s, _f(k)[:, 5] / math.sqrt(128.0), rtol=4e-16, atol=0)


def pin_topk_brute_force(lib):
    rng = np.random.default_rng(12)
    for n in range(1, 13):
        for trial in range(6):
            s = rng.integers(-2, 3, size=n).astype(np.float64)   # many ties
            for K in range(1, n + 2):
                got = oracle.topk(s, K, lib=lib)
                want = _rank_topk(s, K)
                assert sorted(got.tolist()) == want, (s, K, got)
                # rank order: non-increasing score, lower index first on ties
                for a, b in zip(got[:-1], got[1:]):
                    assert s[a] > s[b] or (s[a] == s[b] and a < b)
    # explicit index labels are carried through
    s = np.array([1.0, 3.0, 3.0, 2.0])
    assert oracle.topk(s, 2, idx=np.array([40, 10, 30, 20]), lib=lib).tolist() == [10, 30]


def pin_softmax_closed_forms(lib):
    rng = np.random.default_rng(13)
    v = _bf(rng.standard_normal((6, 128)))
    idx = np.array([0, 2, 5], dtype=np.int32)
    out = oracle.sparse_attention(np.full(3, 0.7), idx, v, lib=lib)
    assert np.allclose(out, _f(v)[idx].mean(axis=0), rtol=0, atol=1e-14)
    a, b = 1.25, -0.5
    w = 1.0 / (1.0 + math.exp(b - a))       # sigma(a - b)
    out = oracle.sparse_attention(np.array([a, b]), np.array([1, 4]), v, lib=lib)
    assert np.allclose(out, w * _f(v)[1] + (1 - w) * _f(v)[4], rtol=0, atol=1e-14)
    # shift invariance holds for the exact expression
    out2 = oracle.sparse_attention(np.array([a + 700.0, b + 700.0]), np.array([1, 4]), v, lib=lib)
    assert np.allclose(out, out2, rtol=0, atol=1e-12)


def pin_dense_equals_sdpa(lib):
    import torch
    rng = np.random.default_rng(14)
    L, d = 37, 128
    q, k, v = _bf(rng.standard_normal(d)), _bf(rng.standard_normal((L, d))), _bf(rng.standard_normal((L, d)))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(_f(q))[None, None, None], torch.from_numpy(_f(k))[None, None],
        torch.from_numpy(_f(v))[None, None])[0, 0, 0].numpy()
    assert np.allclose(oracle.dense_attention(q, k, v, lib=lib), ref, rtol=0, atol=1e-12)
    # Exact Top-K with K >= L selects every key and equals dense attention
    for K in (L, L + 5):
        sup, _, out = oracle.exact_one(q, k, v, L, K, lib=lib)
        assert sup.tolist() == list(range(L))
        assert np.allclose(out, ref, rtol=0, atol=1e-12)


def pin_softmax_merge(lib):
    rng = np.random.default_rng(15)
    v = _bf(rng.standard_normal((10, 128)))
    s = rng.standard_normal(10) * 3
    A, B = np.arange(0, 4), np.arange(4, 10)

    def part(ix):
        m = s[ix].max()
        Z = np.exp(s[ix] - m).sum()
        return m, Z, oracle.sparse_attention(s[ix], ix, v, lib=lib)

    m, Z, o = oracle.softmax_merge(*part(A), *part(B), lib=lib)
    assert np.allclose(o, oracle.sparse_attention(s, np.arange(10), v, lib=lib), rtol=0, atol=1e-13)
    assert math.isclose(m, s.max()) and math.isclose(Z, np.exp(s - s.max()).sum(), rel_tol=1e-13)


def pin_recall_closed_forms(lib):
    from scipy.spatial.distance import cosine
    rng = np.random.default_rng(16)
    qf = rng.standard_normal(128).astype(np.float32)
    q = _bf(qf)
    orth_v = np.zeros(128, np.float32)
    orth_v[0], orth_v[1] = -_f(q)[1], _f(q)[0]                # orthogonal to q exactly
    cached = np.stack([_bf(2 * _f(q)), _bf(-_f(q)), _bf(orth_v), q,
                       _bf(rng.standard_normal(128)), np.zeros(128, np.uint16)])
    rho, top, rmax = oracle.recall(q, cached, 3, lib=lib)
    assert rho[0] == 1.0 or abs(rho[0] - 1.0) < 1e-15
    assert abs(rho[1] + 1.0) < 1e-15 and abs(rho[2]) < 1e-15 and abs(rho[3] - 1.0) < 1e-15
    assert abs(rho[4] - (1.0 - cosine(_f(q), _f(cached[4])))) < 1e-12
    assert rho[5] == -math.inf                                   # zero-norm entry
    # ties (entries 0 and 3 both have rho 1) go to the older entry
    want = sorted(range(6), key=lambda c: (-rho[c], c))[:3]
    assert top.tolist() == want and top[0] == 0 and top[1] == 3
    assert rmax == max(rho)
    rho, top, rmax = oracle.recall(np.zeros(128, np.uint16), cached, 2, lib=lib)
    assert rmax == -math.inf
    rho, top, rmax = oracle.recall(q, cached[:1], 4, lib=lib)   # fewer entries than R
    assert top.tolist() == [0, -1, -1, -1]


def pin_candidates_set_union(lib):
    rng = np.random.default_rng(17)
    for trial in range(40):
        L = int(rng.integers(1, 300))
        W = int(rng.integers(0, 40))
        R = int(rng.integers(1, 5))
        K = int(rng.integers(1, 60))
        sups = [np.sort(rng.choice(L, size=min(K, L), replace=False)) for _ in range(R)]
        got = oracle.candidates(sups, L, W, lib=lib)
        want = sorted(set(range(max(0, L - W), L)).union(*[set(s.tolist()) for s in sups]))
        assert got.tolist() == want
        assert len(got) <= R * K + W


def _small_workload(seed, L0=96, steps=24, Hq=4, Hkv=2, K=8, C=6, d=128):
    rng = np.random.default_rng(seed)
    T = L0 + steps
    mu = rng.standard_normal((Hkv, 5, d)).astype(np.float32)
    z = rng.integers(0, 5, size=(Hkv, T))
    k = _bf(mu[np.arange(Hkv)[:, None], z] + 0.5 * rng.standard_normal((Hkv, T, d)))
    v = _bf(rng.standard_normal((Hkv, T, d)))
    g = rng.integers(0, 5, size=(Hq, C + steps))
    G = Hq // Hkv
    qf = 2 * mu[np.arange(Hq)[:, None] // G, g] + 0.3 * rng.standard_normal((Hq, C + steps, d))
    q = _bf(qf)
    return k, v, q[:, :C].copy(), q[:, C:].transpose(1, 0, 2).copy()


def _brute_exact(q, k, v, L, K):
    s = _f(k[:L]) @ _f(q) / math.sqrt(k.shape[1])
    order = sorted(range(L), key=lambda i: (-s[i], i))[:K]
    sup = sorted(order)
    w = np.exp(s[sup] - s[sup].max())
    return sup, (w[:, None] * _f(v)[sup]).sum(0) / w.sum()


def pin_init_cache_causal(lib):
    Hq, Hkv, K, C, L0 = 4, 2, 8, 6, 96
    k, v, qp, qd = _small_workload(18, L0=L0, Hq=Hq, Hkv=Hkv, K=K, C=C)
    # head 0's prompt queries all point at the final prompt key, which only the
    # last of them may see under causal prefill
    qp[0, :] = k[0, L0 - 1]
    st = oracle.init_cache(qp, k, L0, Hq, Hkv, K, C, lib=lib)
    assert L0 - 1 not in st.fsup[0, 0, :st.flen[0, 0]].tolist()
    assert L0 - 1 in st.fsup[0, C - 1, :st.flen[0, C - 1]].tolist()
    assert st.seq.tolist() == [0, C, 0]
    for h in range(Hq):
        for c in range(C):
            p = L0 - C + c
            sup, _ = _brute_exact(qp[h, c], k[h // (Hq // Hkv)], v[h // (Hq // Hkv)], p + 1, K)
            assert st.fsup[h, c, :st.flen[h, c]].tolist() == sup
            assert np.array_equal(st.fq[h, c], qp[h, c])


def _run(lib, tau, T_r, W, R=2, seed=19, steps=24, K=8, C=6, Hq=4, Hkv=2, L0=96):
    k, v, qp, qd = _small_workload(seed, L0=L0, steps=steps, Hq=Hq, Hkv=Hkv, K=K, C=C)
    st = oracle.init_cache(qp, k, L0, Hq, Hkv, K, C, lib=lib)
    res = []
    for t in range(steps):
        L = L0 + t + 1
        r = oracle.decode_step(st, qd[t], k, v, L, Hkv, W, R, T_r, tau, lib=lib)
        r["L"] = L
        res.append(r)
    return k, v, qd, res, st


def pin_degenerate_paths(lib):
    G = 2
    # tau > 1: every step is exact and equals brute-force Exact Top-K
    k, v, qd, res, _ = _run(lib, tau=1.5, T_r=0, W=4)
    for t, r in enumerate(res):
        assert (r["path"] == 1).all()
        for h in range(4):
            sup, out = _brute_exact(qd[t, h], k[h // G], v[h // G], r["L"], 8)
            assert r["sup"][h, :r["sup_len"][h]].tolist() == sup
            assert np.allclose(r["out"][h], out, rtol=0, atol=1e-12)
    # T_r = 1: every step is a refresh
    _, _, _, res, _ = _run(lib, tau=-2.0, T_r=1, W=4)
    assert all((r["path"] == 2).all() for r in res)
    # tau <= -1 and T_r = 0: every step reuses (cosines are >= -1)
    _, _, _, res, _ = _run(lib, tau=-1.0, T_r=0, W=4)
    assert all((r["path"] == 0).all() for r in res)
    # window covering the whole history: reuse steps equal exact steps
    k, v, qd, res, _ = _run(lib, tau=-1.0, T_r=0, W=10_000)
    for t, r in enumerate(res):
        assert (r["M"] == r["L"]).all()
        for h in range(4):
            sup, out = _brute_exact(qd[t, h], k[h // G], v[h // G], r["L"], 8)
            assert r["sup"][h, :r["sup_len"][h]].tolist() == sup
            assert np.allclose(r["out"][h], out, rtol=0, atol=1e-12)
    # refresh schedule: t_dec counts from 1, refresh at multiples of T_r
    _, _, _, res, _ = _run(lib, tau=-2.0, T_r=5, W=4, steps=21)
    for t, r in enumerate(res):
        assert (r["path"] == (2 if (t + 1) % 5 == 0 else 0)).all(), (t, r["path"])


def pin_rerank_recovers_exact(lib):
    """Eq. (11) remark: if S_t is inside A_t the reranked support equals S_t."""
    G, K, C = 2, 8, 6
    k, v, qp, qd = _small_workload(20, K=K, C=C)
    L = 96 + 1
    for h in range(4):
        st = oracle.init_cache(qp, k, 96, 4, 2, K, C, lib=lib)
        sup, out = _brute_exact(qd[0, h], k[h // G], v[h // G], L, K)
        # plant S_t (plus unrelated keys) in the newest entry, whose query is q_t itself
        slot = (int(st.seq[0]) - 1) % C
        planted = sorted(sup)                 # S_t itself, K entries
        st.fq[h, slot] = qd[0, h]
        st.fsup[h, slot, :] = -1
        st.fsup[h, slot, :len(planted)] = planted
        st.flen[h, slot] = len(planted)
        r = oracle.decode_step(st, qd[0], k, v, L, 2, 0, 1, 0, 0.99, lib=lib)
        assert r["path"][h] == 0 and r["rho_max"][h] == 1.0
        assert r["sup"][h, :r["sup_len"][h]].tolist() == sup
        assert np.allclose(r["out"][h], out, rtol=0, atol=1e-12)


def pin_fifo_contents(lib):
    C = 6
    k, v, qd, res, st = _run(lib, tau=0.8, T_r=7, W=4, C=C, steps=23)
    n = len(res)
    assert st.seq.tolist() == [(C + n) % C, C, n]
    for h in range(4):
        live = st.live(h)
        assert len(live) == C
        for c, (qbits, sup) in enumerate(live):
            t = n - C + c                      # the decode step that inserted entry c
            assert np.array_equal(qbits, qd[t, h])
            assert sup.tolist() == res[t]["sup"][h, :res[t]["sup_len"][h]].tolist()


def pin_recent_retrieval(lib):
    """The "recent-R retrieval" ablation (Table 3): the R newest live entries,
    newest first, with rho_max over them only -- checked on cached queries
    whose cosines with q are known in closed form (parallel, antiparallel,
    orthogonal), the most similar one being the oldest."""
    q = _bf([1, 0, 0, 0])
    cached = _bf([[3, 0, 0, 0],      # cosine  1, oldest
                  [0, 1, 0, 0],      # 0
                  [-2, 0, 0, 0],     # -1
                  [0, 0, 5, 0]])     # 0, newest
    rho = np.empty(4)
    top = np.empty(2, dtype=np.int32)
    ptrs = (__import__("ctypes").c_void_p * 4)(*[cached[c].ctypes.data for c in range(4)])
    rmax = lib.oracle_recall_recent(q.ctypes.data, ptrs, 4, 4, 2, rho.ctypes.data, top.ctypes.data)
    assert top.tolist() == [3, 2], top
    assert rmax == 0.0 and np.allclose(rho, [1.0, 0.0, -1.0, 0.0], rtol=0, atol=1e-15), (rmax, rho)
    top3 = np.empty(5, dtype=np.int32)
    rmax = lib.oracle_recall_recent(q.ctypes.data, ptrs, 4, 4, 5, rho.ctypes.data, top3.ctypes.data)
    assert top3.tolist() == [3, 2, 1, 0, -1] and rmax == 1.0, (top3, rmax)


def pin_fidelity(lib):
    """Support recall, retained mass and the two cosines of the fidelity
    criterion (§Experiments "Attention-support fidelity"; Eq. (2)): a
    hand-worked case, scipy's cosine for both cosines, and the invariants of
    identical and disjoint supports."""
    from scipy.spatial.distance import cosine
    d = 4
    q = _bf([2, 0, 0, 0])
    # scores q.k / sqrt(4): 1, 2, 0, -1
    k = _bf([[1, 0, 0, 0], [2, 0, 0, 0], [0, 0, 0, 0], [-1, 0, 0, 0]])
    o = np.array([1.0, 2.0, 0.0, -1.0])
    oh = np.array([2.0, 1.0, 1.0, 0.0])
    S, Sh = np.array([0, 1]), np.array([1, 2])
    m = oracle.fidelity(q, k, S, Sh, o, oh, lib=lib)
    e = math.e
    assert m[0] == 0.5, m
    # p over S = {0, 1} is (1, e) / (1 + e); S^ keeps key 1
    assert abs(m[1] - e / (1 + e)) < 1e-12, m
    assert abs(m[2] - (1 - cosine(o, oh))) < 1e-12, m
    p = np.array([1.0, e, 0.0, 0.0]) / (1 + e)              # over keys 0..3
    ph = np.array([0.0, e * e, 1.0, 0.0]) / (e * e + 1)       # softmax of (2, 0) on keys 1, 2
    assert abs(m[3] - (1 - cosine(p, ph))) < 1e-12, m
    # a shorter judged support: recall still counts against |S|
    m = oracle.fidelity(q, k, S, np.array([1]), o, oh, lib=lib)
    assert m[0] == 0.5 and abs(m[1] - e / (1 + e)) < 1e-12, m
    # identical supports and outputs: everything 1; disjoint supports: 0
    rng = np.random.default_rng(5)
    kk = _bf(rng.standard_normal((40, d)))
    qq = _bf(rng.standard_normal(d))
    oo = rng.standard_normal(d)
    full = np.arange(0, 40, 3)
    m = oracle.fidelity(qq, kk, full, full, oo, oo, lib=lib)
    assert np.allclose(m, 1.0, rtol=0, atol=1e-12), m
    m = oracle.fidelity(qq, kk, np.arange(0, 20), np.arange(20, 40), oo, -oo, lib=lib)
    assert m[0] == 0.0 and m[1] == 0.0 and m[3] == 0.0 and abs(m[2] + 1.0) < 1e-12, m


def pin_exact_step_batched(lib):
    """The batched Exact Top-K step (Eqs. (1), (4), (12)) against brute force
    per (sequence, query head): ragged lengths (one shorter than K), query
    head h reading KV head h // G of its own sequence, -1 padding past the
    support, the K-th score."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, T, d, K = 2, 4, 2, 70, 128, 9
    G = Hq // Hkv
    q = _bf(rng.standard_normal((B, Hq, d)))
    k = _bf(rng.standard_normal((B, Hkv, T, d)))
    v = _bf(rng.standard_normal((B, Hkv, T, d)))
    L = np.array([70, 6], np.int32)
    sup, sup_len, kth, out = oracle.exact_step(q, k, v, L, K, lib=lib)
    for b in range(B):
        for h in range(Hq):
            want_sup, want_out = _brute_exact(q[b, h], k[b, h // G], v[b, h // G], int(L[b]), K)
            n = int(sup_len[b, h])
            assert sup[b, h, :n].tolist() == want_sup, (b, h)
            assert (sup[b, h, n:] == -1).all(), (b, h)
            assert np.allclose(out[b, h], want_out, rtol=0, atol=1e-12), (b, h)
            s = _f(k[b, h // G, :L[b]]) @ _f(q[b, h]) / math.sqrt(d)
            assert abs(kth[b, h] - np.sort(s)[::-1][min(K, int(L[b])) - 1]) < 1e-12, (b, h)


def pin_attention_on_support_numpy(lib):
    """Eqs. (10) + (12) on a given support (unsorted, arbitrary rows): a numpy
    float64 softmax over the gathered K rows weighting the gathered V rows."""
    rng = np.random.default_rng(22)
    d = 128
    q = _bf(rng.standard_normal(d))
    k = _bf(rng.standard_normal((50, d)))
    v = _bf(rng.standard_normal((50, d)))
    for sup in ([3, 17, 4, 49, 0, 22], [31], list(range(50))):
        sup = np.array(sup, np.int32)
        s = _f(k)[sup] @ _f(q) / math.sqrt(d)
        w = np.exp(s - s.max())
        ref = (w / w.sum()) @ _f(v)[sup]
        got = oracle.attention_on_support(q, k, v, sup, lib=lib)
        assert np.allclose(got, ref, rtol=0, atol=1e-13), sup


def pin_overlap_coverage(lib):
    """Eq. (2) against Python set arithmetic (denominator K, also for a
    support shorter than K) and Eq. (3) with preceding queries whose cosines
    to q are known in closed form, so the R most similar are fixed."""
    rng = np.random.default_rng(23)
    assert oracle.overlap([1, 2, 3, 4], [3, 4, 5, 6], 4, lib=lib) == 0.5
    assert oracle.overlap([0, 1], [1], 4, lib=lib) == 0.25
    for trial in range(30):
        K = int(rng.integers(1, 40))
        L = int(rng.integers(1, 80))
        a = np.sort(rng.choice(L, min(K, L), replace=False))
        b = np.sort(rng.choice(L, min(K, L), replace=False))
        assert oracle.overlap(a, b, K, lib=lib) == len(set(a.tolist()) & set(b.tolist())) / K
    q = _bf([1, 0, 0, 0])
    prev_q = _bf([[0, 1, 0, 0],      # cosine 0, oldest
                  [2, 0, 0, 0],      # 1
                  [-1, 0, 0, 0],     # -1
                  [1, 1, 0, 0],      # 1/sqrt(2)
                  [0, 0, 3, 0]])     # 0, newest
    prev_S = [[0, 1, 2], [10, 11, 12, 13], [20, 21], [12, 13, 14, 30], [40, 41]]
    St = [0, 11, 13, 14, 20, 30, 41, 50]
    K = 8
    for R, want in ((1, [1]), (2, [1, 3]), (3, [1, 3, 0]), (4, [1, 3, 0, 4]), (6, [1, 3, 0, 4, 2, -1])):
        cov, chosen = oracle.coverage(q, prev_q, prev_S, St, R, K, lib=lib)
        assert chosen.tolist() == want, (R, chosen)
        U = set().union(*[set(prev_S[c]) for c in want if c >= 0])
        assert cov == len(set(St) & U) / K, (R, cov)


def pin_window_zero_and_no_fallback(lib):
    """The W = 0 and tau = -inf ablations (Table 3): every step reuses (no
    cosine is below -inf), the candidate set is exactly the union of the
    retrieved entries' supports with no recent window, and the support and
    output are the brute-force Top-K and softmax over that set."""
    Hq, Hkv, K, C, L0, R = 4, 2, 8, 6, 96, 2
    G = Hq // Hkv
    k, v, qp, qd = _small_workload(24, L0=L0, Hq=Hq, Hkv=Hkv, K=K, C=C)
    st = oracle.init_cache(qp, k, L0, Hq, Hkv, K, C, lib=lib)
    for t in range(len(qd)):
        L = L0 + t + 1
        pre = st.copy()
        r = oracle.decode_step(st, qd[t], k, v, L, Hkv, 0, R, 0, -math.inf, lib=lib)
        assert (r["path"] == 0).all(), (t, r["path"])
        for h in range(Hq):
            live = pre.live(h)
            qh = _f(qd[t, h])
            cos = [float(_f(x) @ qh / (np.linalg.norm(_f(x)) * np.linalg.norm(qh))) for x, _ in live]
            top = sorted(range(len(live)), key=lambda c: (-cos[c], c))[:R]
            A = sorted(set().union(*[set(live[c][1].tolist()) for c in top]))
            assert r["cand"][h, :r["M"][h]].tolist() == A, (t, h)
            s = _f(k[h // G])[A] @ qh / math.sqrt(128)
            order = sorted(range(len(A)), key=lambda j: (-s[j], A[j]))[:K]
            sup = sorted(A[j] for j in order)
            assert r["sup"][h, :r["sup_len"][h]].tolist() == sup, (t, h)
            ss = _f(k[h // G])[sup] @ qh / math.sqrt(128)
            w = np.exp(ss - ss.max())
            assert np.allclose(r["out"][h], (w / w.sum()) @ _f(v[h // G])[sup], rtol=0, atol=1e-12), (t, h)


ALL_PINS = [pin_hand_worked_exact, pin_hand_worked_reuse, pin_scores_library_and_closed_form,
            pin_topk_brute_force, pin_softmax_closed_forms, pin_dense_equals_sdpa,
            pin_softmax_merge, pin_recall_closed_forms, pin_candidates_set_union,
            pin_init_cache_causal, pin_degenerate_paths, pin_rerank_recovers_exact,
            pin_fifo_contents, pin_fidelity, pin_recent_retrieval, pin_exact_step_batched,
            pin_attention_on_support_numpy, pin_overlap_coverage, pin_window_zero_and_no_fallback]
