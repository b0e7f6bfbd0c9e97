"""ReTopK decode steps through the C ABI against the fp64 oracle (GPU).

State-forced protocol: before a checked step the GPU's cache state is
exported and handed to the oracle, which computes the same step from that
state; path, rho_max, retrieved entries, candidate set, support, output and
the cache slot written are then compared (tolerances in tests/parity.py).
This keeps one legal near-tie swap from turning every later step into a
mismatch.  Unchecked steps still run on the GPU, so the state being checked
is the GPU's own trajectory.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import compare_decode_step, out_close
from top_sparse_attention_exact_gb300 import synth
from top_sparse_attention_exact_gb300.retopk import RetopkError
from top_sparse_attention_exact_gb300.runner import DecodeRun, ExactRun

pytestmark = pytest.mark.gpu


def run_checked(w, check_steps=None, arrays=None, max_len=None, cluster=0):
    dr = DecodeRun(w, arrays=arrays, max_len=max_len, cluster=cluster)
    k, v, qd = dr.k_host, dr.v_host, dr.qd_host
    errs, agg = [], dict(path_band=0, topR_band=0, swaps=0, heads=0)
    paths = []
    for t in range(w.steps):
        check = check_steps is None or (t + 1) in check_steps
        if check:
            pre = dr.ctx.retopk_export_state()
        dr.step(t)
        if check:
            torch.cuda.synchronize()
            post = dr.ctx.retopk_export_state()
            diag = dr.ctx.retopk_get_diagnostics()
            paths.append(diag["path"].copy())
            L = dr.seqlens.cpu().numpy()
            out = dr.out.cpu().numpy().view(np.uint16)
            e, st = compare_decode_step(pre, post, diag, qd[t], k, v, L, w, out, where=f"{w.name} t{t + 1}")
            errs += e
            for key in agg:
                agg[key] += st[key]
    assert dr.ctx.retopk_get_status() == 0
    # band exemptions (path or retrieval decided within 1e-4 of a tie) are
    # reported, and must stay rare: at most 1 % of the checked heads
    print(f"{w.name}: {agg['heads']} heads checked, path_band {agg['path_band']}, "
          f"topR_band {agg['topR_band']}, near-tie support swaps {agg['swaps']}")
    assert agg["path_band"] + agg["topR_band"] <= max(1, agg["heads"] // 100), agg
    return dr, errs, agg, paths


def test_tiny_full_trajectory():
    w = synth.WORKLOADS["tiny_1h_2k"]
    dr, errs, agg, paths = run_checked(w)
    assert not errs, "\n".join(errs[:20])
    assert agg["path_band"] == 0 and agg["topR_band"] == 0, agg   # no near-tie on this case
    p = np.concatenate(paths)
    # refresh exactly at t_dec = 16, 32, 48, 64
    assert [i + 1 for i, x in enumerate(p) if x == 2] == [16, 32, 48, 64]
    assert (p == 0).sum() > 0 and (p == 1).sum() > 0


def test_tiny_free_running_matches_oracle():
    """Both sides run their own trajectory; on this case no near-ties occur."""
    w = synth.WORKLOADS["tiny_1h_2k"]
    dr = DecodeRun(w)
    k, v, qp, qd = dr.k_host, dr.v_host, dr.qp_host, dr.qd_host
    st = oracle.init_cache(qp[0], k[0], w.L0, w.Hq, w.Hkv, w.K, w.C)
    g0 = dr.ctx.retopk_export_state()
    assert np.array_equal(g0["fifo_len"][0], st.flen)
    for h in range(w.Hq):
        for c in range(w.C):
            n = st.flen[h, c]
            assert np.array_equal(g0["fifo_sup"][0, h, c, :n], st.fsup[h, c, :n])
    for t in range(w.steps):
        dr.step(t)
        r = oracle.decode_step(st, qd[t, 0], k[0], v[0], w.L0 + t + 1, w.Hkv, w.W, w.R, w.T_r, w.tau,
                               recent=w.recent)
        diag = dr.ctx.retopk_get_diagnostics()
        assert diag["path"].tolist() == r["path"].tolist(), t
        assert diag["support"][0, :diag["sup_len"][0]].tolist() == r["sup"][0, :r["sup_len"][0]].tolist(), t
        ok, mx, rel = out_close(diag["out_f32"][0], r["out"][0])
        assert ok, (t, mx, rel)
    g = dr.ctx.retopk_export_state()
    assert g["seq"][0].tolist() == st.seq.tolist()
    assert np.array_equal(g["fifo_q"][0], st.fq)


def test_init_cache_matches_oracle_qwen_shape():
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], steps=1)
    dr = DecodeRun(w)
    g = dr.ctx.retopk_export_state()
    st = oracle.init_cache(dr.qp_host[0], dr.k_host[0], w.L0, w.Hq, w.Hkv, w.K, w.C)
    assert g["seq"][0].tolist() == [0, w.C, 0]
    assert np.array_equal(g["fifo_q"][0], st.fq)
    from parity import support_ok
    for h in range(w.Hq):
        for c in range(w.C):
            n = st.flen[h, c]
            p = w.L0 - w.C + c
            kr = dr.k_host[0, h // 7]
            got = g["fifo_sup"][0, h, c, :g["fifo_len"][0, h, c]]
            if not np.array_equal(got, st.fsup[h, c, :n]):
                s = oracle.scores(dr.qp_host[0, h, c], kr[:p + 1])
                kth = np.sort(s)[::-1][n - 1]
                ok, msg = support_ok(dr.qp_host[0, h, c], kr, got, st.fsup[h, c, :n], kth)
                assert ok, (h, c, msg)


def test_qwen_16k_all_steps():
    w = synth.WORKLOADS["qwen7b_16k"]
    dr, errs, agg, paths = run_checked(w)
    assert not errs, "\n".join(errs[:20])
    c = dr.ctx.retopk_get_counters()
    assert c["reuse"] + c["fallback"] + c["refresh"] == w.steps * w.Hq
    assert c["refresh"] == (w.steps // w.T_r) * w.Hq
    assert c["max_M"] <= w.R * w.K + w.W


@pytest.mark.parametrize("name", ["qwen7b_32k", "qwen7b_64k"])
def test_qwen_longer_sampled(name):
    w = synth.WORKLOADS[name]
    steps = set(range(1, 9)) | set(range(125, 133)) | {200, 255, 256}
    dr, errs, agg, paths = run_checked(w, check_steps=steps)
    assert not errs, "\n".join(errs[:20])


def test_headline_128k_sampled():
    w = synth.WORKLOADS["qwen7b_128k"]
    steps = {1, 2, 3, 64, 127, 128, 129, 256, 384, 511, 512}
    dr, errs, agg, paths = run_checked(w, check_steps=steps)
    assert not errs, "\n".join(errs[:20])


@pytest.fixture(scope="module")
def sweep_arrays():
    w = synth.batched_sweep(256, 0.70, steps=136)
    return w, synth.generate(w)


@pytest.mark.parametrize("K", [256, 1024, 2048])
@pytest.mark.parametrize("tau", [0.70, 0.95])
def test_batched_sweep_sampled(sweep_arrays, K, tau):
    # 136 decode steps of the batch-16 64K sweep (a refresh at step 128),
    # checked at nine sampled steps
    w0, arrays = sweep_arrays
    w = synth.scaled(w0, K=K, tau=tau, name=f"sweep_K{K}_tau{tau}")
    dr, errs, agg, paths = run_checked(w, check_steps={1, 2, 17, 40, 77, 101, 127, 128, 136}, arrays=arrays)
    assert not errs, "\n".join(errs[:20])
    p = np.concatenate(paths)
    assert (p[-2 * w.B * w.Hq:-w.B * w.Hq] == 2).all()   # step 128 refreshes every head


@pytest.mark.parametrize("cluster", [1, 2, 4])
def test_back_end_cluster_sizes(cluster):
    # the decode step's back end with 1, 2 or 4 CTAs per head (a sequence of
    # 28 heads gets 8): every checked step against the oracle, and the same
    # paths and supports as the 8-CTA context on the same inputs
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=4096, steps=12, T_r=5, name=f"cluster{cluster}")
    arrays = synth.generate(w)
    steps = {1, 2, 5, 6, 9, 10, 12}
    dr, errs, agg, paths = run_checked(w, check_steps=steps, arrays=arrays, cluster=cluster)
    assert not errs, "\n".join(errs[:20])
    ref, errs8, _, paths8 = run_checked(w, check_steps=steps, arrays=arrays, cluster=8)
    assert not errs8
    p = np.concatenate(paths)
    assert (p == 0).any() and (p != 0).any()
    assert np.array_equal(p, np.concatenate(paths8))
    d, d8 = dr.ctx.retopk_get_diagnostics(), ref.ctx.retopk_get_diagnostics()
    assert np.array_equal(d["support"], d8["support"]) and np.array_equal(d["M"], d8["M"])
    for h in np.nonzero(d["path"] == 0)[0]:   # A_t of the reuse heads (exact heads list per CTA)
        assert np.array_equal(d["cand"][h, :d["M"][h]], d8["cand"][h, :d["M"][h]]), h
    o = synth.bf16_bits_to_f32(dr.out.cpu().numpy().view(np.uint16))
    o8 = synth.bf16_bits_to_f32(ref.out.cpu().numpy().view(np.uint16)).astype(np.float64)
    for h in range(w.Hq):   # the same support, partial sums grouped differently
        assert out_close(o[0, h], o8[0, h])[0], h


@pytest.mark.parametrize("variant", ["W0", "no_fallback"])
def test_ablation_parity(variant):
    # the W = 0 (no recent window) and tau = -inf (no similarity fallback)
    # ablations of Table 3 against the oracle, every step
    kw = dict(W=0) if variant == "W0" else dict(tau=-float("inf"), T_r=0)
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], steps=40, name=f"qwen7b_16k_{variant}", **kw)
    dr, errs, agg, paths = run_checked(w)
    assert not errs, "\n".join(errs[:20])
    p = np.concatenate(paths)
    if variant == "no_fallback":
        assert (p == 0).all()
    else:
        assert (p == 0).sum() > 0


def _degenerate(tau, T_r, W, steps=12):
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=3000, steps=steps, tau=tau, T_r=T_r, W=W,
                     name=f"deg_tau{tau}_Tr{T_r}_W{W}")
    return w


def test_short_history_ranks_without_keys():
    # L <= 64: the candidate bitmap's slices are 32 positions, so ranks 2..7 of
    # each cluster own no position and contribute empty candidate lists
    w = synth.scaled(synth.WORKLOADS["tiny_1h_2k"], L0=40, steps=24, K=16, C=8, W=8, R=2, tau=0.3,
                     T_r=0, n_topics=4, run=8, name="tiny_short_history")
    dr, errs, agg, paths = run_checked(w)
    assert not errs, "\n".join(errs[:20])
    assert (np.concatenate(paths) == 0).sum() >= 12


def test_largest_max_len_short_history():
    # max_len = 2^23: the reuse path's bitmap slice is 2^20 positions (128 KB)
    # per CTA, the back end runs one CTA per SM; the history itself is short
    w = synth.scaled(synth.WORKLOADS["tiny_1h_2k"], L0=4096, steps=16, Hq=2, K=128, tau=0.5, T_r=8,
                     name="tiny_maxlen_2p23")
    dr, errs, agg, paths = run_checked(w, max_len=1 << 23)
    assert not errs, "\n".join(errs[:20])
    assert (np.concatenate(paths) == 0).sum() >= 4


def test_qwen_1m_prefilter_sampled():
    # 1M keys, 28 heads: a CTA's eighth of an exact head's scores spans
    # several windows, so decode steps run the exact-head prefilter; mixed
    # steps and the refresh at step 128 (every head exact) against the oracle
    w = synth.scaled(synth.WORKLOADS["qwen7b_1m"], steps=130, name="qwen7b_1m_pf")
    dr, errs, agg, paths = run_checked(w, check_steps={1, 2, 3, 4, 5, 6, 127, 128, 129, 130})
    assert not errs, "\n".join(errs[:20])
    p = np.concatenate(paths)
    assert ((p != 0).sum() > 0) and (p[-3 * w.Hq:-2 * w.Hq] == 2).all()


def test_prefiltered_heads_with_massive_ties():
    # 160K keys: one repeated key row at every third position, zero rows
    # elsewhere, so the history's scores take two values.  Exact heads at this
    # length run the prefilter (two windows per CTA), and tens of thousands of
    # keys share the 19-bit prefix: more final candidates than the select
    # stages, so the window lists are compacted in place for the global
    # select.  Every step against the oracle (ties to the lower index).
    w = synth.scaled(synth.WORKLOADS["tiny_1h_2k"], L0=160_000, steps=6, Hq=4, K=512, tau=1.5, T_r=0,
                     name="tiny_pf_ties")
    arrays = synth.generate(w)
    k = arrays[0]
    row = k[0, 0, 1].copy()
    k[:, :, :w.L0] = 0
    k[:, :, :w.L0:3] = row
    dr, errs, agg, paths = run_checked(w, arrays=arrays)
    assert not errs, "\n".join(errs[:20])
    assert (np.concatenate(paths) == 1).all()
    diag = dr.ctx.retopk_get_diagnostics()
    assert (diag["sup_len"] == w.K).all()


def test_long_history_split_bitmap():
    # 3M keys: each rank's bitmap slice covers ~393K positions and the
    # retrieved supports spread over all of them
    w = synth.scaled(synth.WORKLOADS["tiny_1h_2k"], L0=3_000_000, steps=8, K=512, tau=0.3, T_r=0,
                     n_topics=16, run=256, name="tiny_3m")
    dr, errs, agg, paths = run_checked(w)
    assert not errs, "\n".join(errs[:20])
    assert (np.concatenate(paths) == 0).sum() >= 4
    diag = dr.ctx.retopk_get_diagnostics()
    span = ((w.L0 + w.steps + 7) // 8 + 31) // 32 * 32
    ranks = {int(i) // span for i in diag["support"][0] if i >= 0}
    assert len(ranks) >= 4, ranks


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_host_buffer_step_matches_device_step():
    # retopk_decode_step_host (host inputs/outputs, graph replay) against
    # retopk_decode_step_kv on a second context with the same inputs: identical
    # outputs and supports every step; then a second pair of caches (the graph
    # is captured again for the new binding)
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=4096, steps=20, T_r=8, name="host_api")
    arrays = synth.generate(w)
    dev_run, host_run = DecodeRun(w, arrays=arrays), DecodeRun(w, arrays=arrays)
    qh = torch.from_numpy(np.ascontiguousarray(arrays[3]).view(np.int16))
    kh = torch.from_numpy(np.ascontiguousarray(arrays[0][:, :, w.L0:].transpose(2, 0, 1, 3)).view(np.int16))
    vh = torch.from_numpy(np.ascontiguousarray(arrays[1][:, :, w.L0:].transpose(2, 0, 1, 3)).view(np.int16))
    out_h = torch.zeros((w.B, w.Hq, w.d), dtype=torch.int16).pin_memory()
    for t in range(w.steps):
        if t == 12:   # move the host run's caches to new allocations
            host_run.k_cache, host_run.v_cache = host_run.k_cache.clone(), host_run.v_cache.clone()
            host_run.seqlens = host_run.seqlens.clone()
        dev_run.step(t)
        src_q = qh[t] if t % 2 else qh[t].clone().pin_memory()   # pageable and pinned inputs
        host_run.ctx.retopk_decode_step_host(kh[t], vh[t], src_q, host_run.k_cache, host_run.v_cache,
                                             host_run.seqlens, out_h)
        torch.cuda.synchronize()
        assert torch.equal(out_h, dev_run.out.cpu()), t
        da, db = dev_run.ctx.retopk_get_diagnostics(), host_run.ctx.retopk_get_diagnostics()
        for key in ("path", "support", "sup_len", "M"):
            assert np.array_equal(da[key], db[key]), (t, key)
    assert torch.equal(host_run.k_cache, dev_run.k_cache) and torch.equal(host_run.seqlens, dev_run.seqlens)
    assert host_run.ctx.retopk_get_status() == 0
    # a synchronous host-buffer call refuses a capturing stream (and leaves the capture intact)
    s, g = torch.cuda.Stream(), torch.cuda.CUDAGraph()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            with pytest.raises(RetopkError):
                host_run.ctx.retopk_decode_step_host(kh[0], vh[0], qh[0], host_run.k_cache, host_run.v_cache,
                                                     host_run.seqlens, out_h, s)
    torch.cuda.synchronize()


def test_tau_above_one_equals_exact_every_step():
    w = _degenerate(1.5, 0, 32)
    dr = DecodeRun(w)
    ex = ExactRun(dr)
    for t in range(w.steps):
        dr.step(t)
        diag = dr.ctx.retopk_get_diagnostics()
        assert (diag["path"] == 1).all()
        ex.step(dr.q_dec[t])
        torch.cuda.synchronize()
        assert torch.equal(ex.out, dr.out)
        assert np.array_equal(ex.idx.view(-1, w.K).cpu().numpy(), diag["support"])


def test_window_covering_history_equals_exact():
    w = _degenerate(-2.0, 0, 4096)          # W >= L for every step (L <= 3012)
    dr = DecodeRun(w)
    ex = ExactRun(dr)
    for t in range(w.steps):
        dr.step(t)
        diag = dr.ctx.retopk_get_diagnostics()
        assert (diag["path"] == 0).all()
        assert (diag["M"] == w.L0 + t + 1).all()
        ex.step(dr.q_dec[t])
        torch.cuda.synchronize()
        # the rerank scores (CUDA cores) and the scan scores (tensor cores) may
        # round differently, so near-ties may swap; outputs agree to tolerance
        from parity import support_ok
        L = w.L0 + t + 1
        eidx = ex.idx.view(-1, w.K).cpu().numpy()
        for h in range(w.Hq):
            kr = dr.k_host[0, h // 7]
            s = oracle.scores(dr.qd_host[t, 0, h], kr[:L])
            kth = float(np.sort(s)[::-1][w.K - 1])
            ok, msg = support_ok(dr.qd_host[t, 0, h], kr, diag["support"][h], eidx[h], kth)
            assert ok, (t, h, msg)
        a = synth.bf16_bits_to_f32(ex.out.cpu().numpy().view(np.uint16))
        b = synth.bf16_bits_to_f32(dr.out.cpu().numpy().view(np.uint16))
        ok, mx, rel = out_close(a, b)
        assert ok, (t, mx, rel)


def test_refresh_every_step_and_always_reuse():
    dr = DecodeRun(_degenerate(0.85, 1, 32))
    for t in range(dr.w.steps):
        dr.step(t)
        assert (dr.ctx.retopk_get_diagnostics()["path"] == 2).all()
    dr = DecodeRun(_degenerate(-1.0, 0, 32))
    for t in range(dr.w.steps):
        dr.step(t)
        assert (dr.ctx.retopk_get_diagnostics()["path"] == 0).all()


def test_reuse_select_with_heavy_score_ties():
    # keys drawn from 3 distinct rows (scores take 3 values per query): the
    # reranked candidates tie in large groups, so the reuse path's Top-K
    # resolves them by index beyond the warp-ranked case
    w = synth.scaled(synth.WORKLOADS["tiny_1h_2k"], steps=12, tau=-1.0, T_r=0)
    k, v, qp, qd = synth.generate(w)
    rng = np.random.default_rng(11)
    rows = synth.random_bf16(rng, (3, w.d))
    k = rows[rng.integers(0, 3, size=k.shape[2])][None, None].copy()
    dr, errs, agg, paths = run_checked(w, arrays=(k, v, qp, qd))
    assert not errs, "\n".join(errs[:20])
    assert (np.concatenate(paths) == 0).all()


def test_recent_retrieval_ablation_against_oracle():
    # Table 3's "recent-R retrieval": the R newest cache entries, rho_max over them
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], steps=24, recent=True, name="qwen7b_16k_recentR")
    dr, errs, agg, paths = run_checked(w, check_steps=set(range(2, 25, 3)))
    assert not errs, "\n".join(errs[:20])
    topR = dr.ctx.retopk_get_diagnostics()["topR"]
    assert (topR[:, 0] == w.C - 1).all() and (topR[:, 1] == w.C - 2).all()


def test_fidelity_diagnostics_match_oracle():
    # exact shadow: after each checked decode step, the stateless exact step on
    # the same query and caches gives S_t and o_t; the library's fidelity
    # kernel must agree with the oracle's fp64 definitions per head
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], steps=20)
    dr = DecodeRun(w)
    ex = ExactRun(dr)
    seen_reuse = 0
    for t in range(w.steps):
        dr.step(t)
        if t % 4 != 3:
            continue
        ex.step(dr.q_dec[t])
        m = dr.ctx.retopk_fidelity(dr.q_dec[t], dr.k_cache, ex.idx, ex.out, dr.out).cpu().numpy()
        torch.cuda.synchronize()
        diag = dr.ctx.retopk_get_diagnostics()
        S = ex.idx.cpu().numpy()
        o = synth.bf16_bits_to_f32(ex.out.cpu().numpy().view(np.uint16)).astype(np.float64)
        oh = synth.bf16_bits_to_f32(dr.out.cpu().numpy().view(np.uint16)).astype(np.float64)
        L = int(dr.seqlens[0])
        G = w.Hq // w.Hkv
        for h in range(w.Hq):
            ref = oracle.fidelity(dr.qd_host[t, 0, h], dr.k_host[0, h // G, :L], S[0, h], diag["support"][h],
                                  o[0, h], oh[0, h])
            got = m[0, h]
            assert got[0] == ref[0], (t, h, got, ref)
            assert np.allclose(got[1:], ref[1:], rtol=0, atol=2e-3), (t, h, got, ref)
            if diag["path"][h] != 0:   # an exact-path head used the exact support
                assert got[0] == 1.0 and abs(got[1] - 1.0) < 1e-5, (t, h, got)
            else:
                seen_reuse += 1
    assert seen_reuse > 0


def test_support_overlap_and_coverage_match_oracle():
    # Eqs. (2)-(3) on the GPU against the oracle: random ascending supports
    # (some shorter than K, -1 padded), then the decode loop's own quantities
    # -- the Exact Top-K support of q_t and the exact supports of the R cached
    # queries the decision retrieved -- against oracle.coverage, which picks
    # the R most similar preceding queries itself
    from top_sparse_attention_exact_gb300 import retopk
    rng = np.random.default_rng(31)
    rows, R, K, L = 40, 4, 64, 300
    S = np.full((rows, K), -1, np.int32)
    O = np.full((rows, R, K), -1, np.int32)
    for i in range(rows):
        n = K if i % 3 else int(rng.integers(1, K))
        S[i, :n] = np.sort(rng.choice(L, n, replace=False))
        for r in range(R):
            m = K if (i + r) % 4 else int(rng.integers(0, K))
            O[i, r, :m] = np.sort(rng.choice(L, m, replace=False))
    got = retopk.support_overlap(torch.from_numpy(S).cuda(), torch.from_numpy(O).cuda()).cpu().numpy()
    for i in range(rows):
        U = oracle.candidates([O[i, r][O[i, r] >= 0] for r in range(R)], 0, 0)
        assert abs(got[i, 0] - oracle.overlap(S[i], O[i, 0], K)) < 1e-6, i
        assert abs(got[i, 1] - oracle.overlap(S[i], U, K)) < 1e-6, i
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], steps=44, T_r=0)
    dr = DecodeRun(w)
    ex = ExactRun(dr)
    hist, checked = [], 0
    for t in range(w.steps):
        pre = dr.ctx.retopk_export_state()
        dr.step(t)
        ex.step(dr.q_dec[t])
        torch.cuda.synchronize()
        hist.append(ex.idx.cpu().numpy().reshape(w.Hq, w.K).copy())
        if t < w.C:
            continue   # the cache still holds prompt entries (no exact shadow for them)
        topR = dr.ctx.retopk_get_diagnostics()["topR"]
        others = np.stack([np.stack([hist[t - w.C + int(c)][h] for c in topR[h]]) for h in range(w.Hq)])
        got = retopk.support_overlap(ex.idx.view(w.Hq, w.K), torch.from_numpy(others).cuda()).cpu().numpy()
        cs = oracle.state_from_export(pre, 0, w.K)
        for h in range(w.Hq):
            live = cs.live(h)
            prev_q = np.stack([x for x, _ in live])
            prev_S = [hist[t - w.C + c][h] for c in range(len(live))]
            cov, chosen = oracle.coverage(dr.qd_host[t, 0, h], prev_q, prev_S, hist[t][h], w.R, w.K)
            if sorted(chosen.tolist()) != sorted(topR[h].tolist()):
                continue   # a near-tie in the retrieval (checked elsewhere)
            assert abs(got[h, 1] - cov) < 1e-6, (t, h, got[h], cov)
            assert abs(got[h, 0] - oracle.overlap(hist[t][h], prev_S[chosen[0]], w.K)) < 1e-6, (t, h)
            checked += 1
    assert checked >= 10 * w.Hq


def test_graph_replay_matches_eager():
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], steps=40, T_r=16)
    a = DecodeRun(w)
    b = DecodeRun(w, arrays=(a.k_host, a.v_host, a.qp_host, a.qd_host))
    b.capture()
    for t in range(w.steps):
        a.step(t)
        b.replay(t)
        torch.cuda.synchronize()
        assert torch.equal(a.out, b.out), t
    sa, sb = a.ctx.retopk_export_state(), b.ctx.retopk_export_state()
    for key in sa:
        assert np.array_equal(sa[key], sb[key]), key
    assert torch.equal(a.seqlens, b.seqlens)


def test_fused_append_matches_separate_calls():
    # retopk_decode_step_kv == retopk_append_kv + retopk_decode_step, bit for bit,
    # eagerly and as a replayed graph, including the K/V caches and lengths
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], steps=24, T_r=8)
    a = DecodeRun(w, fused=False)
    arrays = (a.k_host, a.v_host, a.qp_host, a.qd_host)
    b = DecodeRun(w, arrays=arrays, fused=True)
    c = DecodeRun(w, arrays=arrays, fused=True)
    c.capture()
    for t in range(w.steps):
        a.step(t)
        b.step(t)
        c.replay(t)
        torch.cuda.synchronize()
        assert torch.equal(a.out, b.out) and torch.equal(a.out, c.out), t
    for x in (b, c):
        sa, sx = a.ctx.retopk_export_state(), x.ctx.retopk_export_state()
        for key in sa:
            assert np.array_equal(sa[key], sx[key]), key
        assert torch.equal(a.seqlens, x.seqlens)
        assert torch.equal(a.k_cache, x.k_cache) and torch.equal(a.v_cache, x.v_cache)


def test_layer_stack_shared_scratch_matches_per_layer_steps():
    # several layer contexts (own caches, own query-support state) sharing one
    # per-step scratch, stepped as one captured graph per token with the layers
    # back to back, against each layer stepped eagerly with its own full
    # workspace: identical outputs every step and identical final states
    from top_sparse_attention_exact_gb300 import retopk
    w0 = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=4096, steps=24, T_r=8, name="stack")
    n_layers = 4
    ws = [synth.scaled(w0, seeds=(50 + i,)) for i in range(n_layers)]
    arrays = [synth.generate(w) for w in ws]
    nb = retopk.scratch_bytes(w0.B, w0.Hq, w0.Hkv, w0.max_len, w0.K, w0.C, w0.W, w0.R, w0.T_r, w0.tau)
    scratch = torch.empty(nb + 256, dtype=torch.uint8, device="cuda")
    stack = [DecodeRun(w, arrays=a, scratch=scratch) for w, a in zip(ws, arrays)]
    ref = [DecodeRun(w, arrays=a) for w, a in zip(ws, arrays)]
    bufs = [(torch.empty_like(r.q_dec[0]), torch.empty_like(r.k_new[0]), torch.empty_like(r.v_new[0])) for r in stack]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for r, (qb, kb, vb) in zip(stack, bufs):
                r.ctx.retopk_decode_step_kv(kb, vb, qb, r.k_cache, r.v_cache, r.seqlens, r.out, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    paths = []
    for t in range(w0.steps):
        for r, (qb, kb, vb) in zip(stack, bufs):
            qb.copy_(r.q_dec[t])
            kb.copy_(r.k_new[t])
            vb.copy_(r.v_new[t])
        g.replay()
        for r in ref:
            r.step(t)
            paths.append(r.ctx.retopk_get_diagnostics()["path"].copy())
        torch.cuda.synchronize()
        for i in range(n_layers):
            assert torch.equal(stack[i].out, ref[i].out), (t, i)
    for i in range(n_layers):
        sa, sb = stack[i].ctx.retopk_export_state(), ref[i].ctx.retopk_export_state()
        for key in sa:
            assert np.array_equal(sa[key], sb[key]), (i, key)
        assert torch.equal(stack[i].k_cache, ref[i].k_cache) and torch.equal(stack[i].seqlens, ref[i].seqlens)
        assert stack[i].ctx.retopk_get_status() == 0
    p = np.concatenate(paths)
    assert (p == 0).sum() > 0 and (p != 0).sum() > 0   # both paths were exercised


def test_state_round_trip_and_status_bits():
    # tau = -1 with no refresh: every head reuses, so every head reads the
    # corrupted cached supports below
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=2048, steps=4, tau=-1.0, T_r=0)
    dr = DecodeRun(w)
    dr.step(0)
    st = dr.ctx.retopk_export_state()
    dr.ctx.retopk_import_state(st)
    st2 = dr.ctx.retopk_export_state()
    for key in st:
        assert np.array_equal(st[key], st2[key])
    # a support index beyond the history is reported, not followed (the last
    # live entry of every cached support: the lists stay ascending)
    bad = {k: v.copy() for k, v in st.items()}
    lens = bad["fifo_len"][0]
    assert (lens > 0).all()
    for h in range(lens.shape[0]):
        for c in range(lens.shape[1]):
            bad["fifo_sup"][0, h, c, lens[h, c] - 1] = 10 ** 6
    dr.ctx.retopk_import_state(bad)
    dr.ctx.retopk_decode_step(dr.q_dec[1], dr.k_cache, dr.v_cache, dr.seqlens, dr.out)
    s = dr.ctx.retopk_get_status(clear=True)
    diag = dr.ctx.retopk_get_diagnostics()
    assert (diag["path"] == 0).all()
    assert s & 0x1
    assert dr.ctx.retopk_get_status() == 0
    # appending to a full cache is reported and leaves the length unchanged
    dr.seqlens.fill_(dr.max_len)
    dr.ctx.retopk_append_kv(dr.k_new[0], dr.v_new[0], dr.k_cache, dr.v_cache, dr.seqlens)
    assert dr.ctx.retopk_get_status(clear=True) & 0x2
    assert (dr.seqlens.cpu() == dr.max_len).all()
    # ... also through the fused append + decode step
    dr.ctx.retopk_decode_step_kv(dr.k_new[0], dr.v_new[0], dr.q_dec[2], dr.k_cache, dr.v_cache, dr.seqlens, dr.out)
    assert dr.ctx.retopk_get_status() & 0x2
    assert (dr.seqlens.cpu() == dr.max_len).all()
    # malformed state buffers are refused on the host: a slot out of range, a
    # support out of order, a negative support index
    from top_sparse_attention_exact_gb300.retopk import RetopkError
    for what in ("slot", "order", "negative"):
        bad = {k: v.copy() for k, v in st.items()}
        if what == "slot":
            bad["seq"][0, 0] = w.C
        elif what == "order":
            s0 = bad["fifo_sup"][0, 3, 1]
            s0[0], s0[1] = s0[1], s0[0]
        else:
            bad["fifo_sup"][0, 3, 1, 0] = -5
        with pytest.raises(RetopkError):
            dr.ctx.retopk_import_state(bad)


def test_nonfinite_scores_are_reported():
    # a NaN in a key row makes its score NaN: the step reports it in the status
    # word (and faults nothing); the finite steps before it leave the word clear
    for tau, T_r in ((1.5, 0), (-1.0, 0)):           # every head exact / every head reuse
        w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=2048, steps=3, tau=tau, T_r=T_r, name=f"nan_tau{tau}")
        dr = DecodeRun(w)
        dr.step(0)
        assert dr.ctx.retopk_get_status() == 0
        # the next token's key (inside every reuse head's recent window) is NaN
        dr.k_new[1][0, 0, 5] = 0x7FC0
        dr.step(1)
        torch.cuda.synchronize()
        s = dr.ctx.retopk_get_status(clear=True)
        assert s & 0x4, (tau, s)
        assert not (s & 0x8), (tau, s)


def test_bounded_wait_expires_and_context_survives():
    """A pipeline wait that nobody satisfies gives up, flags the status word,
    and leaves the context usable (no trap, no hang)."""
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=2048, steps=2, name="selftest")
    dr = DecodeRun(w)
    dr.ctx.retopk_selftest_wait(100_000_000)      # ~50 ms of SM clock
    torch.cuda.synchronize()
    assert dr.ctx.retopk_get_status(clear=True) & 0x8
    assert dr.ctx.retopk_get_status() == 0
    pre = dr.ctx.retopk_export_state()
    dr.step(0)
    torch.cuda.synchronize()
    post = dr.ctx.retopk_export_state()
    diag = dr.ctx.retopk_get_diagnostics()
    errs, _ = compare_decode_step(pre, post, diag, dr.qd_host[0], dr.k_host, dr.v_host,
                                  dr.seqlens.cpu().numpy(), w, dr.out.cpu().numpy().view(np.uint16), "after")
    assert not errs, errs[:5]
    assert dr.ctx.retopk_get_status() == 0
