"""GPU-vs-oracle comparison helpers (used by the -m gpu tests and smoke()).

Tolerances (written here, applied everywhere):
  * path decisions: identical unless the oracle's |rho_max - tau| < 1e-4;
  * rho_max: within RHO_TOL = 1e-5 of the oracle's fp64 value.  The library
    takes the cosine in fp32 (bf16 products are exact in fp32; the 128-term
    sums run as a depth-8 tree), so its error is at most about
    (gamma_8 + 4u) ~ 1.5e-6 (u = 2^-24, Cauchy-Schwarz bounds the sum of
    |products| by the norms); 1e-5 leaves margin and stays far inside the
    1e-4 band the path decision is exempt in;
  * retrieved entries R_t: the same set unless the oracle's R-th and (R+1)-th
    cosines are within 1e-4 of each other; in that band the GPU's candidate
    set must still be exactly the union of the GPU's own retrieved supports
    and the recent window;
  * candidate sets A_t (when path and R_t agree): identical;
  * supports: identical up to swaps among keys whose oracle score lies within
    1e-3 of the oracle's K-th score;
  * outputs: max-abs <= 2e-2 and relative L2 <= 1e-2 against the oracle's
    fp64 Eq. (12) output on the GPU's own support, and separately against the
    oracle's output on the oracle's own support (whenever path and R_t agree).
    Where the two supports differ by legal near-tie swaps, a swap changes the
    output by the swapped keys' own contributions, which can exceed 1e-2 of a
    small output's norm; the second comparison then allows, on top of the
    tolerance, the relative difference the swaps alone cause (the oracle's
    fp64 outputs on the two supports, compared with each other).
Band exemptions are counted and returned, so the tests can report and bound
them.
"""
from __future__ import annotations

import numpy as np

import oracle

TAU_BAND = 1e-4
RHO_TOL = 1e-5
SCORE_BAND = 1e-3
OUT_MAX_ABS = 2e-2
OUT_REL_L2 = 1e-2


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h).astype(np.uint32) << 16).view(np.float32)


def out_close(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    mx = float(np.abs(got - ref).max()) if got.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    return (mx <= OUT_MAX_ABS and rel <= OUT_REL_L2), mx, rel


def out_close_swapped(got, ref_own, ref_gpu_support):
    """Output check against the oracle's output on its own support (ref_own),
    when the GPU's support may differ from it by legal near-tie swaps:
    max-abs <= OUT_MAX_ABS, and relative L2 <= OUT_REL_L2 plus the relative
    difference between the oracle's fp64 outputs on the two supports
    (ref_gpu_support is the oracle's output on the GPU's support; 0 when the
    supports are equal)."""
    ref_own = np.asarray(ref_own, np.float64)
    swap = float(np.linalg.norm(np.asarray(ref_gpu_support, np.float64) - ref_own) /
                 max(np.linalg.norm(ref_own), 1e-30))
    got = np.asarray(got, np.float64)
    mx = float(np.abs(got - ref_own).max()) if got.size else 0.0
    rel = float(np.linalg.norm(got - ref_own) / max(np.linalg.norm(ref_own), 1e-30))
    return (mx <= OUT_MAX_ABS and rel <= OUT_REL_L2 + swap), mx, rel


def support_ok(q, k_rows, got, want, kth):
    """Supports may differ only among keys scoring within SCORE_BAND of the K-th."""
    got = [int(x) for x in got]
    want = [int(x) for x in want]
    if len(got) != len(want):
        return False, f"support length {len(got)} != {len(want)}"
    if len(set(got)) != len(got):
        return False, "duplicate index in support"
    if got != sorted(got):
        return False, "support not ascending"
    diff = sorted(set(got) ^ set(want))
    if not diff:
        return True, ""
    s = oracle.scores(q, k_rows, np.array(diff, dtype=np.int32))
    bad = [(i, float(x)) for i, x in zip(diff, s) if abs(x - kth) > SCORE_BAND]
    if bad:
        return False, f"{len(diff)} differing keys, {len(bad)} outside the band, e.g. {bad[:4]} (kth={kth})"
    return True, f"{len(diff)} near-tie swaps"


def compare_exact(q, k, v, L, K, gpu_idx, gpu_out, where=""):
    """Exact Top-K: q [B,Hq,d], k/v [B,Hkv,T,d] bits, L [B]; gpu_idx [B,Hq,K] (-1 pad); gpu_out [B,Hq,d] f32."""
    B, Hq, d = q.shape
    G = Hq // k.shape[1]
    sup, sup_len, kth, out = oracle.exact_step(q, k, v, L, K)
    errs = []
    for b in range(B):
        for h in range(Hq):
            n = int(sup_len[b, h])
            g = gpu_idx[b, h]
            gs = g[g >= 0]
            if (g[len(gs):] != -1).any() or not (g[:len(gs)] >= 0).all():
                errs.append(f"{where} b{b} h{h}: bad -1 padding")
                continue
            kr = k[b, h // G]
            ok, msg = support_ok(q[b, h], kr, gs, sup[b, h, :n], kth[b, h])
            if not ok:
                errs.append(f"{where} b{b} h{h}: {msg}")
                continue
            ref = oracle.attention_on_support(q[b, h], kr, v[b, h // G], gs)
            ok, mx, rel = out_close(gpu_out[b, h], ref)
            if not ok:
                errs.append(f"{where} b{b} h{h}: out max {mx:.3g} rel {rel:.3g}")
            ok, mx, rel = out_close_swapped(gpu_out[b, h], out[b, h], ref)
            if not ok:
                errs.append(f"{where} b{b} h{h}: out vs oracle support max {mx:.3g} rel {rel:.3g}")
    return errs


def compare_decode_step(pre: dict, post: dict, diag: dict, q_t, k, v, L, w, gpu_out_bf16, where=""):
    """State-forced check of one decode step for every sequence.

    pre / post: the GPU's exported cache state before / after the step.
    q_t [B,Hq,d] bits; k, v [B,Hkv,T,d] bits; L [B] (current token included).
    Returns (errors, stats); stats counts the heads checked, the band
    exemptions (path_band, topR_band) and the supports with near-tie swaps.
    """
    B, Hq, d = q_t.shape
    G = Hq // w.Hkv
    R, K, C = w.R, w.K, w.C
    errs = []
    stats = dict(path_band=0, topR_band=0, swaps=0, heads=0)
    for b in range(B):
        cs = oracle.state_from_export(pre, b, K)
        cs0 = cs.copy()                          # the pre-step cache (decode_step updates cs)
        r = oracle.decode_step(cs, q_t[b], k[b], v[b], int(L[b]), w.Hkv, w.W, R, w.T_r, w.tau,
                               recent=getattr(w, "recent", False))
        for h in range(Hq):
            bh = b * Hq + h
            stats["heads"] += 1
            tag = f"{where} b{b} h{h}"
            po, pg = int(r["path"][h]), int(diag["path"][bh])
            rmax_o, rmax_g = float(r["rho_max"][h]), float(diag["rho_max"][bh])
            if np.isfinite(rmax_o) or np.isfinite(rmax_g):
                if abs(rmax_o - rmax_g) > RHO_TOL:
                    errs.append(f"{tag}: rho_max {rmax_g} vs oracle {rmax_o}")
            if po != pg:
                if po != 2 and pg != 2 and abs(rmax_o - w.tau) < TAU_BAND:
                    stats["path_band"] += 1
                    continue
                errs.append(f"{tag}: path {pg} vs oracle {po} (rho_max {rmax_o})")
                continue
            kr, vr = k[b, h // G], v[b, h // G]
            # retrieved entries (as a set)
            count = int(pre["seq"][b, 1])
            nr = min(R, count)
            to, tg = set(r["topR"][h, :nr].tolist()), set(diag["topR"][bh, :nr].tolist())
            topR_same = to == tg
            if not topR_same:
                rho = np.sort(r["rho"][h, :count])[::-1]
                if nr < count and abs(rho[nr - 1] - rho[nr]) < TAU_BAND:
                    stats["topR_band"] += 1
                else:
                    errs.append(f"{tag}: topR {sorted(tg)} vs oracle {sorted(to)}")
                    continue
            Mg = int(diag["M"][bh])
            if po == 0 and topR_same:
                Mo = int(r["M"][h])
                if Mo != Mg or not np.array_equal(r["cand"][h, :Mo], diag["cand"][bh, :Mg]):
                    errs.append(f"{tag}: candidate set differs (M {Mg} vs {Mo})")
                    continue
            if po == 0 and not topR_same:
                # a different (legal) retrieval: the GPU's candidate set must be the
                # union of the supports of the entries the GPU retrieved, plus the window
                live = cs0.live(h)
                mine = [live[int(c)][1] for c in diag["topR"][bh, :nr]]
                want_A = oracle.candidates(mine, int(L[b]), w.W)
                if Mg != len(want_A) or not np.array_equal(diag["cand"][bh, :Mg], want_A):
                    errs.append(f"{tag}: candidate set is not the union of the GPU's retrieved supports")
                    continue
            gs = diag["support"][bh, :int(diag["sup_len"][bh])]
            if po == 0 and not topR_same:
                # check the GPU's own support against the rerank of its own candidate set
                A = diag["cand"][bh, :Mg]
                e = oracle.scores(q_t[b, h], kr, A)
                want = np.sort(oracle.topk(e, K, idx=A))
                kth = float(np.sort(e)[::-1][min(K, len(e)) - 1]) if len(e) else 0.0
            else:
                want = r["sup"][h, :int(r["sup_len"][h])]
                kth = float(r["kth"][h])
            ok, msg = support_ok(q_t[b, h], kr, gs, want, kth)
            if not ok:
                errs.append(f"{tag}: support {msg}")
                continue
            if msg:
                stats["swaps"] += 1
            got_bf16 = bf16_to_f32(gpu_out_bf16[b, h])
            ref = oracle.attention_on_support(q_t[b, h], kr, vr, gs)
            ok1, mx, rel = out_close(got_bf16, ref)
            ok2, mx2, rel2 = out_close(diag["out_f32"][bh], ref)
            if not (ok1 and ok2):
                errs.append(f"{tag}: out max {mx:.3g}/{mx2:.3g} rel {rel:.3g}/{rel2:.3g}")
            if topR_same:
                # separately: against the oracle's output on the oracle's own support
                ok3, mx3, rel3 = out_close_swapped(got_bf16, r["out"][h], ref)
                if not ok3:
                    errs.append(f"{tag}: out vs oracle support max {mx3:.3g} rel {rel3:.3g}")
            # the cache slot written by this step
            slot = int(pre["seq"][b, 0])
            if not np.array_equal(post["fifo_q"][b, h, slot], q_t[b, h]):
                errs.append(f"{tag}: cached query bits differ")
            n = int(post["fifo_len"][b, h, slot])
            if n != len(gs) or not np.array_equal(post["fifo_sup"][b, h, slot, :n], gs):
                errs.append(f"{tag}: cached support differs from the step's support")
        exp_seq = [(int(pre["seq"][b, 0]) + 1) % C, min(int(pre["seq"][b, 1]) + 1, C), int(pre["seq"][b, 2]) + 1]
        if post["seq"][b].tolist() != exp_seq:
            errs.append(f"{where} b{b}: seq {post['seq'][b].tolist()} vs {exp_seq}")
    return errs, stats
