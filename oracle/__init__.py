"""ctypes front-end of the fp64 CPU oracle (retopk_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports this package, and this package imports nothing from the library.

All inputs are bf16 bit patterns (numpy uint16); results are float64 / int32
numpy arrays.  Shapes follow the C file's comments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "retopk_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no FP contraction)."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        tmp = _OUT + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _OUT)
    return _OUT


def load(path: str | None = None):
    """Load (building if needed) and return the ctypes handle."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_D = ctypes.c_double


def _declare(lib):
    lib.oracle_scores.argtypes = [_P, _P, _L, _P, _I, _I, _P]
    lib.oracle_topk.argtypes = [_P, _P, _I, _I, _P]
    lib.oracle_topk.restype = _I
    lib.oracle_sparse_attention.argtypes = [_P, _P, _I, _P, _L, _I, _P]
    lib.oracle_attention_on_support.argtypes = [_P, _P, _P, _L, _P, _I, _I, _P]
    lib.oracle_dense_attention.argtypes = [_P, _P, _P, _L, _I, _I, _P]
    lib.oracle_softmax_merge.argtypes = [_D, _D, _P, _D, _D, _P, _I, _P, _P, _P]
    lib.oracle_recall.argtypes = [_P, _P, _I, _I, _I, _P, _P]
    lib.oracle_recall.restype = _D
    lib.oracle_candidates.argtypes = [_P, _P, _I, _I, _I, _P]
    lib.oracle_candidates.restype = _I
    lib.oracle_exact_one.argtypes = [_P, _P, _P, _L, _I, _I, _I, _P, _P, _P]
    lib.oracle_exact_one.restype = _I
    lib.oracle_exact_step.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _L, _I, _P, _P, _P, _P]
    lib.oracle_init_cache.argtypes = [_P, _P, _L, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]
    lib.oracle_init_cache.restype = _I
    lib.oracle_recall_recent.argtypes = [_P, _P, _I, _I, _I, _P, _P]
    lib.oracle_recall_recent.restype = _D
    lib.oracle_decode_step.argtypes = [_P, _P, _P, _L, _I, _I, _I, _I, _I, _I, _I, _I, _I, _D, _I,
                                       _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P, _P]
    lib.oracle_fidelity.argtypes = [_P, _P, _L, _I, _P, _I, _P, _I, _P, _P, _P]
    lib.oracle_overlap.argtypes = [_P, _I, _P, _I, _I]
    lib.oracle_overlap.restype = _D
    lib.oracle_coverage.argtypes = [_P, _P, _P, _P, _I, _I, _I, _P, _I, _I, _P]
    lib.oracle_coverage.restype = _D
    lib.oracle_set_threads.argtypes = [_I]
    lib.oracle_get_threads.restype = _I
    return lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def fidelity(q, k, S, Sh, o, oh, lib=None):
    """Support recall, retained Exact Top-K mass, output cosine and attention-
    distribution cosine of support Sh (output oh) against the exact support S
    (output o); supports ascending, -1 entries ignored.  k: [L, d] rows."""
    lib = lib or load()
    q, k = _u16(q), _u16(k)
    S = _i32(np.asarray(S)[np.asarray(S) >= 0])
    Sh = _i32(np.asarray(Sh)[np.asarray(Sh) >= 0])
    o, oh = _f64(o), _f64(oh)
    out = np.zeros(4)
    lib.oracle_fidelity(_p(q), _p(k), k.shape[-1], q.shape[-1], _p(S), len(S), _p(Sh), len(Sh), _p(o), _p(oh),
                        _p(out))
    return out


def overlap(St, Sj, K, lib=None):
    """Eq. (2): |S_t n S_j| / K for two ascending supports (-1 entries ignored)."""
    lib = lib or load()
    St = _i32(np.asarray(St)[np.asarray(St) >= 0])
    Sj = _i32(np.asarray(Sj)[np.asarray(Sj) >= 0])
    return float(lib.oracle_overlap(_p(St), len(St), _p(Sj), len(Sj), int(K)))


def coverage(q, prev_q, prev_S, St, R, K, lib=None):
    """Eq. (3): coverage of St by the union of the supports of the R preceding
    queries most similar to q.  prev_q [n, d] oldest first, prev_S a list of n
    ascending supports.  Returns (coverage, chosen positions [R], -1 padded)."""
    lib = lib or load()
    q = _u16(q)
    prev_q = _u16(prev_q).reshape(-1, q.shape[-1])
    n, d = prev_q.shape
    sups = [_i32(np.asarray(s)[np.asarray(s) >= 0]) for s in prev_S]
    assert len(sups) == n
    qp = (ctypes.c_void_p * max(n, 1))(*[prev_q[c].ctypes.data for c in range(n)])
    sp = (ctypes.c_void_p * max(n, 1))(*[s.ctypes.data for s in sups])
    ln = _i32([len(s) for s in sups] or [0])
    St = _i32(np.asarray(St)[np.asarray(St) >= 0])
    chosen = np.empty(max(R, 1), dtype=np.int32)
    cov = lib.oracle_coverage(_p(q), qp, sp, _p(ln), n, d, int(R), _p(St), len(St), int(K), _p(chosen))
    return float(cov), chosen[:R].copy()


def state_from_export(st: dict, b: int, K: int) -> "CacheState":
    """The oracle's cache state for sequence b from a library state export
    (the dict of arrays the binding's retopk_export_state returns)."""
    Hq, C, d = st["fifo_q"].shape[1], st["fifo_q"].shape[2], st["fifo_q"].shape[3]
    cs = CacheState(Hq, C, K, d)
    cs.fq[...] = st["fifo_q"][b]
    cs.fsup[...] = st["fifo_sup"][b]
    cs.flen[...] = st["fifo_len"][b]
    cs.seq[...] = st["seq"][b]
    return cs


def set_threads(n: int) -> None:
    load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(load().oracle_get_threads())


def scores(q, k, idx=None, lib=None):
    """Eq. (4)/(10): q [d] bf16, k [n_rows, d] bf16 -> float64 scores of idx (or all rows)."""
    lib = lib or load()
    q, k = _u16(q), _u16(k)
    d = q.shape[-1]
    n = k.shape[0] if idx is None else len(idx)
    idx = None if idx is None else _i32(idx)
    out = np.empty(n, dtype=np.float64)
    lib.oracle_scores(_p(q), _p(k), d, _p(idx), n, d, _p(out))
    return out


def topk(score, K, idx=None, lib=None):
    """Eqs. (1)/(11): indices of the K best by (score desc, index asc), rank order."""
    lib = lib or load()
    score = _f64(score)
    n = len(score)
    idx = None if idx is None else _i32(idx)
    out = np.empty(max(min(K, n), 1), dtype=np.int32)
    m = lib.oracle_topk(_p(score), _p(idx), n, int(K), _p(out))
    return out[:m].copy()


def sparse_attention(score, idx, v, lib=None):
    """Eq. (12): softmax over score, weighted sum of v rows idx. v [n_rows, d]."""
    lib = lib or load()
    score, idx, v = _f64(score), _i32(idx), _u16(v)
    d = v.shape[-1]
    out = np.empty(d, dtype=np.float64)
    lib.oracle_sparse_attention(_p(score), _p(idx), len(idx), _p(v), d, d, _p(out))
    return out


def attention_on_support(q, k, v, sup, lib=None):
    """Eqs. (10)+(12) restricted to the given support (rows of k, v [n_rows, d])."""
    lib = lib or load()
    q, k, v, sup = _u16(q), _u16(k), _u16(v), _i32(sup)
    d = q.shape[-1]
    out = np.empty(d, dtype=np.float64)
    lib.oracle_attention_on_support(_p(q), _p(k), _p(v), d, _p(sup), len(sup), d, _p(out))
    return out


def dense_attention(q, k, v, L=None, lib=None):
    """Full softmax attention over rows 0..L-1."""
    lib = lib or load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    d = q.shape[-1]
    L = k.shape[0] if L is None else L
    out = np.empty(d, dtype=np.float64)
    lib.oracle_dense_attention(_p(q), _p(k), _p(v), d, int(L), d, _p(out))
    return out


def softmax_merge(m1, Z1, o1, m2, Z2, o2, lib=None):
    """Merge two disjoint softmax partials (m, Z, o) -> (m, Z, o)."""
    lib = lib or load()
    o1, o2 = _f64(o1), _f64(o2)
    d = len(o1)
    o = np.empty(d, dtype=np.float64)
    m = ctypes.c_double()
    Z = ctypes.c_double()
    lib.oracle_softmax_merge(float(m1), float(Z1), _p(o1), float(m2), float(Z2), _p(o2), d,
                             ctypes.byref(m), ctypes.byref(Z), _p(o))
    return m.value, Z.value, o


def recall(q, cached, R, lib=None):
    """Eqs. (6)-(7): q [d], cached [n, d] oldest first -> (rho [n], topR [R], rho_max)."""
    lib = lib or load()
    q = _u16(q)
    cached = _u16(cached).reshape(-1, q.shape[-1])
    n, d = cached.shape
    ptrs = (ctypes.c_void_p * max(n, 1))(*[cached[c].ctypes.data for c in range(n)])
    rho = np.empty(max(n, 1), dtype=np.float64)
    top = np.empty(max(R, 1), dtype=np.int32)
    rmax = lib.oracle_recall(_p(q), ptrs, n, d, int(R), _p(rho), _p(top))
    return rho[:n].copy(), top[:R].copy(), rmax


def candidates(supports, L, W, lib=None):
    """Eqs. (8)-(9): union of the given supports and the window, ascending."""
    lib = lib or load()
    arrs = [_i32(s) for s in supports]
    ptrs = (ctypes.c_void_p * max(len(arrs), 1))(*[a.ctypes.data for a in arrs])
    lens = _i32([len(a) for a in arrs] or [0])
    cap = sum(len(a) for a in arrs) + max(W, 0) + 1
    out = np.empty(cap, dtype=np.int32)
    m = lib.oracle_candidates(ptrs, _p(lens), len(arrs), int(L), int(W), _p(out))
    return out[:m].copy()


def exact_one(q, k, v, L, K, lib=None):
    """Exact Top-K attention of one query over rows 0..L-1 -> (support asc, kth, out)."""
    lib = lib or load()
    q, k = _u16(q), _u16(k)
    v = None if v is None else _u16(v)
    d = q.shape[-1]
    sup = np.full(max(K, 1), -1, dtype=np.int32)
    kth = ctypes.c_double()
    out = np.empty(d, dtype=np.float64)
    n = lib.oracle_exact_one(_p(q), _p(k), _p(v), d, int(L), d, int(K), _p(sup),
                             ctypes.byref(kth), None if v is None else _p(out))
    return sup[:n].copy(), kth.value, (out if v is not None else None)


def exact_step(q, k, v, L, K, lib=None):
    """Batched Exact Top-K: q [B,Hq,d], k/v [B,Hkv,max_len,d], L [B]."""
    lib = lib or load()
    q, k, v, L = _u16(q), _u16(k), _u16(v), _i32(L)
    B, Hq, d = q.shape
    Hkv, max_len = k.shape[1], k.shape[2]
    sup = np.empty((B, Hq, K), dtype=np.int32)
    sup_len = np.empty((B, Hq), dtype=np.int32)
    kth = np.empty((B, Hq), dtype=np.float64)
    out = np.empty((B, Hq, d), dtype=np.float64)
    lib.oracle_exact_step(_p(q), _p(k), _p(v), _p(L), B, Hq, Hkv, d, max_len, int(K),
                          _p(sup), _p(sup_len), _p(kth), _p(out))
    return sup, sup_len, kth, out


class CacheState:
    """The oracle's query-support cache for ONE sequence (layout: see the C file)."""

    def __init__(self, Hq: int, C: int, K: int, d: int = 128):
        self.Hq, self.C, self.K, self.d = Hq, C, K, d
        self.fq = np.zeros((Hq, C, d), dtype=np.uint16)
        self.fsup = np.full((Hq, C, K), -1, dtype=np.int32)
        self.flen = np.zeros((Hq, C), dtype=np.int32)
        self.seq = np.zeros(3, dtype=np.int32)      # next slot, live count, t_dec

    def copy(self) -> "CacheState":
        c = CacheState(self.Hq, self.C, self.K, self.d)
        c.fq[...] = self.fq
        c.fsup[...] = self.fsup
        c.flen[...] = self.flen
        c.seq[...] = self.seq
        return c

    def live(self, h: int):
        """Live entries of head h oldest first: list of (q bits, support)."""
        head, count = int(self.seq[0]), int(self.seq[1])
        res = []
        for c in range(count):
            s = (head - count + c) % self.C
            res.append((self.fq[h, s].copy(), self.fsup[h, s, :self.flen[h, s]].copy()))
        return res


def init_cache(q_prompt, k, L0, Hq, Hkv, K, C, lib=None) -> CacheState:
    """Cache initialisation for one sequence: q_prompt [Hq,C,d], k [Hkv,max_len,d]."""
    lib = lib or load()
    q_prompt, k = _u16(q_prompt), _u16(k)
    d = q_prompt.shape[-1]
    st = CacheState(Hq, C, K, d)
    rc = lib.oracle_init_cache(_p(q_prompt), _p(k), k.shape[1], int(L0), Hq, Hkv, d, int(K),
                               int(C), _p(st.fq), _p(st.fsup), _p(st.flen), _p(st.seq))
    if rc != 0:
        raise ValueError("oracle_init_cache: need L0 >= C >= 1")
    return st


def decode_step(st: CacheState, q, k, v, L, Hkv, W, R, T_r, tau, lib=None, recent: bool = False) -> dict:
    """One ReTopK decode step for one sequence; updates `st` in place.

    q [Hq,d]; k, v [Hkv,max_len,d]; L = keys including the current one.
    """
    lib = lib or load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    Hq, C, K, d = st.Hq, st.C, st.K, st.d
    cap = R * K + max(W, 0) + 1
    r = dict(
        path=np.empty(Hq, np.int32), rho=np.empty((Hq, C), np.float64),
        rho_max=np.empty(Hq, np.float64), topR=np.empty((Hq, R), np.int32),
        cand=np.full((Hq, cap), -1, np.int32), M=np.empty(Hq, np.int32),
        sup=np.empty((Hq, K), np.int32), sup_len=np.empty(Hq, np.int32),
        kth=np.empty(Hq, np.float64), out=np.empty((Hq, d), np.float64))
    lib.oracle_decode_step(_p(q), _p(k), _p(v), k.shape[1], int(L), Hq, Hkv, d, K, C, int(W),
                           int(R), int(T_r), float(tau), int(bool(recent)), _p(st.fq), _p(st.fsup), _p(st.flen),
                           _p(st.seq), _p(r["path"]), _p(r["rho"]), _p(r["rho_max"]),
                           _p(r["topR"]), _p(r["cand"]), cap, _p(r["M"]), _p(r["sup"]),
                           _p(r["sup_len"]), _p(r["kth"]), _p(r["out"]))
    return r
