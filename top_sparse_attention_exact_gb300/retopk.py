"""Thin ctypes binding of libretopk (include/retopk.h).

Argument marshalling only: every step of the decode path runs in the CUDA
library.  Tensors are torch CUDA tensors (torch is used for device memory and
streams); bf16 tensors may be torch.bfloat16 or int16/uint16 holding the raw
bits.  There is no CPU fallback: if the library cannot be loaded every call
raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import _build

_lib = None

RETOPK_PATH_REUSE, RETOPK_PATH_FALLBACK, RETOPK_PATH_REFRESH = 0, 1, 2
STATUS_BAD_INDEX, STATUS_KV_FULL, STATUS_NONFINITE, STATUS_TIMEOUT, STATUS_GATHER = 0x1, 0x2, 0x4, 0x8, 0x10

EXPORTED = ("retopk_workspace_bytes", "retopk_create", "retopk_destroy", "retopk_init_cache",
            "retopk_append_kv", "retopk_decode_step", "retopk_decode_step_kv", "retopk_get_diagnostics",
            "retopk_get_counters", "retopk_state_bytes", "retopk_export_state",
            "retopk_import_state", "retopk_get_status", "retopk_strerror", "retopk_cuda_error_string",
            "exact_topk_workspace_bytes", "exact_topk_attention_step",
            "retopk_profile_enable", "retopk_profile_read", "retopk_profile_reset",
            "retopk_selftest_wait", "exact_topk_attention_step_noalloc", "retopk_fidelity",
            "retopk_decode_step_host", "retopk_support_overlap", "exact_topk_scan", "exact_topk_select",
            "retopk_state_workspace_bytes", "retopk_scratch_bytes", "retopk_create_shared")

PROF_KERNELS = ("append", "finish", "scan", "select", "clear", "decide")


class RetopkError(RuntimeError):
    pass


class retopk_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_len", ctypes.c_int32), ("K", ctypes.c_int32), ("C", ctypes.c_int32),
                ("W", ctypes.c_int32), ("R", ctypes.c_int32), ("T_r", ctypes.c_int32),
                ("tau", ctypes.c_float), ("retrieval", ctypes.c_int32), ("cluster", ctypes.c_int32)]


_P, _S, _I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int


def _declare(lib):
    cfgp = ctypes.POINTER(retopk_config)
    lib.retopk_workspace_bytes.argtypes = [cfgp]
    lib.retopk_workspace_bytes.restype = _S
    lib.retopk_create.argtypes = [cfgp, _P, _S, ctypes.POINTER(_P)]
    lib.retopk_destroy.argtypes = [_P]
    lib.retopk_state_workspace_bytes.argtypes = [cfgp]
    lib.retopk_state_workspace_bytes.restype = _S
    lib.retopk_scratch_bytes.argtypes = [cfgp]
    lib.retopk_scratch_bytes.restype = _S
    lib.retopk_create_shared.argtypes = [cfgp, _P, _S, _P, _S, ctypes.POINTER(_P)]
    lib.retopk_init_cache.argtypes = [_P, _P, _P, _P, _P]
    lib.retopk_append_kv.argtypes = [_P, _P, _P, _P, _P, _P, _P]
    lib.retopk_decode_step.argtypes = [_P, _P, _P, _P, _P, _P, _P]
    lib.retopk_decode_step_kv.argtypes = [_P] * 9
    lib.retopk_decode_step_host.argtypes = [_P] * 9
    lib.retopk_fidelity.argtypes = [_P] * 8
    lib.retopk_get_diagnostics.argtypes = [_P] + [_P] * 8 + [_P]
    lib.retopk_get_counters.argtypes = [_P, _P, _P]
    lib.retopk_state_bytes.argtypes = [_P]
    lib.retopk_state_bytes.restype = _S
    lib.retopk_export_state.argtypes = [_P, _P, _S, _P]
    lib.retopk_import_state.argtypes = [_P, _P, _S, _P]
    lib.retopk_get_status.argtypes = [_P, _P, _I, _P]
    lib.retopk_strerror.argtypes = [_I]
    lib.retopk_strerror.restype = ctypes.c_char_p
    lib.retopk_cuda_error_string.argtypes = []
    lib.retopk_cuda_error_string.restype = ctypes.c_char_p
    lib.exact_topk_workspace_bytes.argtypes = [_I] * 6
    lib.exact_topk_workspace_bytes.restype = _S
    lib.exact_topk_attention_step.argtypes = [_P, _P, _P, _P] + [_I] * 6 + [_P, _P, _P, _S, _P]
    lib.retopk_profile_enable.argtypes = [_I]
    lib.retopk_profile_read.argtypes = [_P, _P]
    lib.retopk_profile_reset.argtypes = []
    lib.retopk_selftest_wait.argtypes = [_P, ctypes.c_int64, _P]
    lib.exact_topk_attention_step_noalloc.argtypes = [_P, _P, _P, _P] + [_I] * 6 + [_P, _P, _P]
    lib.retopk_support_overlap.argtypes = [_P, _P, _I, _I, _I, _P, _P]
    lib.exact_topk_scan.argtypes = [_P, _P, _P] + [_I] * 6 + [_P, _S, _P]
    lib.exact_topk_select.argtypes = [_P, _P, _P] + [_I] * 6 + [_P, _P, _P, _S, _P]
    for name in EXPORTED:
        getattr(lib, name).restype = getattr(lib, name).restype or ctypes.c_int
    return lib


def library_path() -> str:
    return _build.LIB


def load(build: bool = True):
    """Load libretopk (building it in-tree first if asked and stale)."""
    global _lib
    if _lib is None:
        path = _build.build() if build else _build.LIB
        if not os.path.exists(path):
            raise RetopkError(f"libretopk not built ({path}); run __graft_entry__.build()")
        _lib = _declare(ctypes.CDLL(path))
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load().retopk_strerror(rc).decode()
        if rc == -4:
            msg += ": " + load().retopk_cuda_error_string().decode()
        raise RetopkError(f"{what} failed: {msg} ({rc})")


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise RetopkError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise RetopkError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _hptr(t: torch.Tensor, numel: int):
    """Host (CPU) tensor of exactly `numel` elements, contiguous."""
    if t.is_cuda:
        raise RetopkError("expected a host (CPU) tensor")
    if not t.is_contiguous() or t.numel() != numel:
        raise RetopkError(f"expected a contiguous host tensor of {numel} elements, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


_BF16_TYPES = (torch.bfloat16, torch.int16, torch.uint16)


def _bf16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype not in _BF16_TYPES:
        raise RetopkError(f"bf16 tensor expected, got {t.dtype}")
    return t


def _i32(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.int32:
        raise RetopkError(f"int32 tensor expected, got {t.dtype}")
    return t


def exact_topk_workspace_bytes(B, Hq, Hkv, d, max_len, K) -> int:
    n = load().exact_topk_workspace_bytes(B, Hq, Hkv, d, max_len, K)
    if n == 0:
        raise RetopkError("exact_topk_workspace_bytes: invalid sizes")
    return int(n)


def exact_topk_attention_step(q, k_cache, v_cache, seqlens, K, out, idx_out=None, workspace=None,
                              stream=None):
    """Exact Top-K attention. q [B,Hq,d]; caches [B,Hkv,max_len,d]; out [B,Hq,d]."""
    B, Hq, d = q.shape
    Hkv, max_len = k_cache.shape[1], k_cache.shape[2]
    if workspace is None:
        workspace = torch.empty(exact_topk_workspace_bytes(B, Hq, Hkv, d, max_len, K) + 256,
                                dtype=torch.uint8, device=q.device)
    wp = (workspace.data_ptr() + 255) // 256 * 256
    avail = workspace.numel() - (wp - workspace.data_ptr())
    rc = load().exact_topk_attention_step(
        _ptr(_bf16(q)), _ptr(_bf16(k_cache)), _ptr(_bf16(v_cache)), _ptr(_i32(seqlens)), B, Hq, Hkv, d,
        max_len, int(K), _ptr(_bf16(out)), _ptr(idx_out) if idx_out is not None else None,
        ctypes.c_void_p(wp), avail, _stream(stream))
    _check(rc, "exact_topk_attention_step")
    return out


def _exact_ws(workspace, B, Hq, Hkv, d, max_len, K, device):
    if workspace is None:
        workspace = torch.empty(exact_topk_workspace_bytes(B, Hq, Hkv, d, max_len, K) + 256, dtype=torch.uint8,
                                device=device)
    wp = (workspace.data_ptr() + 255) // 256 * 256
    return workspace, wp, workspace.numel() - (wp - workspace.data_ptr())


def exact_topk_scan(q, k_cache, seqlens, K, workspace, stream=None):
    """First half of the exact step: Eq. (4) scores and first-digit histograms into `workspace`."""
    B, Hq, d = q.shape
    Hkv, max_len = k_cache.shape[1], k_cache.shape[2]
    workspace, wp, avail = _exact_ws(workspace, B, Hq, Hkv, d, max_len, K, q.device)
    _check(load().exact_topk_scan(_ptr(_bf16(q)), _ptr(_bf16(k_cache)), _ptr(_i32(seqlens)), B, Hq, Hkv, d, max_len,
                                  int(K), ctypes.c_void_p(wp), avail, _stream(stream)), "exact_topk_scan")
    return workspace


def exact_topk_select(q, v_cache, seqlens, K, out, idx_out, workspace, stream=None):
    """Second half of the exact step: Eq. (1) and Eq. (12) from the scan half's workspace."""
    B, Hq, d = q.shape
    Hkv, max_len = v_cache.shape[1], v_cache.shape[2]
    workspace, wp, avail = _exact_ws(workspace, B, Hq, Hkv, d, max_len, K, q.device)
    _check(load().exact_topk_select(_ptr(_bf16(q)), _ptr(_bf16(v_cache)), _ptr(_i32(seqlens)), B, Hq, Hkv, d,
                                    max_len, int(K), _ptr(_bf16(out)), _ptr(idx_out) if idx_out is not None else None,
                                    ctypes.c_void_p(wp), avail, _stream(stream)), "exact_topk_select")
    return out


def exact_topk_attention_step_noalloc(q, k_cache, v_cache, seqlens, K, out, idx_out=None, stream=None):
    """Exact Top-K attention with the library's static scratch (no workspace)."""
    B, Hq, d = q.shape
    Hkv, max_len = k_cache.shape[1], k_cache.shape[2]
    rc = load().exact_topk_attention_step_noalloc(
        _ptr(_bf16(q)), _ptr(_bf16(k_cache)), _ptr(_bf16(v_cache)), _ptr(_i32(seqlens)), B, Hq, Hkv, d,
        max_len, int(K), _ptr(_bf16(out)), _ptr(idx_out) if idx_out is not None else None, _stream(stream))
    _check(rc, "exact_topk_attention_step_noalloc")
    return out


def support_overlap(S, others, stream=None):
    """Eqs. (2)-(3): S [rows, K] and others [rows, R, K] int32 CUDA tensors
    (ascending, -1 padded) -> float32 CUDA tensor [rows, 2] = (overlap with
    others[:, 0], coverage by the union of the R)."""
    rows, K = S.shape
    R = others.shape[1]
    if tuple(others.shape) != (rows, R, K):
        raise RetopkError(f"others must be [rows, R, K], got {tuple(others.shape)}")
    out = torch.empty((rows, 2), dtype=torch.float32, device=S.device)
    _check(load().retopk_support_overlap(_ptr(_i32(S)), _ptr(_i32(others)), rows, R, K, _ptr(out), _stream(stream)),
           "retopk_support_overlap")
    return out


def scratch_bytes(B, Hq, Hkv, max_len, K=512, C=32, W=32, R=4, T_r=128, tau=0.85, d=128, recent=False) -> int:
    """Bytes of the per-step scratch a context of this configuration needs (retopk_scratch_bytes)."""
    cfg = retopk_config(B, Hq, Hkv, d, max_len, K, C, W, R, T_r, tau, 1 if recent else 0)
    n = load().retopk_scratch_bytes(ctypes.byref(cfg))
    if n == 0:
        raise RetopkError("retopk_scratch_bytes: invalid configuration")
    return int(n)


def profile_enable(on: bool):
    _check(load().retopk_profile_enable(1 if on else 0), "retopk_profile_enable")


def profile_read() -> dict:
    """Per kernel class: (timed launches, summed ms) -- see retopk_profile_read."""
    n = np.zeros(len(PROF_KERNELS), np.int64)
    ms = np.zeros(len(PROF_KERNELS), np.float64)
    _check(load().retopk_profile_read(n.ctypes.data_as(ctypes.c_void_p), ms.ctypes.data_as(ctypes.c_void_p)),
           "retopk_profile_read")
    return {k: (int(n[i]), float(ms[i])) for i, k in enumerate(PROF_KERNELS)}


def profile_reset():
    _check(load().retopk_profile_reset(), "retopk_profile_reset")


class ReTopK:
    """A ReTopK decode context (query-support cache + scratch in a torch buffer)."""

    def __init__(self, B, Hq, Hkv, max_len, K=512, C=32, W=32, R=4, T_r=128, tau=0.85, d=128,
                 device="cuda", recent: bool = False, scratch: torch.Tensor | None = None, cluster: int = 0):
        """scratch: optional uint8 CUDA tensor of at least scratch_bytes(...) + 256 bytes, shared with
        other contexts whose steps run one after another on one stream (retopk_create_shared)."""
        self.cfg = retopk_config(B, Hq, Hkv, d, max_len, K, C, W, R, T_r, tau, 1 if recent else 0, cluster)
        lib = load()
        h = ctypes.c_void_p()
        if scratch is None:
            n = lib.retopk_workspace_bytes(ctypes.byref(self.cfg))
            if n == 0:
                raise RetopkError("retopk_workspace_bytes: invalid configuration")
            self.workspace = torch.empty(int(n) + 256, dtype=torch.uint8, device=device)
            wp = (self.workspace.data_ptr() + 255) // 256 * 256
            _check(lib.retopk_create(ctypes.byref(self.cfg), ctypes.c_void_p(wp), int(n), ctypes.byref(h)),
                   "retopk_create")
        else:
            ns = lib.retopk_state_workspace_bytes(ctypes.byref(self.cfg))
            if ns == 0:
                raise RetopkError("retopk_state_workspace_bytes: invalid configuration")
            self.workspace = torch.empty(int(ns) + 256, dtype=torch.uint8, device=device)
            self.scratch = scratch
            wp = (self.workspace.data_ptr() + 255) // 256 * 256
            sp = (scratch.data_ptr() + 255) // 256 * 256
            avail = scratch.numel() - (sp - scratch.data_ptr())
            _check(lib.retopk_create_shared(ctypes.byref(self.cfg), ctypes.c_void_p(wp), int(ns), ctypes.c_void_p(sp),
                                            int(avail), ctypes.byref(h)), "retopk_create_shared")
        self.handle = h
        self.B, self.Hq, self.Hkv, self.max_len = B, Hq, Hkv, max_len
        self.K, self.C, self.W, self.R, self.T_r, self.tau, self.d = K, C, W, R, T_r, tau, d

    def close(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.retopk_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- the hot path ---------------------------------------------------------
    def retopk_init_cache(self, q_last, k_cache, prompt_len, stream=None):
        _check(load().retopk_init_cache(self.handle, _ptr(_bf16(q_last)), _ptr(_bf16(k_cache)),
                                        _ptr(_i32(prompt_len)), _stream(stream)), "retopk_init_cache")

    def retopk_append_kv(self, k_new, v_new, k_cache, v_cache, seqlens, stream=None):
        _check(load().retopk_append_kv(self.handle, _ptr(_bf16(k_new)), _ptr(_bf16(v_new)),
                                       _ptr(_bf16(k_cache)), _ptr(_bf16(v_cache)), _ptr(_i32(seqlens)),
                                       _stream(stream)), "retopk_append_kv")

    def retopk_decode_step(self, q, k_cache, v_cache, seqlens, out, stream=None):
        _check(load().retopk_decode_step(self.handle, _ptr(_bf16(q)), _ptr(_bf16(k_cache)),
                                         _ptr(_bf16(v_cache)), _ptr(_i32(seqlens)), _ptr(_bf16(out)),
                                         _stream(stream)), "retopk_decode_step")
        return out

    def retopk_decode_step_kv(self, k_new, v_new, q, k_cache, v_cache, seqlens, out, stream=None):
        """retopk_append_kv + retopk_decode_step in one fewer launch."""
        _check(load().retopk_decode_step_kv(self.handle, _ptr(_bf16(k_new)), _ptr(_bf16(v_new)), _ptr(_bf16(q)),
                                            _ptr(_bf16(k_cache)), _ptr(_bf16(v_cache)), _ptr(_i32(seqlens)),
                                            _ptr(_bf16(out)), _stream(stream)), "retopk_decode_step_kv")
        return out

    def retopk_decode_step_host(self, k_new, v_new, q, k_cache, v_cache, seqlens, out, stream=None):
        """retopk_decode_step_kv with k_new / v_new / q / out in host memory
        (CPU tensors, pinned or not); returns once `out` holds the output.
        The device tensors and the stream are validated once per binding; each
        call checks the four host tensors and passes their addresses."""
        s = stream if stream is not None else torch.cuda.current_stream()
        key = (k_cache.data_ptr(), v_cache.data_ptr(), seqlens.data_ptr(), s.cuda_stream)
        if getattr(self, "_host_key", None) != key:
            _ptr(_bf16(k_cache)), _ptr(_bf16(v_cache)), _ptr(_i32(seqlens))
            self._host_key = key
            self._host_fn = load().retopk_decode_step_host
        nq, nkv = self.B * self.Hq * 128, self.B * self.Hkv * 128
        for t, n in ((k_new, nkv), (v_new, nkv), (q, nq), (out, nq)):
            if t.is_cuda or t.dtype not in _BF16_TYPES or t.numel() != n or not t.is_contiguous():
                _hptr(_bf16(t), n)   # raises with the reason
        rc = self._host_fn(self.handle, k_new.data_ptr(), v_new.data_ptr(), q.data_ptr(), key[0], key[1], key[2],
                           out.data_ptr(), key[3])
        if rc:
            _check(rc, "retopk_decode_step_host")
        return out

    def retopk_fidelity(self, q, k_cache, exact_idx, out_exact, out, stream=None):
        """Fidelity of the last decode step's supports/outputs against the exact
        ones: float32 CUDA tensor [B, Hq, 4] (recall, retained mass, output
        cosine, attention-distribution cosine)."""
        m = torch.empty((self.B, self.Hq, 4), dtype=torch.float32, device=q.device)
        _check(load().retopk_fidelity(self.handle, _ptr(_bf16(q)), _ptr(_bf16(k_cache)), _ptr(_i32(exact_idx)),
                                      _ptr(_bf16(out_exact)), _ptr(_bf16(out)), _ptr(m), _stream(stream)),
               "retopk_fidelity")
        return m

    # --- inspection -------------------------------------------------------------
    def retopk_get_diagnostics(self, stream=None) -> dict:
        BH = self.B * self.Hq
        cap = self.R * self.K + self.W
        r = dict(path=np.empty(BH, np.int32), rho_max=np.empty(BH, np.float32),
                 topR=np.empty((BH, self.R), np.int32), M=np.empty(BH, np.int32),
                 cand=np.empty((BH, cap), np.int32), support=np.empty((BH, self.K), np.int32),
                 sup_len=np.empty(BH, np.int32), out_f32=np.empty((BH, self.d), np.float32))
        p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
        _check(load().retopk_get_diagnostics(self.handle, p(r["path"]), p(r["rho_max"]), p(r["topR"]),
                                             p(r["M"]), p(r["cand"]), p(r["support"]), p(r["sup_len"]),
                                             p(r["out_f32"]), _stream(stream)), "retopk_get_diagnostics")
        return r

    def retopk_get_counters(self, stream=None):
        c = np.zeros(5, np.int64)
        _check(load().retopk_get_counters(self.handle, c.ctypes.data_as(ctypes.c_void_p), _stream(stream)),
               "retopk_get_counters")
        return dict(reuse=int(c[0]), fallback=int(c[1]), refresh=int(c[2]), sum_M=int(c[3]),
                    max_M=int(c[4]))

    def state_bytes(self) -> int:
        return int(load().retopk_state_bytes(self.handle))

    def retopk_export_state(self, stream=None) -> dict:
        n = self.state_bytes()
        buf = np.empty(n, np.uint8)
        _check(load().retopk_export_state(self.handle, buf.ctypes.data_as(ctypes.c_void_p), n,
                                          _stream(stream)), "retopk_export_state")
        return self._unpack(buf)

    def retopk_import_state(self, st: dict, stream=None):
        buf = self._pack(st)
        _check(load().retopk_import_state(self.handle, buf.ctypes.data_as(ctypes.c_void_p), buf.nbytes,
                                          _stream(stream)), "retopk_import_state")

    def retopk_get_status(self, clear=False, stream=None) -> int:
        v = ctypes.c_uint32()
        _check(load().retopk_get_status(self.handle, ctypes.byref(v), 1 if clear else 0, _stream(stream)),
               "retopk_get_status")
        return int(v.value)

    def retopk_selftest_wait(self, wait_cycles: int, stream=None):
        _check(load().retopk_selftest_wait(self.handle, int(wait_cycles), _stream(stream)), "retopk_selftest_wait")

    def _unpack(self, buf: np.ndarray) -> dict:
        B, Hq, C, K, d = self.B, self.Hq, self.C, self.K, self.d
        o = 0

        def take(dtype, shape):
            nonlocal o
            n = int(np.prod(shape)) * np.dtype(dtype).itemsize
            a = buf[o:o + n].view(dtype).reshape(shape).copy()
            o += n
            return a
        return dict(fifo_q=take(np.uint16, (B, Hq, C, d)), fifo_sup=take(np.int32, (B, Hq, C, K)),
                    fifo_len=take(np.int32, (B, Hq, C)), seq=take(np.int32, (B, 3)))

    def _pack(self, st: dict) -> np.ndarray:
        parts = [np.ascontiguousarray(st["fifo_q"], np.uint16), np.ascontiguousarray(st["fifo_sup"], np.int32),
                 np.ascontiguousarray(st["fifo_len"], np.int32), np.ascontiguousarray(st["seq"], np.int32)]
        return np.concatenate([p.reshape(-1).view(np.uint8) for p in parts])
