"""The allocation-free Exact Top-K entry point (static scratch, no workspace).

Some callers cannot allocate device memory at all -- for instance code that
runs under an external memory manager owning the whole device, or a plain C
host with no allocator to hand the library a workspace.  For them the library
exports exact_topk_attention_step_noalloc, whose scratch is one 16 MiB
file-scope device array.  These tests call it through the C ABI and check it
against the workspace entry point on the same inputs, twice in a row (the
array keeps the previous call's contents, so the second call checks that the
entry point clears what it must), and check that a call after the first one
takes no device memory.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from top_sparse_attention_exact_gb300 import retopk, synth
from top_sparse_attention_exact_gb300.runner import to_dev

pytestmark = pytest.mark.gpu


def _case(seed, B=2, Hq=8, Hkv=2, L=(9000, 4097), max_len=9100):
    rng = np.random.default_rng(seed)
    q = synth.random_bf16(rng, (B, Hq, 128))
    k = synth.random_bf16(rng, (B, Hkv, max_len, 128))
    v = synth.random_bf16(rng, (B, Hkv, max_len, 128))
    return to_dev(q, "cuda"), to_dev(k, "cuda"), to_dev(v, "cuda"), torch.tensor(L, dtype=torch.int32, device="cuda")


def _raw_noalloc(q, k, v, sl, K, out, idx):
    """Direct C-ABI call (no Python-side allocation)."""
    lib = retopk.load()
    B, Hq, d = q.shape
    Hkv, max_len = k.shape[1], k.shape[2]
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.exact_topk_attention_step_noalloc(p(q), p(k), p(v), p(sl), B, Hq, Hkv, d, max_len, K, p(out),
                                                 p(idx), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice():
    K = 300
    q, k, v, sl = _case(1)
    B, Hq = q.shape[0], q.shape[1]
    for call in range(2):
        if call == 1:
            q = to_dev(synth.random_bf16(np.random.default_rng(2), (B, Hq, 128)), "cuda")   # new queries
        out_ref = torch.empty((B, Hq, 128), dtype=torch.int16, device="cuda")
        idx_ref = torch.empty((B, Hq, K), dtype=torch.int32, device="cuda")
        retopk.exact_topk_attention_step(q, k, v, sl, K, out_ref, idx_ref)
        out = torch.full((B, Hq, 128), -1, dtype=torch.int16, device="cuda")
        idx = torch.full((B, Hq, K), -7, dtype=torch.int32, device="cuda")
        assert _raw_noalloc(q, k, v, sl, K, out, idx) == 0
        torch.cuda.synchronize()
        # the same kernels on the same inputs: identical bits
        assert torch.equal(idx, idx_ref), f"call {call}: supports differ"
        assert torch.equal(out, out_ref), f"call {call}: outputs differ"


def test_noalloc_call_takes_no_device_memory():
    # the first call on a device may load the library's module there (which
    # reserves the static array); every later call must leave the device's
    # free memory unchanged
    K = 300
    q, k, v, sl = _case(4)
    B, Hq = q.shape[0], q.shape[1]
    out = torch.empty((B, Hq, 128), dtype=torch.int16, device="cuda")
    idx = torch.empty((B, Hq, K), dtype=torch.int32, device="cuda")
    assert _raw_noalloc(q, k, v, sl, K, out, idx) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        assert _raw_noalloc(q, k, v, sl, K, out, idx) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    q, k, v, sl = _case(3, B=1, Hq=28, Hkv=4, L=(100,), max_len=65536)
    out = torch.empty((1, 28, 128), dtype=torch.int16, device="cuda")
    idx = torch.empty((1, 28, 512), dtype=torch.int32, device="cuda")
    assert _raw_noalloc(q, k, v, sl, 512, out, idx) == -7
    assert "static" in retopk.load().retopk_strerror(-7).decode()
    torch.cuda.synchronize()
