"""The C-ABI library builds, loads and exports every declared entry point; the
host-side argument checks answer without a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

from top_sparse_attention_exact_gb300 import retopk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "retopk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)) - {"if", "sizeof"})


@pytest.fixture(scope="module")
def lib():
    return retopk.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(retopk.EXPORTED)


def test_checked_build_exports_every_entry_point():
    # the RETOPK_CHECKED variant (gathered row indices range-checked) builds
    # and carries the same ABI
    from top_sparse_attention_exact_gb300 import _build
    chk = ctypes.CDLL(_build.build(checked=True))
    for n in declared_functions():
        assert hasattr(chk, n), n


def test_config_validation_without_gpu(lib):
    ok = retopk.retopk_config(1, 28, 4, 128, 131584, 512, 32, 32, 4, 128, 0.85)
    assert lib.retopk_workspace_bytes(ctypes.byref(ok)) > 0
    for good in (retopk.retopk_config(1, 28, 4, 128, 1 << 23, 512, 32, 32, 4, 128, 0.85),
                 retopk.retopk_config(16, 28, 4, 128, 65792, 2048, 32, 32, 4, 128, 0.85, 0, 1),
                 retopk.retopk_config(1, 28, 4, 128, 131584, 512, 32, 32, 4, 128, 0.85, 0, 2),
                 retopk.retopk_config(1, 28, 4, 128, 5095424, 4096, 8, 2048, 4, 128, 0.85)):
        assert lib.retopk_workspace_bytes(ctypes.byref(good)) > 0
    bad = [
        retopk.retopk_config(1, 28, 4, 64, 1024, 512, 32, 32, 4, 128, 0.85),    # head_dim
        retopk.retopk_config(1, 28, 5, 128, 1024, 512, 32, 32, 4, 128, 0.85),   # Hq % Hkv
        retopk.retopk_config(1, 28, 4, 128, 1024, 512, 32, 32, 40, 128, 0.85),  # R > C
        retopk.retopk_config(1, 28, 4, 128, 1024, 0, 32, 32, 4, 128, 0.85),     # K
        retopk.retopk_config(1, 28, 4, 128, 1024, 512, 0, 32, 4, 128, 0.85),    # C
        retopk.retopk_config(1, 28, 4, 128, 1024, 512, 32, -1, 4, 128, 0.85),   # W
        retopk.retopk_config(1, 28, 4, 128, (1 << 23) + 1, 512, 32, 32, 4, 128, 0.85),  # max_len
        retopk.retopk_config(32, 28, 4, 128, 1 << 23, 512, 32, 32, 4, 128, 0.85),    # B*Hkv*max_len
        retopk.retopk_config(1, 28, 4, 128, 1024, 4096, 8, 0, 5, 128, 0.85),         # R*K + W
        # R*K + W = 18432: the bitmap slice of max_len / 8 positions no longer fits beside the lists
        retopk.retopk_config(1, 28, 4, 128, 5095424 + 1, 4096, 8, 2048, 4, 128, 0.85),
        retopk.retopk_config(1, 28, 4, 128, 1024, 512, 32, 32, 4, 128, float("nan")),
        retopk.retopk_config(1, 28, 4, 128, 1024, 512, 32, 32, 4, 128, 0.85, 2),   # retrieval mode
        retopk.retopk_config(1, 28, 4, 128, 1024, 512, 32, 32, 4, 128, 0.85, 0, 3),   # cluster size
        retopk.retopk_config(1, 28, 4, 128, 1024, 512, 32, 32, 4, 128, 0.85, 0, 16),
        # a fixed cluster of one CTA: the bitmap over all of max_len no longer fits
        retopk.retopk_config(1, 28, 4, 128, 1 << 23, 512, 32, 32, 4, 128, 0.85, 0, 1),
    ]
    for c in bad:
        assert lib.retopk_workspace_bytes(ctypes.byref(c)) == 0
    h = ctypes.c_void_p()
    assert lib.retopk_create(ctypes.byref(bad[0]), ctypes.c_void_p(256), 1 << 20, ctypes.byref(h)) == -2
    assert lib.retopk_create(ctypes.byref(ok), None, 1 << 20, ctypes.byref(h)) == -1
    assert lib.exact_topk_workspace_bytes(1, 28, 4, 128, 131584, 512) > 0
    assert lib.exact_topk_workspace_bytes(1, 28, 4, 96, 131584, 512) == 0
    assert lib.exact_topk_attention_step(None, None, None, None, 1, 28, 4, 128, 1024, 512,
                                         None, None, None, 0, None) == -1
    assert lib.retopk_strerror(-2).decode().startswith("unsupported")
    assert lib.retopk_decode_step(None, None, None, None, None, None, None) == -1
    assert lib.retopk_decode_step_host(None, None, None, None, None, None, None, None, None) == -1


def test_workspace_scales_with_context():
    lib = retopk.load()
    a = retopk.retopk_config(1, 28, 4, 128, 16640, 512, 32, 32, 4, 128, 0.85)
    b = retopk.retopk_config(1, 28, 4, 128, 131584, 512, 32, 32, 4, 128, 0.85)
    na, nb = lib.retopk_workspace_bytes(ctypes.byref(a)), lib.retopk_workspace_bytes(ctypes.byref(b))
    assert nb > na
    # scores + two candidate arrays per head dominate: about 12 bytes per key per query head
    assert nb < 28 * 131584 * 16 + (64 << 20)
