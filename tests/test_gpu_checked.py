"""The RETOPK_CHECKED build (every gathered K / V row index range-checked
against the sequence length before the load) computes the same results as the
ordinary build and raises no status bit on valid inputs; the fidelity
diagnostic skips, and reports, support entries that would address past the
cache."""
import ctypes

import numpy as np
import pytest
import torch

from top_sparse_attention_exact_gb300 import _build, retopk, synth
from top_sparse_attention_exact_gb300.runner import DecodeRun, ExactRun

pytestmark = pytest.mark.gpu


def _run(w, arrays):
    dr = DecodeRun(w, arrays=arrays)
    outs, sups, paths = [], [], []
    for t in range(w.steps):
        dr.step(t)
        d = dr.ctx.retopk_get_diagnostics()
        outs.append(dr.out.clone())
        sups.append(d["support"].copy())
        paths.append(d["path"].copy())
    ex = ExactRun(dr)
    ex.step(dr.q_dec[w.steps - 1])
    torch.cuda.synchronize()
    res = dict(out=torch.stack(outs).cpu(), support=np.stack(sups), path=np.stack(paths),
               exact_out=ex.out.cpu(), exact_idx=ex.idx.cpu(), status=dr.ctx.retopk_get_status())
    dr.ctx.close()   # with the library that made it
    return res


def test_checked_build_matches_the_ordinary_build():
    # cache initialisation, reuse / fallback / refresh steps and a stateless
    # exact step, each through both libraries on the same inputs
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=4096, steps=12, T_r=5, name="checked")
    arrays = synth.generate(w)
    saved = retopk._lib
    try:
        retopk._lib = retopk._declare(ctypes.CDLL(_build.build(checked=True)))
        chk = _run(w, arrays)
    finally:
        retopk._lib = saved
    ref = _run(w, arrays)
    assert chk["status"] == 0 and ref["status"] == 0
    assert (ref["path"] == 0).any() and (ref["path"] != 0).any()   # both paths ran
    assert torch.equal(chk["out"], ref["out"])
    assert np.array_equal(chk["support"], ref["support"])
    assert np.array_equal(chk["path"], ref["path"])
    assert torch.equal(chk["exact_out"], ref["exact_out"])
    assert torch.equal(chk["exact_idx"], ref["exact_idx"])


def test_fidelity_skips_rows_outside_the_cache():
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=2048, steps=2, name="fid_range")
    dr = DecodeRun(w)
    ex = ExactRun(dr)
    dr.step(0)
    ex.step(dr.q_dec[0])
    dr.ctx.retopk_fidelity(dr.q_dec[0], dr.k_cache, ex.idx, ex.out, dr.out)
    torch.cuda.synchronize()
    assert dr.ctx.retopk_get_status() == 0
    bad = ex.idx.clone()
    bad[0, 3, 5] = dr.max_len + 7
    m = dr.ctx.retopk_fidelity(dr.q_dec[0], dr.k_cache, bad, ex.out, dr.out)
    torch.cuda.synchronize()
    assert dr.ctx.retopk_get_status(clear=True) == retopk.STATUS_GATHER
    assert np.isfinite(m.cpu().numpy()).all()
