"""Each plausible slip in the oracle must be caught by at least one pin.

The oracle source is copied, one mistake is planted by text substitution, the
copy is compiled with gcc into a temporary directory, and the whole pin suite
(tests/oracle_pins.py) is run against it.  CPU only; the committed oracle is
never modified.
"""
import os
import subprocess
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "retopk_oracle.c")

MUTANTS = {
    "no_sqrt_d_scale": ("double inv = 1.0 / sqrt((double)d);", "double inv = 1.0;"),
    "topk_ties_to_higher_index": ("return (x->i < y->i) ? -1 : (x->i > y->i);",
                                  "return (x->i > y->i) ? -1 : (x->i < y->i);"),
    "topk_ascending": ("if (x->s > y->s) return -1;\n    if (x->s < y->s) return 1;",
                       "if (x->s < y->s) return -1;\n    if (x->s > y->s) return 1;"),
    "softmax_not_normalised": ("double w = exp(score[j] - m) / Z;", "double w = exp(score[j] - m);"),
    "value_row_by_position": ("const uint16_t *row = v + (int64_t)idx[j] * ld;",
                              "const uint16_t *row = v + (int64_t)j * ld;"),
    "window_off_by_one": ("int lo = L - W > 0 ? L - W : 0;", "int lo = L - W + 1 > 0 ? L - W + 1 : 0;"),
    "cosine_without_norms": ("? dot_bf(q, cached[c], d) / sqrt(nq * nc)", "? dot_bf(q, cached[c], d)"),
    "fallback_non_strict": ("(rho_max[h] < tau ||", "(rho_max[h] <= tau ||"),
    "t_dec_from_zero": ("int t_dec = seq[2] + 1;", "int t_dec = seq[2];"),
    "fifo_head_not_advanced": ("seq[0] = (head + 1) % C;", "seq[0] = head;"),
    "no_dedup": ("if (M == 0 || all[j] != out[M - 1])", "if (1)"),
    "init_not_causal": ("flen[h * C + c] = oracle_exact_one(qq, kb, NULL, d, p + 1,",
                        "flen[h * C + c] = oracle_exact_one(qq, kb, NULL, d, L0,"),
    "gqa_interleaved": ("const uint16_t *kb = k + (int64_t)(h / G) * max_len * d;\n        const uint16_t *vb",
                        "const uint16_t *kb = k + (int64_t)(h % Hkv) * max_len * d;\n        const uint16_t *vb"),
    "recall_ties_to_newer": ("        p[c].i = c;\n    }\n    qsort(p, (size_t)n, sizeof(pair_t), cmp_pair);",
                             "        p[c].i = n - 1 - c;\n    }\n    qsort(p, (size_t)n, sizeof(pair_t), cmp_pair);\n"
                             "    for (int c = 0; c < n; ++c) p[c].i = n - 1 - p[c].i;"),
    "reuse_ignores_window": ("    total += L - lo;", "    total += 0; lo = L;"),
    "fidelity_mass_unnormalised": ("            const double p = exp(eS[a] - mS) / ZS, ph = exp(eh[b] - mh) / Zh;",
                                   "            const double p = exp(eS[a] - mS), ph = exp(eh[b] - mh) / Zh;"),
    "recent_rho_max_over_all": ("        if (rho[n - 1 - r] > rmax)\n            rmax = rho[n - 1 - r];",
                                "        (void)0;\n    }\n    for (int r = 0; r < n; ++r) {\n"
                                "        if (rho[r] > rmax)\n            rmax = rho[r];"),
    "fidelity_recall_over_judged": ("    out[0] = nS > 0 ? (double)common / nS : 1.0;",
                                    "    out[0] = nh > 0 ? (double)common / nh : 1.0;"),
    "exact_step_gqa_interleaved": ("int b = bh / Hq, h = bh % Hq, hk = h / G;",
                                   "int b = bh / Hq, h = bh % Hq, hk = h % Hkv;"),
    "exact_step_batch_stride": ("const uint16_t *kb = k + ((int64_t)b * Hkv + hk) * max_len * d;",
                                "const uint16_t *kb = k + ((int64_t)hk) * max_len * d;"),
    "exact_step_first_length": ("sup_len[bh] = oracle_exact_one(q + (int64_t)bh * d, kb, vb, d, L[b], d, K, s,",
                                "sup_len[bh] = oracle_exact_one(q + (int64_t)bh * d, kb, vb, d, L[0], d, K, s,"),
    "aos_values_from_k": ("    oracle_sparse_attention(s, sup, n, v, ld, d, out);\n    free(s);",
                          "    oracle_sparse_attention(s, sup, n, k, ld, d, out);\n    free(s);"),
    "overlap_over_own_length": ("    return (double)common / K;", "    return (double)common / nt;"),
    "coverage_recent_instead_of_similar": ("    oracle_recall(q, prev_q, n_prev, d, R, rho, chosen);",
                                           "    oracle_recall_recent(q, prev_q, n_prev, d, R, rho, chosen);"),
    "coverage_top1_only": ("    const double cov = oracle_overlap(St, nt, U, nu, K);",
                           "    const double cov = oracle_overlap(St, nt, sp[0], ln[0], K);"),
}


_RUNNER = """
import sys
sys.path.insert(0, sys.argv[2])
sys.path.insert(0, sys.argv[3])
import oracle, oracle_pins as P
lib = oracle.load(sys.argv[1])
print("LOADED", flush=True)
caught = []
for pin in P.ALL_PINS:
    try:
        pin(lib)
    except AssertionError:
        caught.append(pin.__name__)
print("CAUGHT", ",".join(caught))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    """The pins run in a child process: a planted mistake that corrupts memory
    (e.g. an allocation sized from a wrong window bound) then ends that process
    instead of this one, and counts as caught."""
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-ffp-contract=off", str(mut), "-o", str(so), "-lm"])
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, "-c", _RUNNER, str(so), os.path.dirname(here), here],
                       capture_output=True, text=True, timeout=600)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("CAUGHT")]
    # a crash counts only once the mutant library is loaded and the pins run
    crashed = r.returncode != 0 and "LOADED" in r.stdout
    assert "LOADED" in r.stdout, f"pin runner failed before the pins ran:\n{r.stderr[-2000:]}"
    caught = lines[0].split(" ", 1)[1] if lines and len(lines[0].split(" ", 1)) > 1 else ""
    assert crashed or caught, f"mutant {name} passed every pin"
