"""Planted mistakes: each mutant copy of oracle.c must fail at least one pin.

A mutant is oracle.c with one plausible slip (window off by one, the other stride
phase, a dropped scale, a transposed or wrong operand, a sign error, a missing causal
cut).  It is compiled to a temporary library and run against the same checks as the
real oracle; a mutant that passes every check would show a hole in the pins.
"""
import os
import subprocess

import pytest

import oracle
from pins import ATTENTION_CHECKS, BWD_CHECKS, COUNT_CHECKS, DECODE_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "window_off_by_one_rule": ("gap < m->window * m->dilation", "gap <= m->window * m->dilation"),
    "window_off_by_one_set": ("i - (m->window - 1) * m->dilation;", "i - m->window * m->dilation;"),
    "dilation_ignored_in_rule": ("if (llabs(gap) % m->dilation != 0) return 0;", ""),
    "dilation_phase_ignored": ("lo + (i - lo) % m->dilation;", "lo;"),
    "dilation_span_undilated": ("i - (m->window - 1) * m->dilation;", "i - (m->window - 1);"),
    "stride_phase_zero": ("j % m->stride == m->offset", "j % m->stride == 0"),
    "stride_start_zero": ("(m->stride > 0) ? m->offset : T", "(m->stride > 0) ? 0 : T"),
    "global_row_not_causal": ("const int64_t jmax = m->causal ? i : T - 1;",
                              "const int64_t jmax = T - 1;"),
    "radius_exclusive": ("llabs(gap) <= m->radius * m->dilation", "llabs(gap) < m->radius * m->dilation"),
    "radius_set_short": ("i + m->radius * m->dilation;", "i + m->radius * m->dilation - 1;"),
    "global_col_ignored": ("if (in_global(m, j)) return 1;", ""),
    "dropped_scale": ("s[a] = scale * acc;", "s[a] = acc;"),
    "normaliser_unshifted": ("l += exp(s[a] - mx);", "l += exp(s[a]);"),
    "lse_sign": ("LSE[r] = mx + log(l);", "LSE[r] = mx - log(l);"),
    "value_of_query_row": ("load_elem(V, dtype, j * d + k)", "load_elem(V, dtype, i * d + k)"),
    "key_transposed": ("load_elem(K, dtype, j * d + k)", "load_elem(K, dtype, k * d + j % d)"),
    "random_ignored": ("if (in_random(m, i, j)) return 1;", ""),
    "random_not_causal_in_set": ("int64_t cr = (jr <= jmax && jr < T) ? jr : INT64_MAX;",
                                 "int64_t cr = (jr < T) ? jr : INT64_MAX;"),
    "random_transposed": ("const int64_t qb = i / m->rand_block, kb = j / m->rand_block;",
                          "const int64_t qb = j / m->rand_block, kb = i / m->rand_block;"),
    "random_block_short": ("if (jr % m->rand_block == 0 || jr >= T)",
                           "if (jr % m->rand_block == m->rand_block - 1 || jr >= T)"),
    "first_key_skipped": ("for (int64_t a = 0; a < n; a++) l +=", "for (int64_t a = 1; a < n; a++) l +="),
}

# Slips in the gradient function, checked against the gradient pins only.
BWD_MUTANTS = {
    "bwd_softmax_jacobian_no_D": ("const double ds = a[t] * (da[t] - D);",
                                  "const double ds = a[t] * da[t];"),
    "bwd_D_unweighted": ("D += a[t] * acc;", "D += acc;"),
    "bwd_dV_unweighted": ("dV[j * d + k] += a[t] * load_elem(dO",
                          "dV[j * d + k] += load_elem(dO"),
    "bwd_dQ_no_scale": ("dq_row[k] += scale * ds", "dq_row[k] += ds"),
    "bwd_dK_uses_key": ("dK[j * d + k] += scale * ds * load_elem(Q, dtype, i * d + k);",
                        "dK[j * d + k] += scale * ds * load_elem(K, dtype, i * d + k);"),
    "bwd_dalpha_uses_key": ("acc += load_elem(dO, dtype, i * d + k) * load_elem(V, dtype, set[t] * d + k);",
                            "acc += load_elem(dO, dtype, i * d + k) * load_elem(K, dtype, set[t] * d + k);"),
    "bwd_logit_unscaled": ("    a[t] = scale * acc;\n    if (a[t] > mx)",
                           "    a[t] = acc;\n    if (a[t] > mx)"),
    "bwd_dV_to_query_row": ("dV[j * d + k] +=", "dV[i * d + k] +="),
    "bwd_rows_subset_shifted": ("bwd_row(&m, rows[r], d,", "bwd_row(&m, rows[r] / 2, d,"),
    # the same slips in the key-subset gradient, and ones of its own
    "bwd_keys_rule_transposed": ("if (!allowed(&m, i, j)) continue;",
                                 "if (!allowed(&m, j, i)) continue;"),
    "bwd_keys_D_unweighted": ("D += exp(s[t] - mx) / l * acc;", "D += acc;"),
    "bwd_keys_dK_no_scale": ("dk[k] += scale * ds *", "dk[k] += ds *"),
    "bwd_keys_dV_uses_value": ("dv[k] += alpha * load_elem(dO, dtype, i * d + k);",
                               "dv[k] += alpha * load_elem(V, dtype, i * d + k);"),
    "bwd_keys_normaliser_of_key_row": ("exp(scale * qk - rmax[i]) / rsum[i];",
                                       "exp(scale * qk - rmax[j]) / rsum[j];"),
    "bwd_keys_first_key_rows_missed": ("for (int64_t a = 0; a < n_keys; a++)\n      if (allowed",
                                       "for (int64_t a = 1; a < n_keys; a++)\n      if (allowed"),
}


def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    c = tmp_path / "mut.c"
    so = tmp_path / "libmut.so"
    c.write_text(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                           str(c), "-lm"])
    return str(so)


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_gradient_mutant_is_caught(oracle_mod, tmp_path, name):
    so = _build_mutant(tmp_path, *BWD_MUTANTS[name])
    failures = []
    with oracle.use_library(so):
        for check in BWD_CHECKS:
            failures += check()
            if failures:
                break
    assert failures, f"mutant {name} passed every gradient pin"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(oracle_mod, tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c = tmp_path / "mut.c"
    so = tmp_path / "libmut.so"
    c.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                           str(c), "-lm"])
    failures = []
    with oracle.use_library(str(so)):
        for check in COUNT_CHECKS + ATTENTION_CHECKS:
            failures += check()
            if failures:
                break
    assert failures, f"mutant {name} passed every pin"


# Slips in the decode function, checked against the decode pins only.
DECODE_MUTANTS = {
    "decode_slot_is_position": ("const int64_t slot = (p0 + a) % cap;\n    double acc",
                                "const int64_t slot = (p0 + a) % (cap + 1);\n    double acc"),
    "decode_window_one_short": ("t - w + 1 > 0 ? t - w + 1 : 0", "t - w + 2 > 0 ? t - w + 2 : 0"),
    "decode_value_slot_stale": ("const int64_t slot = (p0 + a) % cap;\n    const double wgt",
                                "const int64_t slot = (p0 + a + 1) % cap;\n    const double wgt"),
    "decode_unnormalised": ("exp(s[a] - mx) / l;", "exp(s[a] - mx);"),
}


@pytest.mark.parametrize("name", sorted(DECODE_MUTANTS))
def test_decode_mutant_is_caught(oracle_mod, tmp_path, name):
    so = _build_mutant(tmp_path, *DECODE_MUTANTS[name])
    failures = []
    with oracle.use_library(so):
        for check in DECODE_CHECKS:
            failures += check()
            if failures:
                break
    assert failures, f"mutant {name} passed every decode pin"
