"""The CPU oracle against the pages' printed numbers, closed forms and library routines."""
import pytest

import oracle
import spattn_workloads as W
from pins import (ATTENTION_CHECKS, BWD_CHECKS, COUNT_CHECKS, DECODE_CHECKS, closed_form_pairs,
                  dense_of)


@pytest.mark.parametrize("check", COUNT_CHECKS + ATTENTION_CHECKS + BWD_CHECKS + DECODE_CHECKS,
                         ids=lambda f: f.__name__)
def test_pin(oracle_mod, check):
    bad = check()
    assert not bad, "\n".join(bad[:20])


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_workload_pair_counts_closed_form(oracle_mod, name):
    """Every benchmark workload's pair count: oracle enumeration == inclusion-exclusion."""
    cfg = W.WORKLOADS[name]
    p = W.mask_params(name)
    m = oracle.Mask.from_params(cfg["T"], p)
    assert m.validate() == 0
    if p.get("rand_block"):
        # random blocks: the numpy dense restatement (the inclusion-exclusion form has
        # no random term)
        cf = int(dense_of(dict(T=cfg["T"], **p)).sum())
    else:
        cf = closed_form_pairs(cfg["T"], p["causal"], p["window"], p["radius"], p["stride"],
                               p["offset"], p["global_pos"], p["dilation"])
    assert m.count_pairs() == cf


def test_known_workload_counts(oracle_mod):
    # 32K / W=4096: E = N W - W (W-1) / 2 (the page's 134M is the N W approximation)
    assert oracle.Mask(32768, 1, 4096).count_pairs() == 125_831_168
    # 16K bidirectional r=256, s=16, 128 seeded globals: the page's additive ~27M
    p = W.mask_params("t16k_r256_s16_g128")
    m = oracle.Mask.from_params(16384, p)
    n = m.count_pairs()
    assert 27_000_000 < n < 30_000_000
    assert n == 28_375_329
