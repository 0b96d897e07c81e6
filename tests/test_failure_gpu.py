"""Failure detection without a GPU fault: a device-side wait that runs out of its
budget is reported to the host as SPATTN_ERR_TIMEOUT, and the context stays usable.

The kernel's test hook makes its MMA warp wait on a barrier that nothing signals,
with a short budget (2e5 cycles, ~0.1 ms); every other wait then runs out too, the
kernel drains its copies, frees its tensor memory and returns."""
import math

import numpy as np
import pytest
import torch

import oracle
import spattn_workloads as W
import sparse_masked_attention_plan_b300 as sp

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives(oracle_mod):
    T, d = 256, 64
    mask = dict(causal=1, window=64, stride=32, offset=5)
    plan = sp.Plan(T, d, **mask)
    Q, K, V = W.qkv(1, 1, T, d, 21, torch.bfloat16)
    q, k, v = (x.cuda() for x in (Q, K, V))
    plan.set_wait_budget(200_000)
    plan.test_wait_timeout(True)
    sp.fwd(plan, q, k, v, 0.125)
    with pytest.raises(sp.SpattnError) as ei:
        plan.check_device()
    assert ei.value.status == sp.ERR_TIMEOUT
    # the error word was cleared and the context is still usable
    plan.test_wait_timeout(False)
    plan.set_wait_budget(8_000_000_000)
    o, lse = sp.fwd(plan, q, k, v, 0.125)
    torch.cuda.synchronize()
    plan.check_device()
    m = oracle.Mask(T, 1, 64, -1, 32, 5, [])
    Oref, Lref = oracle.attention(m, oracle.bf16_bits(Q[0, 0]), oracle.bf16_bits(K[0, 0]),
                                  oracle.bf16_bits(V[0, 0]), 0.125)
    got = o[0, 0].float().cpu().numpy().astype(np.float64)
    assert np.abs(got - Oref).max() <= 1e-2
    assert np.abs(lse[0, 0].cpu().numpy() - Lref).max() <= 1e-4


def test_wait_budget_must_be_positive():
    plan = sp.Plan(128, 64, causal=1, window=8)
    with pytest.raises(sp.SpattnError) as ei:
        plan.set_wait_budget(0)
    assert ei.value.status == sp.ERR_SHAPE
