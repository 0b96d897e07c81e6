"""spattn_fwd_static_scratch: the forward pass for callers that cannot allocate
device memory (their GPU memory is owned by another allocator, or they must not
pay for a cudaMalloc after start-up).  It takes its packing scratch from the
library's fixed 16 MiB device array instead of the plan's allocation.

Each case calls it twice in a row, through the C ABI, on different inputs, and
checks every output against spattn_fwd on the same inputs with the tolerances the
parity tests use.  The file is collected last so that a failure here does not hide
the other tests in a run that stops at the first failure."""
import math

import numpy as np
import pytest
import torch

import spattn_workloads as W
import sparse_masked_attention_plan_b300 as sp

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: dict(max_abs=1e-2, rel_l2=5e-3, lse=1e-4),
       torch.float32: dict(max_abs=1e-5, rel_l2=None, lse=1e-5)}


def close(got, want, lse_got, lse_want, dtype):
    t = TOL[dtype]
    g, w = got.float().cpu().double(), want.float().cpu().double()
    assert torch.isfinite(g).all()
    assert (g - w).abs().max().item() <= t["max_abs"]
    if t["rel_l2"] is not None:
        assert ((g - w).norm() / w.norm()).item() <= t["rel_l2"]
    assert (lse_got.cpu().double() - lse_want.cpu().double()).abs().max().item() <= t["lse"]


CASES = [
    ("t16k_r256_s16_g128", torch.bfloat16),  # strided + global columns and global rows
    ("t512_w128_s64", torch.bfloat16),
    ("t512_w128_s64", torch.float32),
    ("t512_w128_s0", torch.bfloat16),        # no packing: nothing taken from the array
]


@pytest.mark.parametrize("name,dtype", CASES, ids=[f"{n}-{str(d)[6:]}" for n, d in CASES])
def test_static_scratch_matches_allocating_entry(name, dtype):
    cfg = W.WORKLOADS[name]
    p = W.mask_params(name)
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    plan = sp.Plan(T, d, **p)
    scale = 1.0 / math.sqrt(d)
    for seed in (11, 12):  # two calls in a row, different inputs
        q, k, v = (x.cuda() for x in W.qkv(B, H, T, d, seed, dtype))
        o_ref, l_ref = sp.fwd(plan, q, k, v, scale)
        o, l = sp.fwd_static_scratch(plan, q, k, v, scale)
        torch.cuda.synchronize()
        plan.check_device()
        close(o, o_ref, l, l_ref, dtype)


def test_queued_calls_with_different_plans_each_finish_correctly():
    """Two static-scratch calls with different plans and shapes queued on one stream
    before a single sync: the second call's packing overwrites the shared array only
    after the first call's kernels have read it (stream order), so both outputs match
    spattn_fwd."""
    runs = []
    for name, seed in (("t16k_r256_s16_g128", 21), ("t512_w128_s64", 22)):
        cfg = W.WORKLOADS[name]
        B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
        plan = sp.Plan(T, d, **W.mask_params(name))
        q, k, v = (x.cuda() for x in W.qkv(B, H, T, d, seed, torch.bfloat16))
        runs.append((plan, q, k, v, 1.0 / math.sqrt(d)))
    torch.cuda.synchronize()
    outs = [sp.fwd_static_scratch(plan, q, k, v, sc) for plan, q, k, v, sc in runs]
    torch.cuda.synchronize()
    for (plan, q, k, v, sc), (o, l) in zip(runs, outs):
        plan.check_device()
        o_ref, l_ref = sp.fwd(plan, q, k, v, sc)
        torch.cuda.synchronize()
        close(o, o_ref, l, l_ref, torch.bfloat16)


def test_wait_timeout_is_reported_through_this_entry():
    """The plan's device-wait test hook and budget apply to this entry point too: a
    wait that runs out is reported as SPATTN_ERR_TIMEOUT, and the next call is right."""
    name = "t512_w128_s64"
    cfg = W.WORKLOADS[name]
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    plan = sp.Plan(T, d, **W.mask_params(name))
    q, k, v = (x.cuda() for x in W.qkv(B, H, T, d, 31, torch.bfloat16))
    plan.set_wait_budget(200_000)
    plan.test_wait_timeout(True)
    sp.fwd_static_scratch(plan, q, k, v, 0.125)
    with pytest.raises(sp.SpattnError) as ei:
        plan.check_device()
    assert ei.value.status == sp.ERR_TIMEOUT
    plan.test_wait_timeout(False)
    plan.set_wait_budget(8_000_000_000)
    o, l = sp.fwd_static_scratch(plan, q, k, v, 0.125)
    o_ref, l_ref = sp.fwd(plan, q, k, v, 0.125)
    torch.cuda.synchronize()
    plan.check_device()
    close(o, o_ref, l, l_ref, torch.bfloat16)


def test_oversize_request_is_rejected():
    # T=16384, stride 16: 1024 packed columns; d=128, B*H=64 bf16 needs
    # 64 * 2 * 1024 * 256 B = 32 MiB > 16 MiB
    plan = sp.Plan(16384, 128, causal=0, radius=256, stride=16)
    q = torch.zeros(1, 64, 16384, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(sp.SpattnError) as ei:
        sp.fwd_static_scratch(plan, q, q, q, 0.1)
    assert ei.value.status == sp.ERR_SHAPE
    assert b"16 MiB" in sp.lib().spattn_last_error()
