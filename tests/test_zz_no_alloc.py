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


def test_oversize_request_is_rejected():
    # T=16384, stride 16: 1024 packed columns; d=128, B*H=64 bf16 needs
    # 64 * 2 * 1024 * 256 B = 32 MiB > 16 MiB
    plan = sp.Plan(16384, 128, causal=0, radius=256, stride=16)
    q = torch.zeros(1, 64, 16384, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(sp.SpattnError) as ei:
        sp.fwd_static_scratch(plan, q, q, q, 0.1)
    assert ei.value.status == sp.ERR_SHAPE
    assert b"16 MiB" in sp.lib().spattn_last_error()
