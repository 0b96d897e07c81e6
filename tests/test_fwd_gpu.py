"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element.  Small cases compare every row of every
head; the full-size workloads compare sampled rows (edges, window and block
boundaries, global rows) of a few heads, in the launch configuration the
benchmark times."""
import math

import numpy as np
import pytest
import torch

import spattn_workloads as W
import sparse_masked_attention_plan_b300 as sp
from gpu_cases import edge_rows, run_and_compare, workload

pytestmark = pytest.mark.gpu

SMALL = ["t512_w128_s0", "t512_w128_s64", "t512_full_causal"]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("name", SMALL)
def test_small_workloads_every_row(oracle_mod, name, dtype):
    cfg, p = workload(name)
    run_and_compare(cfg["B"], cfg["H"], cfg["T"], cfg["d"], p, dtype, seed=0)


SWEEP = [
    # (B, H, T, d, mask)
    (1, 2, 1, 64, dict(causal=1, window=0)),
    (1, 1, 37, 128, dict(causal=1, window=5)),
    (2, 3, 128, 64, dict(causal=1, window=1)),
    (1, 2, 129, 128, dict(causal=0, radius=0)),
    (1, 2, 300, 64, dict(causal=1, window=300)),
    (1, 2, 300, 128, dict(causal=1, window=77, stride=3, offset=2)),
    (2, 1, 513, 64, dict(causal=0, radius=40, stride=64, offset=63, global_pos=[0, 77, 512])),
    (1, 2, 777, 128, dict(causal=1, window=130, stride=17, offset=5,
                          global_pos=[0, 3, 129, 500, 776])),
    (1, 2, 1000, 64, dict(causal=0, radius=-1, global_pos=[999])),
    (1, 1, 1000, 128, dict(causal=0, radius=128, stride=16, offset=0,
                           global_pos=list(range(0, 1000, 97)))),
    (1, 2, 1100, 64, dict(causal=1, window=0, stride=64)),
    (1, 1, 1300, 128, dict(causal=0, radius=300, global_pos=list(range(5, 1300, 4)))),
    # dilated local windows ("Attention variants" dilated(n, w, d)), alone and mixed
    (1, 2, 1000, 64, dict(causal=1, window=64, dilation=2)),
    (2, 1, 777, 128, dict(causal=1, window=50, dilation=5, stride=64, offset=3,
                          global_pos=[1, 400])),
    (1, 2, 900, 64, dict(causal=0, radius=30, dilation=4, stride=100, offset=0,
                         global_pos=[17, 600])),
    (1, 1, 513, 128, dict(causal=1, window=0, dilation=3)),
    (1, 2, 1024, 128, dict(causal=0, radius=50, dilation=4)),
    (2, 1, 600, 64, dict(causal=1, window=70, dilation=6)),
    # BigBird random blocks ("Sparse and sliding-window attention", Block-sparse
    # attention: BigBird): alone, with globals, with strided columns, causal
    (1, 2, 700, 64, dict(causal=0, radius=40, global_pos=[0, 1, 650], rand_block=64,
                         rand_pairs=[(0, 9), (1, 5), (3, 0), (3, 10), (10, 2), (10, 10)])),
    (2, 1, 520, 128, dict(causal=1, window=70, stride=33, offset=4, rand_block=16,
                          rand_pairs=[(20, 3), (20, 19), (31, 0), (32, 32), (5, 30)])),
    (1, 2, 600, 128, dict(causal=0, radius=0, rand_block=128, rand_pairs=[(0, 4), (4, 0), (2, 2)])),
    (1, 1, 1100, 64, dict(causal=1, window=96, global_pos=list(range(64)), rand_block=32,
                          rand_pairs=[(q, (7 * q + 3) % (q + 1)) for q in range(35)])),
]


@pytest.mark.parametrize("mask,T,views", [
    (dict(causal=1, window=64, dilation=2), 1000, True),
    (dict(causal=0, radius=50, dilation=4), 1024, True),
    (dict(causal=1, window=64, dilation=3), 1000, False),          # 3 does not divide T
    (dict(causal=1, window=64, dilation=2, stride=16), 1000, False),  # strided columns
])
def test_dilated_view_is_used_exactly_when_it_applies(mask, T, views):
    plan = sp.Plan(T, 64, **mask)
    items, _, products = plan.schedule(2)
    assert (len(items) > 0) == views
    if views:  # the residue classes partition the rows: same pair count, fewer products
        _, _, plain = plan.schedule(0)
        assert products <= plain


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("k", range(len(SWEEP)))
def test_sweep_every_row(oracle_mod, k, dtype):
    B, H, T, d, mask = SWEEP[k]
    run_and_compare(B, H, T, d, mask, dtype, seed=k + 1)


@pytest.mark.parametrize("name", ["t2048_w256_s0", "t2048_w256_s64"])
def test_t2048_workloads(oracle_mod, name):
    cfg, p = workload(name)
    run_and_compare(cfg["B"], cfg["H"], cfg["T"], cfg["d"], p, "bf16", seed=1,
                    heads=[(0, 0), (1, 5), (3, 11)])


@pytest.mark.parametrize("name", ["t32k_w4096", "t16k_r256_s16_g128", "t8k_full_causal",
                                  "t128k_w4096_s1024", "t4096_bigbird", "t32k_w512_d2"])
def test_large_workloads_sampled_rows(oracle_mod, name):
    cfg, p = workload(name)
    T = cfg["T"]
    rows = W.sample_rows(T, 192, seed=3, must=edge_rows(T, p))
    heads = [(0, 0), (cfg["B"] - 1, cfg["H"] - 1)]
    run_and_compare(cfg["B"], cfg["H"], T, cfg["d"], p, "bf16", seed=2, heads=heads,
                    rows=rows)


def test_scale_and_repeat_calls_are_stable(oracle_mod):
    cfg, p = workload("t512_w128_s64")
    plan = sp.Plan(cfg["T"], cfg["d"], **p)
    for scale in (0.05, 1.0 / math.sqrt(cfg["d"]), 0.3):
        run_and_compare(cfg["B"], cfg["H"], cfg["T"], cfg["d"], p, "bf16", seed=9, scale=scale,
                        plan=plan)


def test_bad_arguments_are_rejected():
    plan = sp.Plan(256, 64, causal=1, window=16)
    q = torch.zeros(1, 1, 256, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(sp.SpattnError) as ei:
        sp.fwd(plan, q, q, q, -1.0)
    assert ei.value.status == sp.ERR_INVALID_SPEC
    flat = torch.zeros(256 * 64 + 8, device="cuda", dtype=torch.bfloat16)
    qm = flat[1:1 + 256 * 64].view(1, 1, 256, 64)  # 2 bytes off a 16-byte boundary
    with pytest.raises(sp.SpattnError) as ei:
        sp.fwd(plan, qm, qm, qm, 1.0)
    assert ei.value.status == sp.ERR_ALIGN
    with pytest.raises(sp.SpattnError) as ei:
        sp.Plan(256, 96, causal=1, window=16)
    assert ei.value.status == sp.ERR_SHAPE


def test_host_buffer_entry_matches_device_entry(oracle_mod):
    cfg, p = workload("t512_w128_s64")
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    Q, K, V = W.qkv(B, H, T, d, 4, torch.bfloat16)
    plan = sp.Plan(T, d, **p)
    o_dev, l_dev = sp.fwd(plan, Q.cuda(), K.cuda(), V.cuda(), 0.125)
    hq, hk, hv = (x.pin_memory() for x in (Q, K, V))
    ho = torch.empty_like(Q).pin_memory()
    hl = torch.empty(B, H, T, dtype=torch.float32).pin_memory()
    bufs = (torch.empty_like(Q, device="cuda"), torch.empty_like(K, device="cuda"),
            torch.empty_like(V, device="cuda"), torch.empty_like(Q, device="cuda"),
            torch.empty(B, H, T, dtype=torch.float32, device="cuda"))
    sp.fwd_host(plan, hq, hk, hv, 0.125, ho, hl, bufs)
    assert torch.equal(ho, o_dev.cpu())
    assert torch.equal(hl, l_dev.cpu())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,with_lse", [(3, 5, True), (1, 1, True), (2, 8, False), (1, 19, True),
                                           (2, 19, True)])
def test_host_buffer_pipeline_chunks(B, H, with_lse, dtype):
    """The host-buffer entry splits the (batch, head) units into chunks whose copies
    overlap the forward of their neighbours: unit counts that do and do not divide
    evenly (15, 16, 19, a single unit), packed strided / global columns (plan scratch
    reused across chunks), with and without LSE, both dtypes, equal bit for bit to one
    device call; and a second call on the same plan after work queued on the stream
    writes the device buffers."""
    T, d = 700, 64
    plan = sp.Plan(T, d, causal=1, window=150, stride=48, offset=7, global_pos=[3, 333])
    Q, K, V = W.qkv(B, H, T, d, 21, dtype)
    o_dev, l_dev = sp.fwd(plan, Q.cuda(), K.cuda(), V.cuda(), 0.1)
    torch.cuda.synchronize()  # the plan's scratch is shared with the calls below
    hq, hk, hv = (x.pin_memory() for x in (Q, K, V))
    ho = torch.empty_like(Q).pin_memory()
    hl = torch.empty(B, H, T, dtype=torch.float32).pin_memory() if with_lse else None
    qd, kd, vd, od = (torch.empty_like(Q, device="cuda") for _ in range(4))
    ld = torch.empty(B, H, T, dtype=torch.float32, device="cuda") if with_lse else None
    s = torch.cuda.Stream()
    for rep in range(2):
        with torch.cuda.stream(s):
            for x in (qd, kd, vd, od):  # queued before the call: the copies must follow it
                x.fill_(7.0)
        sp.fwd_host(plan, hq, hk, hv, 0.1, ho, hl, (qd, kd, vd, od, ld), stream=s)
        assert torch.equal(ho, o_dev.cpu()), f"call {rep}"
        if with_lse:
            assert torch.equal(hl, l_dev.cpu()), f"call {rep}"
    plan.check_device()
