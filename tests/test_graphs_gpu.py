"""CUDA-graph capture of the library's calls: every entry point is host work plus
launches on the caller's stream (tensor maps are encoded on the host and passed by
value), so after a first call (which may allocate the plan's scratch) a forward, a
backward and a whole decode step (append, decode, combine) can be captured once and
replayed, with new inputs written into the same buffers between replays."""
import math

import numpy as np
import pytest
import torch

import spattn_workloads as W
import sparse_masked_attention_plan_b300 as sp

pytestmark = pytest.mark.gpu


def _replay_matches(capture, direct, refill, n=3):
    """Capture `capture()` into a graph; for n rounds write new inputs (`refill(k)`),
    replay, and compare the graph's outputs with a direct call's, bit for bit."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        capture()  # first call outside the capture: scratch, attributes
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = capture()
    for k in range(n):
        refill(k)
        g.replay()
        torch.cuda.synchronize()
        got = [o.clone() for o in outs]
        want = direct()
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a, b), f"replay {k} differs from a direct call"


def test_forward_graph_replay():
    B, H, T, d = 2, 4, 1500, 128
    mask = dict(causal=1, window=300, stride=64, offset=5, global_pos=[7, 800])
    plan = sp.Plan(T, d, **mask)
    q, k, v = (x.cuda() for x in W.qkv(B, H, T, d, 0))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    scale = 1 / math.sqrt(d)

    def capture():
        sp.fwd(plan, q, k, v, scale, out=o, lse=lse)
        return [o, lse]

    def direct():
        return list(sp.fwd(plan, q, k, v, scale))

    def refill(r):
        for x, y in zip((q, k, v), W.qkv(B, H, T, d, 10 + r)):
            x.copy_(y.cuda())

    _replay_matches(capture, direct, refill)
    plan.check_device()


def test_backward_graph_replay():
    B, H, T, d = 1, 2, 1200, 64
    mask = dict(causal=0, radius=100, stride=40, offset=3, global_pos=[0, 600])
    plan = sp.Plan(T, d, **mask)
    q, k, v = (x.cuda() for x in W.qkv(B, H, T, d, 1))
    do = W.grad_out(B, H, T, d, 1).cuda()
    scale = 1 / math.sqrt(d)
    o, lse = sp.fwd(plan, q, k, v, scale)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))

    def capture():
        sp.bwd(plan, q, k, v, o, lse, do, scale, dq, dk, dv)
        return [dq, dk, dv]

    def direct():
        return list(sp.bwd(plan, q, k, v, o, lse, do, scale))

    def refill(r):
        do.copy_(W.grad_out(B, H, T, d, 20 + r).cuda())

    _replay_matches(capture, direct, refill)
    plan.check_device()


def test_decode_step_graph_replay():
    """A generation loop as a graph: the positions are a device tensor the graph reads,
    so advancing them in place between replays moves the step along the sequence."""
    B, Hq, Hkv, cap, d = 4, 8, 2, 256, 128
    c = sp.DecodeCache(B, Hq, Hkv, cap, d, window=200)
    g = torch.Generator().manual_seed(5)
    c.K.copy_(torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16).cuda())
    c.V.copy_(torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16).cuda())
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).cuda()
    kn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    vn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    pos = torch.tensor(np.array([5, 255, 256, 1000]), dtype=torch.int64, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, device="cuda")

    def capture():
        c.append(kn, vn, pos)
        c.step(q, pos, 0.09, out=out, lse=lse)
        return [out, lse]

    def direct():
        # the graph already appended this step's rows; decoding again reads the same cache
        return list(c.step(q, pos, 0.09))

    def refill(r):
        pos.add_(1)
        q.copy_(torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).cuda())
        kn.copy_(torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda())

    _replay_matches(capture, direct, refill)
    c.check()


def test_fused_decode_step_graph_replay():
    """The same generation loop through spattn_decode_append (the decode kernel appends
    the step's rows): each replay's output equals a direct decode of the cache the replay
    left behind, at the advanced positions."""
    B, Hq, Hkv, cap, d = 4, 8, 2, 256, 128
    c = sp.DecodeCache(B, Hq, Hkv, cap, d, window=200)
    g = torch.Generator().manual_seed(6)
    c.K.copy_(torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16).cuda())
    c.V.copy_(torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16).cuda())
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).cuda()
    kn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    vn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    pos = torch.tensor(np.array([7, 255, 256, 999]), dtype=torch.int64, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, device="cuda")

    def capture():
        c.append_step(kn, vn, q, pos, 0.09, out=out, lse=lse)
        return [out, lse]

    def direct():
        return list(c.step(q, pos, 0.09))

    def refill(r):
        pos.add_(1)
        q.copy_(torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).cuda())
        kn.copy_(torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda())
        vn.copy_(torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda())

    _replay_matches(capture, direct, refill)
    c.check()
