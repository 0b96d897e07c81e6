"""Decode parity: one generation step against a ring-buffer KV cache (spattn_kv_append +
spattn_decode through the C ABI) against the fp64 oracle's decode step, and a whole
generation loop against rows of the forward oracle on the full sequence.  The fused
step (spattn_decode_append, the append done by the decode kernel for bf16) must give
exactly the results and cache contents of the two calls."""
import math

import numpy as np
import pytest
import torch

import oracle
import spattn_workloads as W
import sparse_masked_attention_plan_b300 as sp
from gpu_cases import TOL, host_view, torch_dtype

pytestmark = pytest.mark.gpu

POISON = 3000.0  # written to every slot a step must not read


def _fill_cache(B, Hkv, cap, d, pos, window, dtype, g):
    """Random N(0,1) rows in the slots each batch row's step reads, POISON elsewhere."""
    K = torch.full((B, Hkv, cap, d), POISON)
    V = torch.full((B, Hkv, cap, d), -POISON)
    for b, t in enumerate(pos):
        if t < 0:
            continue
        w = window or cap
        for p in range(max(0, t - w + 1), t + 1):
            K[b, :, p % cap] = torch.randn(Hkv, d, generator=g)
            V[b, :, p % cap] = torch.randn(Hkv, d, generator=g)
    return K.to(torch_dtype(dtype)), V.to(torch_dtype(dtype))


def _compare(out, lse, q, K, V, pos, window, scale, dtype, G):
    tol = TOL[dtype]
    B, Hq, d = q.shape
    cap = K.shape[2]
    for b in range(B):
        for h in range(Hq):
            ref, ref_lse = oracle.decode(host_view(q[b, h]), host_view(K[b, h // G]),
                                         host_view(V[b, h // G]), int(pos[b]), window or cap,
                                         scale)
            got = out[b, h].astype(np.float64)
            err = np.abs(got - ref).max()
            assert err <= tol["max_abs"], f"(b, h) = {(b, h)} t = {pos[b]}: max-abs {err:.3g}"
            if tol["rel_l2"] is not None and np.linalg.norm(ref) > 0:
                rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
                assert rel <= tol["rel_l2"], f"(b, h) = {(b, h)}: rel-L2 {rel:.3g}"
            if ref_lse == -math.inf:
                assert lse[b, h] == -math.inf and not got.any()
            else:
                assert abs(lse[b, h] - ref_lse) <= tol["lse"], f"(b, h) = {(b, h)} LSE"


CASES = [
    # (B, Hq, Hkv, cap, window, d, positions)
    (3, 8, 2, 4096, 0, 128, [5, 4095, 100000]),
    (2, 4, 4, 100, 37, 64, [36, 250]),
    (1, 8, 1, 300, 300, 128, [1000]),
    (2, 4, 2, 64, 1, 64, [0, 77]),
    (2, 2, 1, 130, 65, 128, [-1, 129]),
    (4, 16, 8, 1000, 999, 64, [998, 999, 1500, 3]),
    (1, 2, 2, 5000, 4000, 128, [4999]),
    (2, 16, 2, 200, 150, 64, [199, 1000]),  # G = 8 at d = 64
    (1, 8, 2, 512, 0, 64, [600]),           # G = 4 at d = 64, full window, wrapped
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("k", range(len(CASES)))
def test_decode_step(oracle_mod, k, dtype):
    B, Hq, Hkv, cap, window, d, pos = CASES[k]
    g = torch.Generator().manual_seed(500 + k)
    K, V = _fill_cache(B, Hkv, cap, d, pos, window, dtype, g)
    q = torch.randn(B, Hq, d, generator=g).to(torch_dtype(dtype))
    scale = 1.0 / math.sqrt(d)
    c = sp.DecodeCache(B, Hq, Hkv, cap, d, window=window, dtype=torch_dtype(dtype))
    c.K.copy_(K.cuda())
    c.V.copy_(V.cuda())
    p = torch.tensor(pos, dtype=torch.int64, device="cuda")
    out, lse = c.step(q.cuda(), p, scale)
    c.check()
    _compare(out.float().cpu().numpy(), lse.cpu().numpy(), q, K, V, pos, window, scale, dtype,
             Hq // Hkv)


def test_append_writes_the_ring_slot():
    B, Hkv, cap, d = 3, 2, 50, 64
    c = sp.DecodeCache(B, 4, Hkv, cap, d)
    g = torch.Generator().manual_seed(1)
    before = torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16)
    c.K.copy_(before.cuda())
    c.V.copy_(before.cuda())
    kn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16)
    pos = [7, 149, -3]
    c.append(kn.cuda(), vn.cuda(), torch.tensor(pos, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    want_k, want_v = before.clone(), before.clone()
    for b, t in enumerate(pos):
        if t >= 0:
            want_k[b, :, t % cap] = kn[b]
            want_v[b, :, t % cap] = vn[b]
    assert torch.equal(c.K.cpu(), want_k) and torch.equal(c.V.cpu(), want_v)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("k", range(len(CASES)))
def test_fused_append_step_equals_append_then_step(k, dtype):
    B, Hq, Hkv, cap, window, d, pos = CASES[k]
    g = torch.Generator().manual_seed(700 + k)
    K, V = _fill_cache(B, Hkv, cap, d, pos, window, dtype, g)
    q = torch.randn(B, Hq, d, generator=g).to(torch_dtype(dtype)).cuda()
    kn = torch.randn(B, Hkv, d, generator=g).to(torch_dtype(dtype)).cuda()
    vn = torch.randn(B, Hkv, d, generator=g).to(torch_dtype(dtype)).cuda()
    p = torch.tensor(pos, dtype=torch.int64, device="cuda")
    caches = [sp.DecodeCache(B, Hq, Hkv, cap, d, window=window, dtype=torch_dtype(dtype))
              for _ in range(2)]
    for c in caches:
        c.K.copy_(K.cuda())
        c.V.copy_(V.cuda())
    caches[0].append(kn, vn, p)
    o1, l1 = caches[0].step(q, p, 0.11)
    o2, l2 = caches[1].append_step(kn, vn, q, p, 0.11)
    for c in caches:
        c.check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(caches[0].K, caches[1].K) and torch.equal(caches[0].V, caches[1].V)


def test_fused_append_full_size_equals_two_calls():
    """B = 8 sequences of the benchmark's shape (Hq 32, Hkv 8, cap = W = 4096, d = 128):
    several fused steps in a row equal the two-call steps, outputs and caches."""
    B, Hq, Hkv, cap, d = 8, 32, 8, 4096, 128
    g = torch.Generator().manual_seed(23)
    K = torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16).cuda()
    V = torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16).cuda()
    pos0 = torch.from_numpy(np.random.default_rng(4).integers(cap, 10 ** 6, size=B)).cuda()
    caches = [sp.DecodeCache(B, Hq, Hkv, cap, d) for _ in range(2)]
    for c in caches:
        c.K.copy_(K)
        c.V.copy_(V)
    for s in range(3):
        q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16).cuda()
        kn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda()
        vn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16).cuda()
        p = pos0 + s
        caches[0].append(kn, vn, p)
        o1, l1 = caches[0].step(q, p, 1 / math.sqrt(d))
        o2, l2 = caches[1].append_step(kn, vn, q, p, 1 / math.sqrt(d))
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for c in caches:
        c.check()
    assert torch.equal(caches[0].K, caches[1].K) and torch.equal(caches[0].V, caches[1].V)


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_generation_loop_matches_sequence_rows(oracle_mod, dtype, fused):
    """Append + decode token by token with a cache smaller than the sequence; every
    step must equal row t of the forward oracle over the whole sequence with the
    causal window."""
    T, Hq, Hkv, cap, window, d = 300, 4, 2, 64, 48, 64
    G = Hq // Hkv
    g = torch.Generator().manual_seed(9)
    Q = torch.randn(Hq, T, d, generator=g).to(torch_dtype(dtype))
    K = torch.randn(Hkv, T, d, generator=g).to(torch_dtype(dtype))
    V = torch.randn(Hkv, T, d, generator=g).to(torch_dtype(dtype))
    scale = 0.2
    c = sp.DecodeCache(1, Hq, Hkv, cap, d, window=window, dtype=torch_dtype(dtype))
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    outs, lses = [], []
    for t in range(T):
        p = torch.tensor([t], dtype=torch.int64, device="cuda")
        if fused:
            o, l = c.append_step(Kd[None, :, t].contiguous(), Vd[None, :, t].contiguous(),
                                 Qd[None, :, t].contiguous(), p, scale)
        else:
            c.append(Kd[None, :, t].contiguous(), Vd[None, :, t].contiguous(), p)
            o, l = c.step(Qd[None, :, t].contiguous(), p, scale)
        outs.append(o[0].float().cpu())
        lses.append(l[0].cpu())
    c.check()
    out = torch.stack(outs, 1).numpy()  # [Hq, T, d]
    lse = torch.stack(lses, 1).numpy()
    m = oracle.Mask(T, 1, window)
    tol = TOL[dtype]
    for h in range(Hq):
        O, L = oracle.attention(m, host_view(Q[h]), host_view(K[h // G]), host_view(V[h // G]),
                                scale)
        err = np.abs(out[h] - O).max()
        assert err <= tol["max_abs"], f"head {h}: max-abs {err:.3g}"
        assert np.abs(lse[h] - L).max() <= tol["lse"], f"head {h}: LSE"


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name", ["decode_b32_w4096", "decode_b8_w4096"])
def test_full_size_every_head(oracle_mod, name, fused):
    """The benchmark's decode configurations (cap = W = 4096, Hq = 32, Hkv = 8, d = 128)
    with every batch row past the cap at its own position: every (b, h) of the step,
    element by element, against the oracle at the bf16 tolerances (max-abs, rel-L2,
    LSE).  With `fused` the step's rows go in through spattn_decode_append, so the
    oracle reads the cache with those rows written into their ring slots."""
    cfg = W.DECODE_WORKLOADS[name]
    B, Hq, Hkv, cap, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["cap"], cfg["d"]
    g = torch.Generator().manual_seed(17 + B)
    K = torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16)
    V = torch.randn(B, Hkv, cap, d, generator=g).to(torch.bfloat16)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    kn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, d, generator=g).to(torch.bfloat16)
    pos = np.random.default_rng(3 + B).integers(cap, 10 ** 6, size=B)
    c = sp.DecodeCache(B, Hq, Hkv, cap, d)
    c.K.copy_(K.cuda())
    c.V.copy_(V.cuda())
    pos_d = torch.tensor(pos, device="cuda")
    scale = 1 / math.sqrt(d)
    if fused:
        out, lse = c.append_step(kn.cuda(), vn.cuda(), q.cuda(), pos_d, scale)
        for b in range(B):
            K[b, :, pos[b] % cap] = kn[b]
            V[b, :, pos[b] % cap] = vn[b]
    else:
        out, lse = c.step(q.cuda(), pos_d, scale)
    c.check()
    _compare(out.float().cpu().numpy(), lse.cpu().numpy(), q, K, V, pos, cap, scale, "bf16",
             Hq // Hkv)


def test_bad_arguments():
    import ctypes
    lib = sp.lib()
    n = ctypes.c_size_t()
    assert lib.spattn_decode_workspace_bytes(2, 6, 4, 100, 64, ctypes.byref(n)) == sp.ERR_SHAPE
    assert lib.spattn_decode_workspace_bytes(2, 32, 2, 100, 64, ctypes.byref(n)) == sp.ERR_SHAPE
    assert lib.spattn_decode_workspace_bytes(2, 8, 2, 100, 96, ctypes.byref(n)) == sp.ERR_SHAPE
    assert lib.spattn_decode_workspace_bytes(2, 8, 2, 100, 64, ctypes.byref(n)) == sp.OK
    c = sp.DecodeCache(2, 8, 2, 100, 64)
    q = torch.zeros(2, 8, 64, dtype=torch.bfloat16, device="cuda")
    p = torch.zeros(2, dtype=torch.int64, device="cuda")
    out = torch.empty_like(q)
    st = lib.spattn_decode(2, 8, 2, 100, 101, 64, 0, q.data_ptr(), c.K.data_ptr(), c.V.data_ptr(),
                           p.data_ptr(), 0.1, out.data_ptr(), None, c.workspace.data_ptr(),
                           c.workspace.numel(), None)
    assert st == sp.ERR_INVALID_SPEC
    st = lib.spattn_decode(2, 8, 2, 100, 0, 64, 0, q.data_ptr(), c.K.data_ptr(), c.V.data_ptr(),
                           p.data_ptr(), 0.1, out.data_ptr(), None, c.workspace.data_ptr(),
                           16, None)
    assert st == sp.ERR_SHAPE
    st = lib.spattn_decode(2, 8, 2, 100, 0, 64, 0, q.data_ptr(), c.K.data_ptr(), c.V.data_ptr(),
                           None, 0.1, out.data_ptr(), None, c.workspace.data_ptr(),
                           c.workspace.numel(), None)
    assert st == sp.ERR_NULL
