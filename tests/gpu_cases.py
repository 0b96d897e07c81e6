"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the fp64 oracle on the same (bf16-rounded) values.

Tolerances (from the workload statement, checked element by element):
  * bf16 inputs, fp32 accumulation: max |O - O_ref| <= 1e-2 and
    ||O - O_ref||_2 / ||O_ref||_2 <= 5e-3;
  * fp32 inputs: max |O - O_ref| <= 1e-5;
  * LSE (fp32 in both paths; not named by the statement): the logits, their
    maximum and the fp32 sum of exponentials carry relative error ~1e-6, so
    |LSE - LSE_ref| <= 1e-4 (fp32 inputs: 1e-5) leaves a wide margin.
  * gradients dQ, dK, dV (the statement names no tolerance for them): max-abs as
    above taken relative to the tensor's size, max |g - g_ref| <= tol *
    max(1, max |g_ref|), because a gradient sums many terms and can exceed 1 where an
    output (a convex combination of values) cannot.  bf16 rel-L2 <= 1e-2 (twice the
    output's figure), with the reference norm floored at an rms of 1e-3 (an exactly
    zero gradient, e.g. dQ of a row that reads one key, has no scale).  Where the
    error comes from: the bf16 rounding of the outputs (2^-9 relative, ~1.7e-3 rms
    measured) and the row dot D_i = dO_i . O_i, which the backward takes from the
    forward's stored O, itself rounded to bf16: in rows that read a few keys,
    dp_ij - D_i is small next to D_i's rounding error ~ sqrt(d) 2^-9 |dO| |O|, and
    that term alone (reproduced in fp64 from the stored O) measured up to ~4e-3
    relative in such rows at T = 32K.  fp32 gradients keep the 1e-5 max-abs figure.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import spattn_workloads as W
import sparse_masked_attention_plan_b300 as sp

TOL = {"bf16": dict(max_abs=1e-2, rel_l2=5e-3, lse=1e-4, grad_rel_l2=1e-2),
       "fp32": dict(max_abs=1e-5, rel_l2=None, lse=1e-5, grad_rel_l2=None)}


def torch_dtype(name):
    return torch.bfloat16 if name == "bf16" else torch.float32


def host_view(t):
    """Oracle input view of a CPU tensor: fp32 values, or bf16 bit patterns."""
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits(t)
    return t.contiguous().numpy()


def edge_rows(T, mask, tile=128):
    """Rows where the mask or the tiling changes: ends, window edges, block edges,
    global rows and their neighbours."""
    w = mask.get("window", 0)
    r = mask.get("radius", -1)
    rows = {0, 1, 2, T - 1, T - 2, T // 2}
    for x in (w - 1, w, w + 1, r, r + 1, 2 * r):
        rows.add(x)
    for b in range(0, T, tile * 16):
        rows.update({b - 1, b, b + 1})
    for k in (1, 2, 3, 255, 256, 257):
        rows.add(tile * k - 1)
        rows.add(tile * k)
    for g in np.asarray(mask.get("global_pos", ()))[:64]:
        rows.update({int(g) - 1, int(g), int(g) + 1})
    s = mask.get("stride", 0)
    if s:
        rows.update({s - 1, s, s + 1, 3 * s})
    return sorted(x for x in rows if 0 <= x < T)


def run_and_compare(B, H, T, d, mask, dtype="bf16", seed=0, heads=None, rows=None,
                    scale=None, plan=None):
    """Run spattn_fwd on seeded [B,H,T,d] inputs; compare the chosen heads/rows with
    the oracle.  Returns a dict of the observed errors; asserts the tolerances."""
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    Q, K, V = W.qkv(B, H, T, d, seed, torch_dtype(dtype))
    if plan is None:
        plan = sp.Plan(T, d, **mask)
    q, k, v = (x.cuda() for x in (Q, K, V))
    o, lse = sp.fwd(plan, q, k, v, scale)
    torch.cuda.synchronize()
    plan.check_device()
    O = o.float().cpu().numpy()
    L = lse.cpu().numpy()
    m = oracle_mask(T, mask)
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    tol = TOL[dtype]
    worst = dict(max_abs=0.0, rel_l2=0.0, lse=0.0)
    for (b, h) in heads:
        rr = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
        Oref, Lref = oracle.attention(m, host_view(Q[b, h]), host_view(K[b, h]),
                                      host_view(V[b, h]), scale, rr)
        got = O[b, h][rr].astype(np.float64)
        assert np.all(np.isfinite(got)), f"non-finite output in head {(b, h)}"
        err = np.abs(got - Oref)
        max_abs = float(err.max()) if err.size else 0.0
        rel = float(np.linalg.norm(got - Oref) / max(np.linalg.norm(Oref), 1e-30))
        lerr = float(np.abs(L[b, h][rr].astype(np.float64) - Lref).max()) if rr.size else 0.0
        worst["max_abs"] = max(worst["max_abs"], max_abs)
        worst["rel_l2"] = max(worst["rel_l2"], rel)
        worst["lse"] = max(worst["lse"], lerr)
        where = int(np.unravel_index(np.argmax(err), err.shape)[0]) if err.size else -1
        assert max_abs <= tol["max_abs"], (
            f"head {(b, h)}: max-abs {max_abs:.3g} at row {rr[where] if where >= 0 else -1}")
        if tol["rel_l2"] is not None:
            assert rel <= tol["rel_l2"], f"head {(b, h)}: rel-L2 {rel:.3g}"
        assert lerr <= tol["lse"], f"head {(b, h)}: LSE error {lerr:.3g}"
    return worst


def check_grad(name, got, ref, dtype, where=""):
    """Compare one gradient tensor (any shape, host arrays) with its fp64 reference."""
    tol = TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}{where}: non-finite values"
    err = np.abs(got - ref)
    if not err.size:
        return 0.0
    bound = tol["max_abs"] * max(1.0, float(np.abs(ref).max()))
    k = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= bound, (f"{name}{where}: max-abs {err.max():.3g} > {bound:.3g} at {k} "
                                f"(got {got[k]:.6g}, want {ref[k]:.6g})")
    if tol["grad_rel_l2"] is not None:
        # relative to the reference's norm, floored at an rms of 1e-3: a reference that
        # is (almost) zero, e.g. dQ when a row reads one key, has no relative scale
        den = max(np.linalg.norm(ref), 1e-3 * math.sqrt(ref.size))
        rel = float(np.linalg.norm(got - ref) / den)
        assert rel <= tol["grad_rel_l2"], f"{name}{where}: rel-L2 {rel:.3g}"
    return float(err.max())


def oracle_mask(T, mask):
    rp = np.asarray(mask.get("rand_pairs", ()), dtype=np.int32).reshape(-1, 2)
    rp = rp[np.lexsort((rp[:, 1], rp[:, 0]))] if len(rp) else rp
    return oracle.Mask(T, mask.get("causal", 1), mask.get("window", 0), mask.get("radius", -1),
                       mask.get("stride", 0), mask.get("offset", 0),
                       np.sort(np.asarray(mask.get("global_pos", ()), dtype=np.int32)),
                       mask.get("dilation", 1), mask.get("rand_block", 0), rp)


def run_bwd(B, H, T, d, mask, dtype="bf16", seed=0, scale=None, plan=None):
    """Forward then backward on the GPU for seeded Q, K, V, dO.  Returns the CPU
    inputs, the plan, and the GPU results (O, LSE, dQ, dK, dV) on the host."""
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    Q, K, V = W.qkv(B, H, T, d, seed, torch_dtype(dtype))
    dO = W.grad_out(B, H, T, d, seed, torch_dtype(dtype))
    if plan is None:
        plan = sp.Plan(T, d, **mask)
    q, k, v, do = (x.cuda() for x in (Q, K, V, dO))
    o, lse = sp.fwd(plan, q, k, v, scale)
    dq, dk, dv = sp.bwd(plan, q, k, v, o, lse, do, scale)
    torch.cuda.synchronize()
    plan.check_device()
    res = tuple(x.float().cpu().numpy() for x in (o, lse, dq, dk, dv))
    return (Q, K, V, dO), plan, res, scale


def bwd_and_compare(B, H, T, d, mask, dtype="bf16", seed=0, scale=None, heads=None):
    """Every element of dQ, dK, dV of the chosen heads against the fp64 oracle."""
    (Q, K, V, dO), _, (_, _, dq, dk, dv), scale = run_bwd(B, H, T, d, mask, dtype, seed, scale)
    m = oracle_mask(T, mask)
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for (b, h) in heads:
        ref = oracle.attention_bwd(m, host_view(Q[b, h]), host_view(K[b, h]), host_view(V[b, h]),
                                   host_view(dO[b, h]), scale)
        for name, got, r in zip(("dQ", "dK", "dV"), (dq[b, h], dk[b, h], dv[b, h]), ref):
            check_grad(name, got, r, dtype, where=f" head {(b, h)}")


def workload(name):
    cfg = W.WORKLOADS[name]
    return cfg, W.mask_params(name)
