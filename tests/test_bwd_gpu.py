"""Backward parity: dQ, dK, dV from spattn_bwd (through the C ABI, after spattn_fwd on
the GPU) against the fp64 oracle's gradients on the same seeded inputs.

Small and mid-size cases compare every element of every (or of chosen) heads.  At
the benchmark's full sizes the oracle computes dQ of sampled rows and dK, dV of
sampled keys exactly (a row's dQ needs only its own allowed set; a key's dK, dV need
the rows that read it), element by element; identities that hold at any size (sums
over keys of a softmax over each row's set) are checked on every head besides:
  sum_j dV_j = sum_i dO_i,  sum_j dK_j = 0,
  sum_i q_i . dQ_i = sum_j k_j . dK_j,  sum_j v_j . dV_j = sum_i dO_i . O_i.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import spattn_workloads as W
import sparse_masked_attention_plan_b300 as sp
from gpu_cases import (TOL, bwd_and_compare, check_grad, edge_rows, host_view, oracle_mask,
                       run_bwd, workload)
from pins import np_dense_mask
from test_fwd_gpu import SWEEP

pytestmark = pytest.mark.gpu

SMALL = ["t512_w128_s0", "t512_w128_s64", "t512_full_causal"]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("name", SMALL)
def test_small_workloads_every_element(oracle_mod, name, dtype):
    cfg, p = workload(name)
    bwd_and_compare(cfg["B"], cfg["H"], cfg["T"], cfg["d"], p, dtype, seed=3)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("k", range(len(SWEEP)))
def test_sweep_every_element(oracle_mod, k, dtype):
    B, H, T, d, mask = SWEEP[k]
    bwd_and_compare(B, H, T, d, mask, dtype, seed=100 + k)


EDGES = [
    (1, 1, 1, 64, dict(causal=1, window=0)),
    (1, 2, 65, 128, dict(causal=1, window=3)),
    (1, 1, 200, 64, dict(causal=0, radius=2, global_pos=list(range(0, 200, 2)))),  # half global
    (1, 1, 130, 64, dict(causal=1, window=10, global_pos=list(range(130)))),       # all global
    (1, 1, 257, 128, dict(causal=0, radius=0, stride=1, offset=0)),  # every column strided
    (2, 2, 190, 64, dict(causal=1, window=1, stride=7, offset=6, global_pos=[0, 64, 189])),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("k", range(len(EDGES)))
def test_edge_cases_every_element(oracle_mod, k, dtype):
    B, H, T, d, mask = EDGES[k]
    bwd_and_compare(B, H, T, d, mask, dtype, seed=200 + k)


@pytest.mark.parametrize("scale", [0.05, 0.3])
def test_scales(oracle_mod, scale):
    bwd_and_compare(1, 2, 700, 64, dict(causal=1, window=90, stride=32, offset=1,
                                         global_pos=[5, 300]), "bf16", seed=9, scale=scale)


@pytest.mark.parametrize("name", ["t2048_w256_s0", "t2048_w256_s64"])
def test_t2048_workloads_two_heads(oracle_mod, name):
    cfg, p = workload(name)
    bwd_and_compare(cfg["B"], cfg["H"], cfg["T"], cfg["d"], p, "bf16", seed=1,
                    heads=[(0, 0), (cfg["B"] - 1, cfg["H"] - 1)])


def _identities(Q, K, V, dO, res, dtype):
    """The four any-size identities on every head, in fp64 from the GPU outputs."""
    o, _, dq, dk, dv = res
    q, k, v, g = (x.double().numpy() for x in (Q, K, V, dO))
    tol = 1e-2 if dtype == "bf16" else 1e-5
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            dvh, dkh, dqh = (x[b, h].astype(np.float64) for x in (dv, dk, dq))
            lhs, rhs = dvh.sum(0), g[b, h].sum(0)
            assert np.abs(lhs - rhs).max() <= tol * (np.linalg.norm(dvh) + 1), \
                f"sum dV != sum dO in head {(b, h)}: {np.abs(lhs - rhs).max():.3g}"
            assert np.abs(dkh.sum(0)).max() <= tol * (np.linalg.norm(dkh) + 1e-3), \
                f"sum dK != 0 in head {(b, h)}: {np.abs(dkh.sum(0)).max():.3g}"
            a1 = float((q[b, h] * dqh).sum())
            a2 = float((k[b, h] * dkh).sum())
            ref = np.linalg.norm(q[b, h] * dqh) + np.linalg.norm(k[b, h] * dkh) + 1e-3
            assert abs(a1 - a2) <= tol * ref, f"q.dQ != k.dK in head {(b, h)}: {a1} {a2}"
            c1 = float((v[b, h] * dvh).sum())
            c2 = float((g[b, h] * o[b, h].astype(np.float64)).sum())
            ref = np.linalg.norm(v[b, h] * dvh) + np.linalg.norm(g[b, h] * o[b, h]) + 1e-3
            assert abs(c1 - c2) <= tol * ref, f"v.dV != dO.O in head {(b, h)}: {c1} {c2}"


def sample_keys(T, p, n, seed):
    """Keys whose dK/dV the full-size tests check: the sequence ends, tile and window
    edges, the first strided and global columns (packed columns of the kernels) and
    the keys of a random block, plus n seeded ones."""
    keys = set(edge_rows(T, p)[:40])
    s = p.get("stride", 0)
    if s:
        keys.update(range(p.get("offset", 0), min(T, 4 * s), s))
    g = np.asarray(p.get("global_pos", ()), dtype=np.int64)
    keys.update(int(x) for x in g[:4])
    keys.update(int(x) for x in g[-2:])
    rp = np.asarray(p.get("rand_pairs", ()), dtype=np.int64).reshape(-1, 2)
    if len(rp):
        b = p["rand_block"]
        k0 = int(rp[len(rp) // 2, 1]) * b
        keys.update({k0, k0 + 1, min(T - 1, k0 + b - 1)})
    return W.sample_rows(T, n, seed=seed, must=sorted(x for x in keys if 0 <= x < T))


@pytest.mark.parametrize("name", ["t32k_w4096", "t16k_r256_s16_g128", "t32k_w512_d2",
                                  "t4096_bigbird"])
def test_full_size_sampled_rows_keys_and_identities(oracle_mod, name):
    """At the benchmark's sizes and launch configuration: dQ of sampled rows and dK, dV
    of sampled keys element by element against the oracle, and the identities on
    every head."""
    cfg, p = workload(name)
    B, H, T, d = cfg["B"], cfg["H"], cfg["T"], cfg["d"]
    (Q, K, V, dO), _, res, scale = run_bwd(B, H, T, d, p, "bf16", seed=0)
    _identities(Q, K, V, dO, res, "bf16")
    dq, dk, dv = res[2], res[3], res[4]
    m = oracle_mask(T, p)
    rows = W.sample_rows(T, 24, seed=5, must=edge_rows(T, p)[:40])
    keys = sample_keys(T, p, 16, seed=6)
    for (b, h) in [(0, 0), (B - 1, H - 1)]:
        args = [host_view(x[b, h]) for x in (Q, K, V, dO)]
        ref = oracle.attention_bwd_dq(m, *args, scale, rows)
        check_grad("dQ", dq[b, h][rows], ref, "bf16", where=f" head {(b, h)}")
        rk, rv = oracle.attention_bwd_dkdv(m, *args, scale, keys)
        check_grad("dK", dk[b, h][keys], rk, "bf16", where=f" head {(b, h)}")
        check_grad("dV", dv[b, h][keys], rv, "bf16", where=f" head {(b, h)}")


def test_identities_fp32_mid_size(oracle_mod):
    mask = dict(causal=0, radius=100, stride=50, offset=7, global_pos=[3, 999, 2000])
    (Q, K, V, dO), _, res, _ = run_bwd(1, 3, 4096, 64, mask, "fp32", seed=4)
    _identities(Q, K, V, dO, res, "fp32")


def test_backward_is_deterministic(oracle_mod):
    mask = dict(causal=1, window=300, stride=64, offset=1, global_pos=[10, 700, 1500])
    (Q, K, V, dO), plan, res1, scale = run_bwd(2, 2, 2000, 128, mask, "bf16", seed=6)
    _, _, res2, _ = run_bwd(2, 2, 2000, 128, mask, "bf16", seed=6, plan=plan)
    for a, b in zip(res1[2:], res2[2:]):
        assert np.array_equal(a, b)


def _key_major_cover(plan, T, mask, which=3, rows_per=64, keys_per=64):
    """How often the key-major schedule visits each (query, key) pair: a band entry
    visits the allowed pairs of its non-global rows inside its unit, a random entry
    their random-block pairs that are not sparse columns, a packed entry its packed
    columns [a, b), a gathered dense entry the allowed pairs of its global rows inside
    its unit.  A band entry marked fully allowed (flag bit 1) must have every pair of
    its rows and keys allowed."""
    items, ents, _ = plan.schedule(which)
    cols = plan.columns()
    g = np.asarray(sorted(mask.get("global_pos", [])), dtype=np.int64)
    M = np_dense_mask(T, mask.get("causal", 1), mask.get("window", 0), mask.get("radius", -1),
                      mask.get("stride", 0), mask.get("offset", 0), list(g),
                      mask.get("dilation", 1), mask.get("rand_block", 0),
                      mask.get("rand_pairs", ()))
    Rm = np.zeros((T, T), bool)  # the random blocks alone
    rb = mask.get("rand_block", 0)
    for q, k in np.asarray(mask.get("rand_pairs", ()), dtype=np.int64).reshape(-1, 2):
        Rm[q * rb:(q + 1) * rb, k * rb:(k + 1) * rb] = True
    if mask.get("causal", 1):
        Rm &= np.tri(T, dtype=bool)
    colset = np.zeros(T, bool)
    colset[cols] = True
    isg = np.zeros(T, bool)
    isg[g] = True
    cov = np.zeros((T, T), np.int32)
    for key0, off, cnt, flags in items:
        packed_unit = flags & 1
        for q0, ef, a, b in ents[off:off + cnt]:
            kind = (ef >> 4) & 3
            if ef & 2:  # marked fully allowed: every pair of its rows and keys is allowed
                assert kind == 0 and not packed_unit and not ef & 1
                blk = M[q0:min(q0 + rows_per, T), key0:min(key0 + keys_per, T)]
                assert blk.all(), f"entry ({q0}, unit {key0}) marked full has disallowed pairs"
            if ef & 1:
                rows = g[q0:q0 + rows_per]
            else:
                rows = np.arange(q0, min(q0 + rows_per, T))
                rows = rows[~isg[rows]]
            if packed_unit:
                assert kind == 1
                keys = cols[a:b]
                cov[np.ix_(rows, keys)] += 1
            else:
                keys = np.arange(key0, min(key0 + keys_per, T))
                if kind == 3:  # random-only unit: random keys that are not sparse columns
                    sub = (Rm[np.ix_(rows, keys)] & ~colset[keys][None, :]).astype(np.int32)
                else:
                    sub = M[np.ix_(rows, keys)].astype(np.int32)
                cov[np.ix_(rows, keys)] += sub
    return cov, M


@pytest.mark.parametrize("granule", [(3, 64, 64), (4, 128, 128)], ids=["fp32", "tc"])
@pytest.mark.parametrize("k", range(len(SWEEP)))
def test_key_major_schedule_covers_every_pair_once(k, granule):
    _, _, T, d, mask = SWEEP[k]
    plan = sp.Plan(T, d, **mask)
    cov, M = _key_major_cover(plan, T, mask, *granule)
    bad = np.argwhere(cov != M.astype(np.int32))
    assert bad.size == 0, f"pairs visited {cov[tuple(bad[0])]} times, allowed {M[tuple(bad[0])]}: {bad[:5]}"


def test_bad_arguments():
    plan = sp.Plan(256, 64, causal=1, window=16)
    q = torch.zeros(1, 1, 256, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 256, device="cuda")
    lib = sp.lib()
    args = [q.data_ptr()] * 4
    st = lib.spattn_bwd(plan.handle, 1, 1, 0, *args, None, q.data_ptr(), 0.1, *[q.data_ptr()] * 3,
                        None)
    assert st == sp.ERR_NULL
    st = lib.spattn_bwd(plan.handle, 1, 1, 0, *args, lse.data_ptr(), q.data_ptr() + 2, 0.1,
                        *[q.data_ptr()] * 3, None)
    assert st == sp.ERR_ALIGN
    st = lib.spattn_bwd(plan.handle, 1, 1, 0, *args, lse.data_ptr(), q.data_ptr(), -1.0,
                        *[q.data_ptr()] * 3, None)
    assert st == sp.ERR_INVALID_SPEC
    st = lib.spattn_bwd(plan.handle, 0, 1, 0, *args, lse.data_ptr(), q.data_ptr(), 0.1,
                        *[q.data_ptr()] * 3, None)
    assert st == sp.ERR_SHAPE
