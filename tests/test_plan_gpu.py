"""Plan builder on the GPU against the oracle: pair counts, the non-empty tile list
(block, count, class) and the compacted column list must match bit for bit; the
execution schedule must compute only non-empty tiles and cover every allowed pair
exactly once."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import spattn_workloads as W
import sparse_masked_attention_plan_b300 as sp
import gpu_cases
from pins import random_blocks, small_specs

pytestmark = pytest.mark.gpu

EDGE_SPECS = [
    dict(T=1, causal=1, window=0),
    dict(T=1, causal=0, radius=0),
    dict(T=300, causal=1, window=1),
    dict(T=300, causal=1, window=300),
    dict(T=300, causal=1, window=10_000),
    dict(T=257, causal=0, radius=0),
    dict(T=257, causal=0, radius=1000),
    dict(T=500, causal=1, window=37, stride=1, offset=0),
    dict(T=777, causal=1, window=130, stride=17, offset=5, global_pos=[0, 3, 129, 500, 776]),
    dict(T=777, causal=0, radius=60, stride=128, offset=127, global_pos=[5, 6, 7, 640]),
    dict(T=1000, causal=0, radius=-1, global_pos=[999]),
    dict(T=1024, causal=1, window=0, stride=64, offset=0),
    dict(T=600, causal=1, window=200, stride=1000, offset=3),
    dict(T=600, causal=1, window=200, stride=1000, offset=700),
    dict(T=700, causal=1, window=37, dilation=3),
    dict(T=900, causal=1, window=100, dilation=2, stride=64, offset=1, global_pos=[0, 7, 450]),
    dict(T=640, causal=0, radius=20, dilation=5, stride=16, offset=3, global_pos=[2, 300]),
    dict(T=500, causal=1, window=0, dilation=7),
    dict(T=300, causal=1, window=40, dilation=301),
    dict(T=1000, causal=0, radius=3, dilation=200),
    # BigBird random blocks, with and without the other rules
    dict(T=700, causal=0, radius=40, global_pos=[0, 1, 650], rand_block=64,
         rand_pairs=[(0, 9), (1, 5), (3, 0), (3, 10), (10, 2), (10, 10)]),
    dict(T=520, causal=1, window=70, stride=33, offset=4, rand_block=16,
         rand_pairs=[(20, 3), (20, 19), (31, 0), (32, 32), (5, 30)]),
    dict(T=600, causal=0, radius=0, rand_block=128, rand_pairs=[(0, 4), (4, 0), (2, 2)]),
    dict(T=900, causal=1, window=0, rand_block=32, rand_pairs=[(27, 28), (28, 0)]),
]


def oracle_mask(T, p):
    return gpu_cases.oracle_mask(T, p)


def expected_columns(T, p):
    """Strided U global columns, straight from the definition (numpy)."""
    j = np.arange(T)
    s = p.get("stride", 0)
    sel = (j % s == p.get("offset", 0)) if s else np.zeros(T, bool)
    g = np.asarray(p.get("global_pos", ()), dtype=np.int64)
    sel[g] = True
    return np.nonzero(sel)[0].astype(np.int32)


def check_plan(T, p, d=64):
    m = oracle_mask(T, p)
    plan = sp.Plan(T, d, **{k: p[k] for k in p if k != "T"})
    info = plan.info()
    assert info["pairs_per_head"] == m.count_pairs()
    qb, kb, cnt, cls, (nf, npart, ne) = oracle.tile_list(m, 128, 128)
    gq, gk, gc, gcl = plan.tiles()
    assert np.array_equal(gq, qb) and np.array_equal(gk, kb)
    assert np.array_equal(gc, cnt)
    assert np.array_equal(gcl, cls)
    assert (info["n_full"], info["n_partial"], info["n_empty"]) == (nf, npart, ne)
    assert np.array_equal(plan.columns(), expected_columns(T, p))
    return plan, m


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_workload_plan_matches_oracle(oracle_mod, name):
    cfg = W.WORKLOADS[name]
    p = W.mask_params(name)
    plan, m = check_plan(cfg["T"], p, cfg["d"])
    # the page-derived pair count of the 32K / W=4096 workload
    if name == "t32k_w4096":
        assert plan.info()["pairs_per_head"] == 125_831_168


@pytest.mark.parametrize("k", range(len(EDGE_SPECS)))
def test_edge_spec_plan_matches_oracle(oracle_mod, k):
    e = dict(EDGE_SPECS[k])
    T = e.pop("T")
    check_plan(T, e)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_spec_plans_match_oracle(oracle_mod, seed):
    for e in small_specs(seed, n=40):
        e = dict(e)
        T = e.pop("T")
        check_plan(T, e)
    rng = np.random.default_rng(100 + seed)
    for _ in range(12):  # longer sequences, several tiles, ragged tails
        T = int(rng.integers(129, 1500))
        causal = int(rng.integers(0, 2))
        s = int(rng.choice([0, 1, 3, 17, 64, 200]))
        e = dict(causal=causal, window=int(rng.choice([0, 1, 50, 129, 700])) if causal else 0,
                 radius=-1 if causal else int(rng.choice([-1, 0, 20, 128, 400])),
                 stride=s, offset=int(rng.integers(0, s)) if s else 0,
                 global_pos=np.sort(rng.choice(T, int(rng.choice([0, 1, 9])), replace=False)),
                 dilation=int(rng.choice([1, 1, 2, 3, 130])))
        if rng.random() < 0.4:
            e["rand_block"], e["rand_pairs"] = random_blocks(T, int(rng.choice([16, 64, 128])),
                                                             int(rng.integers(1, 4)), rng)
        check_plan(T, e)


def covered_keys(plan_sched, cols, T, group_rows, qtile_rows, i, grow, p):
    """Keys the schedule lets row i read: band tiles via the predicate rule of the
    kernels' definition (local window U strided/global bits), packed chunks via C."""
    items, ents, _ = plan_sched
    keys = []
    colset = set(cols.tolist())
    causal = p.get("causal", 1)
    for it in items:
        q0, off, cnt, fl = it
        if fl & 1:  # gathered global rows
            rows = p["global_pos_sorted"][q0:q0 + group_rows]
            if i not in rows:
                continue
            # split items: both query tiles hold these rows, key tiles alternate
            tiles = (0, 1) if fl & 2 else (int(np.nonzero(rows == i)[0][0]) // qtile_rows,)
        else:
            if grow or not (q0 <= i < q0 + group_rows):
                continue
            tiles = ((i - q0) // qtile_rows,)
        for (src, f, kb, lim) in ents[off:off + cnt]:
            for t in tiles:
                if f & (1 << t):
                    keys += entry_keys(src, f, lim, t, i, T, cols, colset, causal, p)
    return keys


def in_random(p, i, j):
    b = p.get("rand_block", 0)
    if not b:
        return False
    return (i // b, j // b) in {tuple(x) for x in np.asarray(p["rand_pairs"]).reshape(-1, 2).tolist()}


def entry_keys(src, f, lim, t, i, T, cols, colset, causal, p):
    kind = (f >> 4) & 3
    full = bool(f & (4 << t))  # the kernels skip the predicate: the whole tile counts
    if kind == 1:
        return [int(c) for c in (cols[src:src + 128] if full else cols[src:lim])]
    out = []
    for j in range(src, src + 128):
        if full:
            ok = True
        elif j >= T:
            ok = False
        elif kind == 2:
            ok = (j <= i) if causal else True
        elif kind == 3:  # random-only tile: random keys that are not sparse columns
            ok = in_random(p, i, j) and j not in colset and (j <= i or not causal)
        elif causal:
            w, dl = p.get("window", 0), p.get("dilation", 1)
            ok = j <= i and (((w == 0 or i - j < w * dl) and (i - j) % dl == 0) or
                             j in colset or in_random(p, i, j))
        else:
            r, dl = p.get("radius", -1), p.get("dilation", 1)
            ok = (((r < 0 or abs(i - j) <= r * dl) and abs(i - j) % dl == 0) or j in colset or
                  in_random(p, i, j))
        if ok:
            out.append(j)
    return out


@pytest.mark.parametrize("k", range(len(EDGE_SPECS)))
def test_schedule_covers_each_allowed_pair_once(oracle_mod, k):
    e = dict(EDGE_SPECS[k])
    T = e.pop("T")
    plan, m = check_plan(T, e)
    qb, kb, cnt, cls, _ = oracle.tile_list(m, 128, 128)
    nonempty = set(zip(qb.tolist(), kb.tolist()))
    cols = plan.columns()
    gpos = np.sort(np.asarray(e.get("global_pos", ()), dtype=np.int64))
    e["global_pos_sorted"] = gpos
    for which, (group_rows, qtile_rows) in enumerate([(256, 128), (64, 64)]):
        sched = plan.schedule(which)
        items, ents, products = sched
        # every computed band tile is a non-empty tile of the natural grid
        n_products = 0
        for (q0, off, cnt_, fl) in items:
            for (src, f, kbi, lim) in ents[off:off + cnt_]:
                for t in range(2):
                    if not (f & (1 << t)):
                        continue
                    n_products += 1
                    if ((f >> 4) & 3) == 0 and not (fl & 1):
                        qbi = (q0 + t * qtile_rows) // 128
                        assert (qbi, kbi) in nonempty, (which, q0, t, kbi)
        assert n_products == products
        for i in range(T):
            grow = i in set(gpos.tolist())
            got = sorted(covered_keys(sched, cols, T, group_rows, qtile_rows, i, grow, e))
            assert got == m.row_set(i).tolist(), (which, i)


GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_counts.json")))


def _spec(e):
    return {k: e[k] for k in ("causal", "window", "radius", "stride", "offset", "global_pos")}


@pytest.mark.parametrize("k", range(len(GOLDEN["pair_counts"])))
def test_page_printed_counts_through_gpu_plan(oracle_mod, k):
    """The pages' own small masks (six tokens with w = 2 and full causal; sixteen
    tokens full, causal, w = 4, w = 2 + stride 4, radius 2 + global token 0) built by
    spattn_plan_create: the pair count equals the printed integer, and the tile list
    equals the oracle's."""
    e = GOLDEN["pair_counts"][k]
    plan, _ = check_plan(e["T"], _spec(e))
    assert plan.info()["pairs_per_head"] == e["pairs"], e["source"]


@pytest.mark.parametrize("k", range(len(GOLDEN["row_sets"])))
def test_page_printed_row_sets_through_gpu_schedule(oracle_mod, k):
    """The keys the GPU plan's forward schedule lets the printed query read are the
    printed set (query 12 of the sixteen-token examples, query 0 when global, the
    sixth of six tokens, token 8000 of an 8192-token window of 512)."""
    e = GOLDEN["row_sets"][k]
    T, i = e["T"], e["row"]
    spec = _spec(e)
    plan, _ = check_plan(T, spec)
    want = e["set"] if "set" in e else list(range(e["range"][0], e["range"][1] + 1))
    spec["global_pos_sorted"] = np.sort(np.asarray(spec["global_pos"], dtype=np.int64))
    grow = i in set(spec["global_pos"])
    for which, (group_rows, qtile_rows) in enumerate([(256, 128), (64, 64)]):
        got = sorted(covered_keys(plan.schedule(which), plan.columns(), T, group_rows,
                                  qtile_rows, i, grow, spec))
        assert got == want, (which, e["source"])


def test_walk_counter_counts_scheduled_products(oracle_mod):
    T, d = 1000, 64
    p = dict(causal=1, window=130, stride=17, offset=5, global_pos=[3, 500])
    plan = sp.Plan(T, d, **p)
    plan.set_walk_counter(True)
    B, H = 2, 3
    q = torch.randn(B, H, T, d, device="cuda", dtype=torch.bfloat16)
    sp.fwd(plan, q, q, q, 0.125)
    _, _, products = plan.schedule(0)
    assert plan.walk_count() == products * B * H
    plan.set_walk_counter(True)
    sp.fwd(plan, q.float(), q.float(), q.float(), 0.125)
    _, _, products32 = plan.schedule(1)
    assert plan.walk_count() == products32 * B * H
