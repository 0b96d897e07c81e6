"""Checks that pin the CPU oracle to something other than itself.

Each ``check_*`` function returns a list of failure strings (empty = pass), so the
same checks serve the oracle tests and the mutation tests (which must see at least
one failure for every planted mistake).  What each check leans on:

  * numbers printed on the pages (tests/golden/page_counts.json, each with its source);
  * closed forms: the glossary's edge count E = n w - w(w-1)/2, n(n+1)/2 for the
    causal triangle, the L-layer reach L(w-1)+1, window = 0 / window >= n equal causal;
  * an independent dense-boolean restatement of the mask rules written here in numpy
    (np.indices grids, the style the pages use) and an independent inclusion-exclusion
    pair counter;
  * library routines: torch's scaled_dot_product_attention and logsumexp in fp64;
  * exact special cases: w = 1 gives y_i = v_i, Q = 0 gives the mean of the allowed
    values, and a constant shift of every key leaves y unchanged.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "page_counts.json")))


def mask_of(e) -> oracle.Mask:
    return oracle.Mask(e["T"], e.get("causal", 1), e.get("window", 0),
                       e.get("radius", -1), e.get("stride", 0), e.get("offset", 0),
                       e.get("global_pos", []), e.get("dilation", 1), e.get("rand_block", 0),
                       e.get("rand_pairs", ()))


def dense_of(e) -> np.ndarray:
    return np_dense_mask(e["T"], e.get("causal", 1), e.get("window", 0), e.get("radius", -1),
                         e.get("stride", 0), e.get("offset", 0), e.get("global_pos", []),
                         e.get("dilation", 1), e.get("rand_block", 0), e.get("rand_pairs", ()))


# ---------------------------------------------------------------- independent rules

def np_dense_mask(T, causal, window, radius, stride, offset, gpos, dilation=1, rand_block=0,
                  rand_pairs=()) -> np.ndarray:
    """Dense boolean mask, True = may attend, from index grids (independent of oracle.c).
    The dilated local rule is the "Attention variants" exercise's dilated(n, w, d):
    gap >= 0, gap % d == 0, gap < w d (bidirectional: |gap| <= r d, |gap| % d == 0).
    Random blocks (BigBird): the b x b blocks (query block, key block) listed."""
    i, j = np.indices((T, T))
    past = j <= i
    gap = i - j
    on_grid = (np.abs(gap) % dilation) == 0
    if causal:
        local = past & on_grid & ((gap < window * dilation) if window > 0 else True)
    else:
        local = on_grid & ((np.abs(gap) <= radius * dilation) if radius >= 0 else True)
    m = local.copy()
    if stride > 0:
        col = (j % stride == offset)
        m |= (col & past) if causal else col
    g = np.zeros(T, dtype=bool)
    g[np.asarray(gpos, dtype=np.int64)] = True
    gcol = np.broadcast_to(g[None, :], (T, T))
    grow = np.broadcast_to(g[:, None], (T, T))
    m |= (gcol & past) if causal else gcol
    m |= (grow & past) if causal else grow
    if rand_block and len(rand_pairs):
        nb = -(-T // rand_block)
        blk = np.zeros((nb, nb), dtype=bool)
        rp = np.asarray(rand_pairs, dtype=np.int64).reshape(-1, 2)
        blk[rp[:, 0], rp[:, 1]] = True
        r = blk[i // rand_block, j // rand_block]
        m |= (r & past) if causal else r
    return m


def closed_form_pairs(T, causal, window, radius, stride, offset, gpos, dilation=1) -> int:
    """Pair count by inclusion-exclusion per row: |L| + |S minus L| + |G minus (L u S)|.
    With a dilation d > 1 the row terms are counted by brute force over each row's
    local span (still independent of oracle.c)."""
    if dilation > 1:
        if stride == 0 and len(gpos) == 0:  # local keys only: i - k d for k in the window
            i = np.arange(T, dtype=np.int64)
            if causal:
                back = i // dilation
                return int((np.minimum(back, window - 1) + 1 if window else back + 1).sum())
            back, fwd = i // dilation, (T - 1 - i) // dilation
            if radius >= 0:
                back, fwd = np.minimum(back, radius), np.minimum(fwd, radius)
            return int((back + fwd + 1).sum())
        D = np_dense_mask(T, causal, window, radius, stride, offset, gpos, dilation)
        return int(D.sum())
    i = np.arange(T, dtype=np.int64)
    jmax = i if causal else np.full(T, T - 1, dtype=np.int64)
    if causal:
        lo = np.zeros(T, np.int64) if window == 0 else np.maximum(0, i - window + 1)
        hi = i.copy()
    else:
        lo = np.zeros(T, np.int64) if radius < 0 else np.maximum(0, i - radius)
        hi = np.full(T, T - 1, np.int64) if radius < 0 else np.minimum(T - 1, i + radius)
    n_local = hi - lo + 1

    def ap_upto(x):  # #{0 <= j <= x : j % stride == offset}
        if stride == 0:
            return np.zeros_like(x)
        return np.where(x >= offset, (x - offset) // stride + 1, 0)

    n_strided_out = ap_upto(jmax) - (ap_upto(hi) - ap_upto(lo - 1))
    G = np.asarray(gpos, dtype=np.int64)
    if len(G):
        gg = G[None, :]
        inrange = gg <= jmax[:, None]
        inlocal = (gg >= lo[:, None]) & (gg <= hi[:, None])
        strided = (gg % stride == offset) if stride > 0 else np.zeros_like(gg, bool)
        n_g = (inrange & ~inlocal & ~strided).sum(axis=1)
    else:
        n_g = 0
    per_row = n_local + n_strided_out + n_g
    isg = np.zeros(T, bool)
    isg[G] = True
    per_row = np.where(isg, jmax + 1, per_row)
    return int(per_row.sum())


def reach_after(M: np.ndarray, layers: int) -> np.ndarray:
    """Boolean matrix power: which originals can influence each position."""
    R = np.eye(len(M), dtype=bool)
    Mi = M.astype(np.int64)
    for _ in range(layers):
        R = (Mi @ R.astype(np.int64)) > 0
    return R


def oracle_dense(m: oracle.Mask) -> np.ndarray:
    D = np.zeros((m.T, m.T), dtype=bool)
    for i in range(m.T):
        D[i, m.row_set(i)] = True
    return D


def small_specs(seed=0, n=60):
    """Seeded sweep of small masks covering every rule and edge (ragged T, w=1,
    w >= T, r = 0, stride 1..17, offsets, globals overlapping the window/stride)."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        T = int(rng.integers(1, 90))
        causal = int(rng.integers(0, 2))
        window = int(rng.choice([0, 1, 2, 3, 5, 8, T, T + 3])) if causal else 0
        radius = -1 if causal else int(rng.choice([-1, 0, 1, 2, 7, T]))
        stride = int(rng.choice([0, 0, 1, 2, 3, 4, 17]))
        offset = int(rng.integers(0, stride)) if stride else 0
        g = int(rng.choice([0, 0, 1, 3, 5]))
        gpos = np.sort(rng.choice(T, size=min(g, T), replace=False)).tolist()
        dilation = int(rng.choice([1, 1, 1, 2, 3, 5]))
        out.append(dict(T=T, causal=causal, window=window, radius=radius, stride=stride,
                        offset=offset, global_pos=gpos, dilation=dilation))
    # random blocks on a third of the specs, from a stream of their own (the draws
    # above stay what they were)
    rr = np.random.default_rng(seed + 1000)
    for e in out:
        if rr.random() < 1 / 3:
            e["rand_block"], e["rand_pairs"] = random_blocks(e["T"], int(rr.choice([16, 32])),
                                                             int(rr.integers(1, 4)), rr)
    return out


def random_blocks(T, b, R, rng):
    """BigBird-style random blocks: for every query block, R distinct key blocks drawn
    uniformly from all blocks (fewer when there are fewer blocks); sorted pairs."""
    nb = -(-T // b)
    pairs = []
    for q in range(nb):
        for k in sorted(rng.choice(nb, size=min(R, nb), replace=False).tolist()):
            pairs.append((q, int(k)))
    return b, pairs


# ---------------------------------------------------------------- count / set pins

def check_page_counts():
    bad = []
    for e in GOLDEN["pair_counts"]:
        got = mask_of(e).count_pairs()
        if got != e["pairs"]:
            bad.append(f"pairs {e['source']}: got {got}, page says {e['pairs']}")
    return bad


def check_row_sets():
    bad = []
    for e in GOLDEN["row_sets"]:
        got = mask_of(e).row_set(e["row"]).tolist()
        want = e["set"] if "set" in e else list(range(e["range"][0], e["range"][1] + 1))
        if got != want:
            bad.append(f"row set {e['source']}: got {got[:8]}..({len(got)}), want "
                       f"{want[:8]}..({len(want)})")
    return bad


def check_reach():
    bad = []
    for e in GOLDEN["reach"]:
        m = oracle.Mask(e["T"], 1, e["window"])
        R = reach_after(oracle_dense(m), e["layers"])
        got = np.nonzero(R[e["row"]])[0].tolist()
        if "set" in e and got != e["set"]:
            bad.append(f"reach {e['source']}: got {got}")
        if "width" in e and len(got) != e["width"]:
            bad.append(f"reach width {e['source']}: got {len(got)}")
    # the closed form at every depth and every row (glossary reach formula)
    for T, w in [(16, 4), (6, 2), (32, 8), (20, 1)]:
        M = oracle_dense(oracle.Mask(T, 1, w))
        for L in range(0, 7):
            R = reach_after(M, L)
            for i in range(T):
                want = list(range(max(0, i - L * (w - 1)), i + 1))
                got = np.nonzero(R[i])[0].tolist()
                if got != want:
                    bad.append(f"reach T={T} w={w} L={L} i={i}: {got} != {want}")
                    break
    # exercise: n = 32, w = 8: last token reaches the first after ceil(31/7) = 5 layers
    M = oracle_dense(oracle.Mask(32, 1, 8))
    first = next(L for L in range(1, 40) if reach_after(M, L)[31, 0])
    if first != 5:
        bad.append(f"n=32 w=8 layers to reach first token: {first} != 5")
    return bad


def check_edge_formula():
    bad = []
    for n in range(1, 41):
        for w in range(1, n + 1):
            got = oracle.Mask(n, 1, w).count_pairs()
            want = n * w - w * (w - 1) // 2
            if got != want:
                bad.append(f"E(n={n}, w={w}) = {got} != {want}")
    # the exercise's n = 32, w = 8 (answer not printed; formula gives 228)
    if oracle.Mask(32, 1, 8).count_pairs() != 228:
        bad.append("n=32 w=8 != 228")
    # the 32K / W=4096 workload: exact E, the page's 134M is N*W
    if oracle.Mask(32768, 1, 4096).count_pairs() != 32768 * 4096 - 4096 * 4095 // 2:
        bad.append("E(32768, 4096)")
    return bad


def check_dilated_counts():
    """The dilated causal window of the "Attention variants" exercise (section 6,
    dilated(n, w, d)): row i reads i, i-d, ..., i-(w-1)d, those >= 0, so its count is
    min(w, floor(i/d) + 1).  The exercise asks for n=16, w=4, d=2 (not printed: the
    closed form gives 52)."""
    bad = []
    for n, w, d in [(16, 4, 2), (30, 5, 3), (64, 8, 7), (20, 1, 4), (33, 40, 2), (50, 0, 3)]:
        cap = w if w else n  # window 0: no limit
        want = sum(min(cap, i // d + 1) for i in range(n))
        got = oracle.Mask(n, 1, w, dilation=d).count_pairs()
        if got != want:
            bad.append(f"dilated count n={n} w={w} d={d}: {got} != {want}")
    if oracle.Mask(16, 1, 4, dilation=2).count_pairs() != 52:
        bad.append("dilated(16, 4, 2) != 52")
    if oracle.Mask(16, 1, 4, dilation=2).row_set(15).tolist() != [9, 11, 13, 15]:
        bad.append("dilated(16, 4, 2): query 15 does not read 9, 11, 13, 15")
    # bidirectional radius r on the dilation grid: 2r+1 keys away from the ends
    m = oracle.Mask(40, 0, 0, 3, dilation=4)
    if m.row_set(20).tolist() != [8, 12, 16, 20, 24, 28, 32]:
        bad.append("bidirectional r=3 d=4 row 20")
    # dilation 1 is the contiguous window
    for T, w in [(30, 7), (17, 1)]:
        if oracle.Mask(T, 1, w, dilation=1).count_pairs() != oracle.Mask(T, 1, w).count_pairs():
            bad.append("dilation 1 differs from the plain window")
    return bad


def check_causal_equivalences():
    bad = []
    for T in [1, 2, 5, 16, 33]:
        tri = T * (T + 1) // 2
        for s in [0, 3]:
            if oracle.Mask(T, 1, 0, -1, s, 0).count_pairs() != tri:
                bad.append(f"window=0 stride={s} T={T} is not the triangle")
        for w in [T, T + 1, 5 * T]:
            for i in range(T):
                if oracle.Mask(T, 1, w).row_set(i).tolist() != list(range(i + 1)):
                    bad.append(f"window={w} >= T={T} row {i} is not causal")
                    break
        if oracle.Mask(T, 0, 0, -1).count_pairs() != T * T:
            bad.append(f"unbounded bidirectional T={T} is not full")
    return bad


def check_against_numpy_rules(seed=0):
    bad = []
    for e in small_specs(seed):
        m = mask_of(e)
        if m.validate() != 0:
            bad.append(f"valid spec rejected: {e}")
            continue
        D = dense_of(e)
        for i in range(e["T"]):
            u = m.row_set(i, "union").tolist()
            s = m.row_set(i, "scan").tolist()
            ref = np.nonzero(D[i])[0].tolist()
            if u != ref or s != ref:
                bad.append(f"row {i} of {e}: union {u[:6]} scan {s[:6]} numpy {ref[:6]}")
                break
        if m.count_pairs() != int(D.sum()):
            bad.append(f"count of {e}")
        if not e.get("rand_pairs") and closed_form_pairs(
                e["T"], e["causal"], e["window"], e["radius"], e["stride"], e["offset"],
                e["global_pos"], e["dilation"]) != int(D.sum()):
            bad.append(f"closed form of {e}")
        for BM, BN in [(4, 4), (8, 16), (128, 128)]:
            cnt = m.tile_counts(BM, BN)
            T = e["T"]
            nq, nk = -(-T // BM), -(-T // BN)
            P = np.zeros((nq * BM, nk * BN), dtype=np.int64)
            P[:T, :T] = D
            ref = P.reshape(nq, BM, nk, BN).sum(axis=(1, 3))
            if not np.array_equal(cnt, ref):
                bad.append(f"tiles {BM}x{BN} of {e}")
    return bad


def check_bigbird_cost():
    """"Sparse and sliding-window attention", §Block-sparse attention: BigBird: a token
    pays W + R + G instead of N, with block 64, W = 3 blocks = 192, R = 3 random blocks
    and G = 2 global blocks.  Causal reading: window 192, the first 128 tokens global,
    three random key blocks per query block drawn from the blocks that lie wholly before
    the query block's window and after the global blocks, so the rules do not overlap:
    every non-global row i >= 5 * 64 + 192 reads exactly 192 + 3 * 64 + 128 = 512 keys."""
    bad = []
    T, b = 2048, 64
    rng = np.random.default_rng(11)
    pairs = []
    for q in range(T // b):
        first_window_block = max(0, (q * b - 191) // b)
        cand = [k for k in range(2, first_window_block)]
        if len(cand) >= 3:
            pairs += [(q, int(k)) for k in sorted(rng.choice(cand, 3, replace=False))]
    m = oracle.Mask(T, 1, 192, -1, 0, 0, list(range(128)), 1, b, pairs)
    if m.validate() != 0:
        return ["BigBird spec rejected"]
    have = {q for q, _ in pairs}
    for i in range(5 * b + 192, T, 37):
        if i // b not in have:
            continue
        n = len(m.row_set(i))
        if n != 512:
            bad.append(f"BigBird row {i}: {n} keys, page cost W + R + G = 512")
    if not bad and not any(i // b in have for i in range(5 * b + 192, T, 37)):
        bad.append("no eligible BigBird row")
    return bad


def check_rejects_invalid():
    bad = []
    for rb, pairs in [(48, [(0, 0)]), (16, [(0, 5)]), (16, [(1, 0), (0, 0)]),
                      (16, [(0, 1), (0, 1)]), (16, [(-1, 0)])]:
        if oracle.Mask(40, 0, 0, 2, 0, 0, [], 1, rb, pairs).validate() == 0:
            bad.append(f"invalid random blocks accepted: {rb} {pairs}")
    cases = [
        dict(T=0), dict(T=8, causal=2), dict(T=8, causal=1, window=-1),
        dict(T=8, causal=1, radius=2), dict(T=8, causal=0, radius=-2),
        dict(T=8, causal=0, window=3, radius=1), dict(T=8, stride=-1),
        dict(T=8, stride=4, offset=4), dict(T=8, stride=0, offset=1),
        dict(T=8, global_pos=[8]), dict(T=8, global_pos=[-1]),
        dict(T=8, global_pos=[3, 3]), dict(T=8, dilation=0),
    ]
    for c in cases:
        if mask_of(c).validate() == 0:
            bad.append(f"invalid spec accepted: {c}")
    return bad


# ---------------------------------------------------------------- attention pins

def _rand(T, d, seed, scale_std=1.0):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(T, d, generator=g, dtype=torch.float32) * scale_std)
            for _ in range(3)]


def _oracle_attn(m, Q, K, V, scale, rows=None):
    return oracle.attention(m, Q.numpy(), K.numpy(), V.numpy(), scale, rows)


def check_sdpa_dense():
    """Unrestricted masks against torch's fp64 SDPA (a library routine)."""
    bad = []
    for T, d, seed in [(37, 16, 1), (64, 64, 2), (129, 32, 3)]:
        Q, K, V = _rand(T, d, seed)
        sc = 1.0 / math.sqrt(d)
        q, k, v = (x.double()[None, None] for x in (Q, K, V))
        full = torch.nn.functional.scaled_dot_product_attention(q, k, v)[0, 0].numpy()
        caus = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=True)[0, 0].numpy()
        logits = (q @ k.transpose(-1, -2))[0, 0] * sc
        lse_full = torch.logsumexp(logits, dim=-1).numpy()
        tri = torch.ones(T, T, dtype=torch.bool).tril()
        lse_caus = torch.logsumexp(logits.masked_fill(~tri, -math.inf), dim=-1).numpy()
        O, L = _oracle_attn(oracle.Mask(T, 0, 0, -1), Q, K, V, sc)
        if not (np.allclose(O, full, rtol=0, atol=1e-12) and
                np.allclose(L, lse_full, rtol=0, atol=1e-12)):
            bad.append(f"all-true mask vs SDPA T={T} d={d}: "
                       f"{np.abs(O - full).max():.3g} {np.abs(L - lse_full).max():.3g}")
        O, L = _oracle_attn(oracle.Mask(T, 1, 0), Q, K, V, sc)
        if not (np.allclose(O, caus, rtol=0, atol=1e-12) and
                np.allclose(L, lse_caus, rtol=0, atol=1e-12)):
            bad.append(f"window=0 vs causal SDPA T={T} d={d}")
    return bad


def check_sdpa_masked(seed=5):
    """Every sweep mask against SDPA with the independent numpy boolean mask."""
    bad = []
    for n, e in enumerate(small_specs(seed, n=25)):
        T = e["T"]
        d = 8 + 8 * (n % 3)
        Q, K, V = _rand(T, d, 100 + n)
        sc = 0.7 / math.sqrt(d)
        D = torch.from_numpy(dense_of(e))
        q, k, v = (x.double()[None, None] for x in (Q, K, V))
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=D[None, None], scale=sc)[0, 0].numpy()
        lse = torch.logsumexp(((q @ k.transpose(-1, -2))[0, 0] * sc).masked_fill(
            ~D, -math.inf), dim=-1).numpy()
        O, L = _oracle_attn(mask_of(e), Q, K, V, sc)
        if not (np.allclose(O, ref, rtol=0, atol=1e-12) and
                np.allclose(L, lse, rtol=0, atol=1e-12)):
            bad.append(f"masked SDPA mismatch for {e}: {np.abs(O - ref).max():.3g}")
    return bad


def check_special_values():
    bad = []
    T, d = 50, 16
    Q, K, V = _rand(T, d, 11)
    sc = 1.0 / math.sqrt(d)
    # w = 1: S_i = {i}, so y_i = v_i exactly and LSE_i = scale q_i.k_i
    O, L = _oracle_attn(oracle.Mask(T, 1, 1), Q, K, V, sc)
    if not np.array_equal(O, V.double().numpy()):
        bad.append("w=1 does not return V")
    s_ii = sc * (Q.double() * K.double()).sum(-1).numpy()
    if not np.allclose(L, s_ii, rtol=0, atol=1e-13):
        bad.append("w=1 LSE is not the self logit")
    # Q = 0: uniform weights over S_i: y_i = mean of allowed values, LSE = ln |S_i|
    for e in small_specs(9, n=8) + [dict(T=T, causal=1, window=7, stride=5, offset=2,
                                         global_pos=[3, 40])]:
        m = mask_of(e)
        Tn = e["T"]
        Qz = torch.zeros(Tn, d)
        _, Kr, Vr = _rand(Tn, d, 12)
        O, L = _oracle_attn(m, Qz, Kr, Vr, sc)
        for i in range(Tn):
            S = m.row_set(i)
            want = Vr.double().numpy()[S].mean(axis=0)
            if not np.allclose(O[i], want, rtol=0, atol=1e-13) or not math.isclose(
                    L[i], math.log(len(S)), abs_tol=1e-13):
                bad.append(f"Q=0 row {i} of {e}")
                break
    # shift invariance: k_j -> k_j + u adds scale q_i.u to every logit of row i
    m = oracle.Mask(T, 0, 0, 3, 4, 1, [7, 30])
    u = torch.randn(d, generator=torch.Generator().manual_seed(13))
    O1, L1 = _oracle_attn(m, Q, K, V, sc)
    O2, L2 = _oracle_attn(m, Q, K + u, V, sc)
    shift = sc * (Q.double() @ u.double()).numpy()
    if not (np.allclose(O1, O2, rtol=0, atol=1e-6) and
            np.allclose(L2 - L1, shift, rtol=0, atol=1e-5)):
        bad.append("key-shift invariance")
    # bf16 bit-pattern input path equals the fp32 path on the same (exact) values
    Qb, Kb, Vb = (x.to(torch.bfloat16) for x in (Q, K, V))
    Ob, Lb = oracle.attention(m, oracle.bf16_bits(Qb), oracle.bf16_bits(Kb),
                              oracle.bf16_bits(Vb), sc)
    Of, Lf = _oracle_attn(m, Qb.float(), Kb.float(), Vb.float(), sc)
    if not (np.array_equal(Ob, Of) and np.array_equal(Lb, Lf)):
        bad.append("bf16-bits input path differs from the fp32 path")
    # row subsets give the same rows as the full evaluation
    rows = np.array([0, 5, 49, 17], dtype=np.int64)
    Os, Ls = _oracle_attn(m, Q, K, V, sc, rows)
    if not (np.array_equal(Os, O1[rows]) and np.array_equal(Ls, L1[rows])):
        bad.append("row subset differs")
    # renormalising over S_i is not the same as deleting weights after a full
    # softmax (glossary, §Choose the available reads)
    full = torch.softmax(sc * Q.double() @ K.double().T, dim=-1)
    D = torch.from_numpy(np_dense_mask(T, 0, 0, 3, 4, 1, [7, 30]))
    deleted = (full * D) @ V.double()
    if np.allclose(O1, deleted.numpy(), atol=1e-3):
        bad.append("renormalised result equals the deleted-weights result")
    return bad


# ---------------------------------------------------------------- gradient pins

def _oracle_bwd(m, Q, K, V, dO, scale):
    return oracle.attention_bwd(m, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), scale)


def check_bwd_autograd(seed=21):
    """Gradients against torch's fp64 autograd through SDPA with the independent numpy
    boolean mask (a library routine): one dense, one causal and the sweep masks."""
    bad = []
    specs = [dict(T=33, causal=0, window=0, radius=-1, stride=0, offset=0, global_pos=[],
                  dilation=1),
             dict(T=40, causal=1, window=0, radius=-1, stride=0, offset=0, global_pos=[],
                  dilation=1)] + small_specs(seed, n=16)
    for n, e in enumerate(specs):
        T = e["T"]
        d = 8 + 8 * (n % 2)
        g = torch.Generator().manual_seed(300 + n)
        Q, K, V, dO = (torch.randn(T, d, generator=g) for _ in range(4))
        sc = 0.6 / math.sqrt(d)
        D = torch.from_numpy(dense_of(e))
        q, k, v = (x.double().requires_grad_(True) for x in (Q, K, V))
        y = torch.nn.functional.scaled_dot_product_attention(
            q[None, None], k[None, None], v[None, None], attn_mask=D[None, None],
            scale=sc)[0, 0]
        y.backward(dO.double())
        got = _oracle_bwd(mask_of(e), Q, K, V, dO, sc)
        for name, a, b in zip("QKV", got, (q.grad, k.grad, v.grad)):
            if not np.allclose(a, b.numpy(), rtol=0, atol=1e-11):
                bad.append(f"d{name} vs autograd for {e}: {np.abs(a - b.numpy()).max():.3g}")
    return bad


def check_bwd_finite_differences():
    """Central differences of the forward oracle's loss L = sum(y * dO) for sampled
    entries of Q, K and V (fp32 inputs; the step actually taken is the fp32 one)."""
    bad = []
    T, d = 24, 8
    m = oracle.Mask(T, 1, 6, -1, 5, 3, [2, 17])
    g = torch.Generator().manual_seed(41)
    X = [torch.randn(T, d, generator=g) for _ in range(3)]
    dO = torch.randn(T, d, generator=g)
    sc = 0.5
    grads = _oracle_bwd(m, *X, dO, sc)
    W = dO.double().numpy()

    def loss(Xs):
        O, _ = oracle.attention(m, *(x.numpy() for x in Xs), sc)
        return float((O * W).sum())

    rng = np.random.default_rng(7)
    for which in range(3):
        for _ in range(12):
            i, k = int(rng.integers(T)), int(rng.integers(d))
            base = X[which][i, k].item()
            hp = np.float32(base + 1e-2)
            hm = np.float32(base - 1e-2)
            Xp = [x.clone() for x in X]
            Xm = [x.clone() for x in X]
            Xp[which][i, k] = float(hp)
            Xm[which][i, k] = float(hm)
            fd = (loss(Xp) - loss(Xm)) / (float(hp) - float(hm))
            if not math.isclose(fd, grads[which][i, k], rel_tol=1e-3, abs_tol=1e-5):
                bad.append(f"d{'QKV'[which]}[{i},{k}] = {grads[which][i, k]:.6g}, "
                           f"central difference {fd:.6g}")
    return bad


def check_bwd_invariants():
    """Identities of the softmax over S_i: sum_j dV_j = sum_i dO_i (weights sum to 1);
    sum_j dK_j = 0 (each row's ds sums to 0); with w = 1 (S_i = {i}) dV = dO and
    dQ = dK = 0; with Q = 0 and dO = 0 everything is 0."""
    bad = []
    for e in small_specs(33, n=10):
        T = e["T"]
        d = 8
        g = torch.Generator().manual_seed(500 + T)
        Q, K, V, dO = (torch.randn(T, d, generator=g) for _ in range(4))
        dQ, dK, dV = _oracle_bwd(mask_of(e), Q, K, V, dO, 0.4)
        if not np.allclose(dV.sum(0), dO.double().numpy().sum(0), rtol=0, atol=1e-10):
            bad.append(f"sum dV != sum dO for {e}")
        if not np.allclose(dK.sum(0), 0.0, rtol=0, atol=1e-10):
            bad.append(f"sum dK != 0 for {e}")
    T, d = 30, 8
    g = torch.Generator().manual_seed(77)
    Q, K, V, dO = (torch.randn(T, d, generator=g) for _ in range(4))
    dQ, dK, dV = _oracle_bwd(oracle.Mask(T, 1, 1), Q, K, V, dO, 0.4)
    if not (np.array_equal(dV, dO.double().numpy()) and not dQ.any() and not dK.any()):
        bad.append("w=1 gradients")
    dQ, dK, dV = _oracle_bwd(oracle.Mask(T, 0, 0, 4), Q, K, V, torch.zeros(T, d), 0.4)
    if dQ.any() or dK.any() or dV.any():
        bad.append("dO = 0 gives nonzero gradients")
    # the row-subset dQ equals the full evaluation's rows
    m = oracle.Mask(T, 1, 5, -1, 4, 1, [3, 20])
    dQ, _, _ = _oracle_bwd(m, Q, K, V, dO, 0.4)
    rows = np.array([29, 0, 3, 20, 11], dtype=np.int64)
    sub = oracle.attention_bwd_dq(m, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), 0.4, rows)
    if not np.array_equal(sub, dQ[rows]):
        bad.append("row-subset dQ differs from the full evaluation")
    return bad


def check_bwd_key_subset(seed=23):
    """dK and dV of listed keys only, against torch's fp64 autograd through SDPA with
    the independent numpy mask (the same library pin as the full gradient), on masks
    with every rule (dilated, strided, global, random blocks), the edge keys 0 and
    T - 1 always among the listed ones; and equal to the full evaluation's rows."""
    bad = []
    specs = [dict(T=37, causal=1, window=5, radius=-1, stride=4, offset=1, global_pos=[3, 30],
                  dilation=1),
             dict(T=45, causal=0, window=0, radius=3, stride=0, offset=0, global_pos=[0],
                  dilation=2)] + small_specs(seed, n=14)
    rng = np.random.default_rng(seed)
    for n, e in enumerate(specs):
        T = e["T"]
        d = 8
        g = torch.Generator().manual_seed(700 + n)
        Q, K, V, dO = (torch.randn(T, d, generator=g) for _ in range(4))
        sc = 0.5 / math.sqrt(d)
        keys = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=min(T, 5),
                                                                replace=False)])).astype(np.int64)
        rng.shuffle(keys)
        D = torch.from_numpy(dense_of(e))
        q, k, v = (x.double().requires_grad_(True) for x in (Q, K, V))
        y = torch.nn.functional.scaled_dot_product_attention(
            q[None, None], k[None, None], v[None, None], attn_mask=D[None, None],
            scale=sc)[0, 0]
        y.backward(dO.double())
        m = mask_of(e)
        dK, dV = oracle.attention_bwd_dkdv(m, Q.numpy(), K.numpy(), V.numpy(), dO.numpy(), sc,
                                           keys)
        for name, a, b in (("dK", dK, k.grad), ("dV", dV, v.grad)):
            ref = b.numpy()[keys]
            if not np.allclose(a, ref, rtol=0, atol=1e-11):
                bad.append(f"{name} of keys {keys.tolist()} vs autograd for {e}: "
                           f"{np.abs(a - ref).max():.3g}")
        _, fK, fV = _oracle_bwd(m, Q, K, V, dO, sc)
        if not (np.allclose(dK, fK[keys], rtol=0, atol=1e-12) and
                np.allclose(dV, fV[keys], rtol=0, atol=1e-12)):
            bad.append(f"key-subset dK/dV differ from the full evaluation for {e}")
    return bad


# ---------------------------------------------------------------- decode pins

def ring_fill(K, t, cap):
    """The cache after writing positions 0..t of K in order, position p to slot
    p % cap (later positions overwrite earlier ones)."""
    Kc = np.zeros((cap, K.shape[1]), K.dtype)
    for p in range(t + 1):
        Kc[p % cap] = K[p]
    return Kc


def check_decode_matches_sequence_rows():
    """A decode step equals row t of the forward oracle on the whole sequence with the
    causal window w, for a cache filled by the ring rule (t below, at and far above
    the capacity; window below and equal to the capacity)."""
    bad = []
    T, d = 300, 16
    g = torch.Generator().manual_seed(61)
    Q, K, V = (torch.randn(T, d, generator=g).numpy() for _ in range(3))
    for cap, w in [(64, 64), (64, 17), (100, 1), (37, 37)]:
        m = oracle.Mask(T, 1, w)
        for t in [0, 5, cap - 1, cap, cap + 3, 2 * cap + 7, T - 1]:
            O, L = oracle.attention(m, Q, K, V, 0.3, np.array([t], dtype=np.int64))
            out, lse = oracle.decode(Q[t], ring_fill(K, t, cap), ring_fill(V, t, cap), t, w, 0.3)
            if not (np.allclose(out, O[0], rtol=0, atol=1e-12) and abs(lse - L[0]) < 1e-12):
                bad.append(f"decode cap={cap} w={w} t={t} != sequence row")
    return bad


def check_decode_special():
    """Against torch fp64 SDPA: with t < cap and w = cap the cache is the prefix and
    the step is the causal attention row; the cache's slot order does not matter
    (softmax over a set); a token before any key (t < 0) reads nothing."""
    bad = []
    cap, d = 50, 8
    g = torch.Generator().manual_seed(62)
    q, K, V = torch.randn(d, generator=g), torch.randn(cap, d, generator=g), torch.randn(cap, d, generator=g)
    for t in [0, 1, 20, 49]:
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.double()[None, None, None], K.double()[None, None, :t + 1],
            V.double()[None, None, :t + 1], scale=0.5)[0, 0, 0].numpy()
        out, _ = oracle.decode(q.numpy(), K.numpy(), V.numpy(), t, cap, 0.5)
        if not np.allclose(out, ref, rtol=0, atol=1e-12):
            bad.append(f"prefix decode t={t} vs SDPA")
    # t >= cap - 1 with w = cap reads every slot: any permutation of the slots agrees
    perm = np.random.default_rng(3).permutation(cap)
    a, la = oracle.decode(q.numpy(), K.numpy(), V.numpy(), 1000, cap, 0.5)
    b, lb = oracle.decode(q.numpy(), K.numpy()[perm], V.numpy()[perm], 1000, cap, 0.5)
    if not (np.allclose(a, b, rtol=0, atol=1e-12) and abs(la - lb) < 1e-12):
        bad.append("full-cache decode depends on slot order")
    out, lse = oracle.decode(q.numpy(), K.numpy(), V.numpy(), -1, cap, 0.5)
    if out.any() or lse != -math.inf:
        bad.append("t < 0 is not empty")
    return bad


DECODE_CHECKS = [check_decode_matches_sequence_rows, check_decode_special]

BWD_CHECKS = [check_bwd_autograd, check_bwd_finite_differences, check_bwd_invariants,
              check_bwd_key_subset]

COUNT_CHECKS = [check_page_counts, check_row_sets, check_reach, check_edge_formula,
                check_dilated_counts, check_causal_equivalences, check_against_numpy_rules,
                check_rejects_invalid, check_bigbird_cost]
ATTENTION_CHECKS = [check_sdpa_dense, check_sdpa_masked, check_special_values]
