"""Seeded synthetic workloads shared by the tests, the benchmark and the smoke check.

This module only *draws inputs*: shapes, mask-rule parameters and random numbers.  It
holds none of the attention arithmetic (no masks, no counts, no softmax), so the CPU
oracle and the CUDA path can both be fed from it without sharing any of the method.

Workload shapes follow the pages' own examples:
  * EXP-017 lab note ("Sparse attention", octlm.ramaa.tech, §Worse on code, and no
    faster at this length): 512-token context, windows 128/256, strides 0/64.
  * "Sparse and sliding-window attention" (getnybble.com, §Sliding window attention):
    Mistral-style W=4096 at a 32K context, and the 128K context it compares against.
  * "Sparse Attention" (ai360xpert.com, §Combined complexity): N=16384, W=512,
    stride 16, 128 global tokens.
  * "Sparse and sliding-window attention" (getnybble.com, §Dilated sliding window):
    W=512 keys with dilation 2, here at the 32K context.
Q, K and V are i.i.d. N(0, 1) drawn in fp32 from ``torch.Generator().manual_seed``;
bf16 inputs are the round-to-nearest-even casts of those fp32 draws.
"""
from __future__ import annotations

import numpy as np
import torch

# Mask-rule parameters.  causal=1 uses `window` (0 = unbounded); causal=0 uses
# `radius` (-1 = unbounded).  `stride`/`offset` select strided global columns
# (j % stride == offset); `n_global` positions are drawn by `global_positions`.
WORKLOADS = {
    # 512-token EXP-017 shapes (B=1, H=2, d=64); fp32 and bf16 inputs.
    "t512_w128_s0": dict(B=1, H=2, T=512, d=64, causal=1, window=128, radius=-1,
                         stride=0, offset=0, n_global=0),
    "t512_w128_s64": dict(B=1, H=2, T=512, d=64, causal=1, window=128, radius=-1,
                          stride=64, offset=0, n_global=0),
    "t512_full_causal": dict(B=1, H=2, T=512, d=64, causal=1, window=0, radius=-1,
                             stride=0, offset=0, n_global=0),
    # 2048-token, 4x12 heads, window 256.
    "t2048_w256_s0": dict(B=4, H=12, T=2048, d=64, causal=1, window=256, radius=-1,
                          stride=0, offset=0, n_global=0),
    "t2048_w256_s64": dict(B=4, H=12, T=2048, d=64, causal=1, window=256, radius=-1,
                           stride=64, offset=0, n_global=0),
    # Mistral-style sliding window at a 32K context.
    "t32k_w4096": dict(B=1, H=32, T=32768, d=128, causal=1, window=4096, radius=-1,
                       stride=0, offset=0, n_global=0),
    # Long-document encoder pattern: radius 256 (width 512), stride 16, 128 globals.
    "t16k_r256_s16_g128": dict(B=1, H=16, T=16384, d=64, causal=0, window=0,
                               radius=256, stride=16, offset=0, n_global=128,
                               global_seed=0),
    # 128K context with window 4096 and landmark columns every 1024 keys,
    # and the full causal 8K run it is compared against.
    "t128k_w4096_s1024": dict(B=1, H=32, T=131072, d=128, causal=1, window=4096,
                              radius=-1, stride=1024, offset=0, n_global=0),
    "t8k_full_causal": dict(B=1, H=32, T=8192, d=128, causal=1, window=0, radius=-1,
                            stride=0, offset=0, n_global=0),
    # BigBird encoder ("Sparse and sliding-window attention", Block-sparse attention:
    # BigBird): block 64, a window of 3 blocks (radius 96), R = 3 random key blocks
    # per query block, G = 2 global blocks (the first 128 tokens); BigBird-base shape
    # (12 heads of 64) at 4096 tokens.
    "t4096_bigbird": dict(B=8, H=12, T=4096, d=64, causal=0, window=0, radius=96, stride=0,
                          offset=0, n_global=0, global_first=128, rand_block=64, rand_per_block=3,
                          rand_seed=0),
    # Longformer-style dilated window: 512 keys spaced 2 apart (a 1023-token span).
    "t32k_w512_d2": dict(B=1, H=32, T=32768, d=128, causal=1, window=512, radius=-1,
                         stride=0, offset=0, n_global=0, dilation=2),
}


# Decode workloads: one generation step of B sequences against a ring-buffer KV cache
# of cap = W = 4096 slots (the Mistral 7B shape of "Sparse and sliding-window
# attention": W = 4096, 32 query heads over 8 key/value heads, d = 128), every
# sequence past the cap so the whole window is read.
DECODE_WORKLOADS = {
    "decode_b32_w4096": dict(B=32, Hq=32, Hkv=8, cap=4096, window=4096, d=128),
    "decode_b8_w4096": dict(B=8, Hq=32, Hkv=8, cap=4096, window=4096, d=128),
}


def decode_positions(B: int, cap: int, seed: int) -> np.ndarray:
    """Per-sequence positions, all past the cap (seeded uniform in [cap, 2^20))."""
    return np.random.default_rng(seed + 31337).integers(cap, 1 << 20, size=B).astype(np.int64)


def global_positions(T: int, g: int, seed: int) -> np.ndarray:
    """`g` distinct token positions in [0, T), sorted, drawn from numpy's PCG64."""
    if g == 0:
        return np.zeros(0, dtype=np.int32)
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(T, size=g, replace=False)).astype(np.int32)


def mask_params(name_or_cfg, seed_override=None) -> dict:
    """The mask-rule fields of a workload, with global positions drawn."""
    cfg = WORKLOADS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    gseed = cfg.get("global_seed", 0) if seed_override is None else seed_override
    if cfg.get("global_first"):
        gpos = np.arange(cfg["global_first"], dtype=np.int32)
    else:
        gpos = global_positions(cfg["T"], cfg["n_global"], gseed)
    out = dict(causal=cfg["causal"], window=cfg["window"], radius=cfg["radius"],
               stride=cfg["stride"], offset=cfg["offset"], global_pos=gpos,
               dilation=cfg.get("dilation", 1))
    if cfg.get("rand_block"):
        out["rand_block"] = cfg["rand_block"]
        out["rand_pairs"] = random_block_pairs(cfg["T"], cfg["rand_block"],
                                               cfg["rand_per_block"], cfg.get("rand_seed", 0))
    return out


def random_block_pairs(T: int, b: int, R: int, seed: int) -> np.ndarray:
    """BigBird random connections as (query block, key block) pairs: for every query
    block, R distinct key blocks drawn uniformly from all ceil(T / b) blocks with
    numpy's PCG64 (fewer when there are fewer blocks).  [n, 2] int32, sorted."""
    rng = np.random.default_rng(seed + 4242)
    nb = -(-T // b)
    pairs = [(q, int(k)) for q in range(nb)
             for k in np.sort(rng.choice(nb, size=min(R, nb), replace=False))]
    return np.asarray(pairs, dtype=np.int32).reshape(-1, 2)


def qkv(B: int, H: int, T: int, d: int, seed: int, dtype=torch.bfloat16):
    """Q, K, V of shape [B, H, T, d] (contiguous, CPU), i.i.d. N(0,1) from `seed`."""
    g = torch.Generator().manual_seed(int(seed))
    out = []
    for _ in range(3):
        x = torch.randn(B, H, T, d, generator=g, dtype=torch.float32)
        out.append(x.to(dtype).contiguous())
    return tuple(out)


def grad_out(B: int, H: int, T: int, d: int, seed: int, dtype=torch.bfloat16):
    """dO of shape [B, H, T, d] (contiguous, CPU), i.i.d. N(0,1), drawn from a stream
    of its own (seed + 104729) so that it is independent of Q, K, V."""
    g = torch.Generator().manual_seed(int(seed) + 104729)
    return torch.randn(B, H, T, d, generator=g, dtype=torch.float32).to(dtype).contiguous()


def sample_rows(T: int, n: int, seed: int, must=()) -> np.ndarray:
    """Sorted distinct query rows: `must` (clipped to [0,T)) plus seeded uniform picks."""
    rng = np.random.default_rng(seed + 7919)
    rows = set(int(r) for r in must if 0 <= int(r) < T)
    want = min(T, max(n, len(rows)))
    while len(rows) < want:
        rows.update(int(x) for x in rng.integers(0, T, size=want - len(rows)))
    return np.array(sorted(rows), dtype=np.int64)
