"""Python entry points to the fp64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke`` and by
the benchmark's CPU-baseline / reference leg.  The CUDA library never imports it.

Every function takes the mask as plain fields (causal, window, radius, stride,
offset, global_pos, dilation) and calls the C code compiled from ``oracle.c`` with gcc.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc -O2 -fopenmp, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    spec = [ctypes.c_int, _i64, _i64, _i64, _i64, _i64, _i64, _i32p, _i64, _i64, _i64, _i32p]
    lib.oracle_validate.argtypes = spec
    lib.oracle_validate.restype = ctypes.c_int
    lib.oracle_allowed.argtypes = spec + [_i64, _i64]
    lib.oracle_allowed.restype = ctypes.c_int
    lib.oracle_row_set.argtypes = spec + [_i64, ctypes.c_int, _i32p]
    lib.oracle_row_set.restype = _i64
    lib.oracle_count_pairs.argtypes = spec
    lib.oracle_count_pairs.restype = _i64
    lib.oracle_tile_counts.argtypes = spec + [_i64, _i64, _i32p]
    lib.oracle_tile_counts.restype = None
    lib.oracle_attention_head.argtypes = spec + [
        _i64, ctypes.c_int, _vp, _vp, _vp, ctypes.c_double,
        ctypes.POINTER(ctypes.c_int64), _i64,
        ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    lib.oracle_attention_head.restype = _i64
    lib.oracle_attention_bwd_head.argtypes = spec + [
        _i64, ctypes.c_int, _vp, _vp, _vp, _vp, ctypes.c_double,
        ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
        ctypes.POINTER(ctypes.c_double)]
    lib.oracle_attention_bwd_head.restype = None
    lib.oracle_attention_bwd_dq_rows.argtypes = spec + [
        _i64, ctypes.c_int, _vp, _vp, _vp, _vp, ctypes.c_double, _vp, _i64,
        ctypes.POINTER(ctypes.c_double)]
    lib.oracle_attention_bwd_dq_rows.restype = None
    lib.oracle_attention_bwd_dkdv_keys.argtypes = spec + [
        _i64, ctypes.c_int, _vp, _vp, _vp, _vp, ctypes.c_double, _vp, _i64,
        ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    lib.oracle_attention_bwd_dkdv_keys.restype = None
    lib.oracle_decode.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int, _vp, _vp, _vp,
                                  ctypes.c_double, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double)]
    lib.oracle_decode.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


class use_library:
    """Context manager: route every oracle call through another build of oracle.c.

    Used by the mutation tests, which compile deliberately broken copies of the
    oracle and check that the pins reject them."""

    def __init__(self, so_path: str):
        self.lib = _configure(ctypes.CDLL(so_path))

    def __enter__(self):
        global _lib
        _load()
        self.saved = _lib
        _lib = self.lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


class Mask:
    """A mask rule: causal window / bidirectional radius (optionally dilated), strided
    columns, globals."""

    def __init__(self, T, causal=1, window=0, radius=-1, stride=0, offset=0,
                 global_pos=(), dilation=1, rand_block=0, rand_pairs=()):
        self.T = int(T)
        self.causal = int(causal)
        self.window = int(window)
        self.radius = int(radius)
        self.dilation = int(dilation)
        self.stride = int(stride)
        self.offset = int(offset)
        self.gpos = np.ascontiguousarray(np.asarray(global_pos, dtype=np.int32))
        self.rand_block = int(rand_block)
        rp = np.asarray(rand_pairs, dtype=np.int32).reshape(-1, 2)
        self.rand_pairs = np.ascontiguousarray(rp)

    @classmethod
    def from_params(cls, T, p):
        return cls(T, p["causal"], p["window"], p["radius"], p["stride"], p["offset"],
                   p.get("global_pos", ()), p.get("dilation", 1), p.get("rand_block", 0),
                   p.get("rand_pairs", ()))

    def _args(self):
        return (self.causal, self.window, self.radius, self.dilation, self.stride, self.offset,
                len(self.gpos), self.gpos.ctypes.data_as(_i32p), self.T, self.rand_block,
                len(self.rand_pairs), self.rand_pairs.ctypes.data_as(_i32p))

    def validate(self) -> int:
        return _load().oracle_validate(*self._args())

    def allowed(self, i, j) -> bool:
        return bool(_load().oracle_allowed(*self._args(), int(i), int(j)))

    def row_set(self, i, method: str = "union") -> np.ndarray:
        out = np.empty(self.T, dtype=np.int32)
        n = _load().oracle_row_set(*self._args(), int(i), 1 if method == "scan" else 0,
                                   out.ctypes.data_as(_i32p))
        return out[:n].copy()

    def count_pairs(self) -> int:
        return int(_load().oracle_count_pairs(*self._args()))

    def tile_counts(self, BM: int, BN: int) -> np.ndarray:
        nqb = -(-self.T // BM)
        nkb = -(-self.T // BN)
        cnt = np.zeros((nqb, nkb), dtype=np.int32)
        _load().oracle_tile_counts(*self._args(), int(BM), int(BN),
                                   cnt.ctypes.data_as(_i32p))
        return cnt


def tile_list(mask: Mask, BM: int, BN: int):
    """Non-empty tiles in canonical order (qb ascending, then kb ascending).

    Returns (qb, kb, cnt, cls) int32/uint8 arrays; cls 1 = full (every cell of the
    tile inside [0,T)^2 is allowed), 2 = partial.  Also returns the class totals
    (n_full, n_partial, n_empty) over all tiles of the grid.
    """
    cnt = mask.tile_counts(BM, BN)
    T = mask.T
    nqb, nkb = cnt.shape
    rows = np.minimum(BM, T - np.arange(nqb) * BM)[:, None]
    cols = np.minimum(BN, T - np.arange(nkb) * BN)[None, :]
    cells = rows * cols
    qb, kb = np.nonzero(cnt)
    c = cnt[qb, kb]
    cls = np.where(c == cells[qb, kb], 1, 2).astype(np.uint8)
    n_full = int((cls == 1).sum())
    n_partial = int((cls == 2).sum())
    n_empty = int(nqb * nkb - len(c))
    return (qb.astype(np.int32), kb.astype(np.int32), c.astype(np.int32), cls,
            (n_full, n_partial, n_empty))


def attention(mask: Mask, Q, K, V, scale: float, rows=None):
    """fp64 masked attention for one head.

    Q, K, V: [T, d] numpy arrays, float32, or uint16 holding bf16 bit patterns.
    rows: query indices to evaluate (default: all).  Returns (O [n,d] f64, LSE [n] f64).
    """
    T, d = Q.shape
    assert T == mask.T and K.shape == (T, d) and V.shape == (T, d)
    if Q.dtype == np.float32:
        dt = 0
    elif Q.dtype == np.uint16:
        dt = 1
    else:
        raise TypeError("Q/K/V must be float32 or uint16 (bf16 bits)")
    assert K.dtype == Q.dtype and V.dtype == Q.dtype
    Q = np.ascontiguousarray(Q)
    K = np.ascontiguousarray(K)
    V = np.ascontiguousarray(V)
    rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(
        np.asarray(rows, dtype=np.int64))
    O = np.zeros((len(rows), d), dtype=np.float64)
    L = np.zeros(len(rows), dtype=np.float64)
    _load().oracle_attention_head(
        *mask._args(), int(d), dt, Q.ctypes.data, K.ctypes.data, V.ctypes.data,
        float(scale), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(rows),
        O.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        L.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return O, L


def attention_bwd(mask: Mask, Q, K, V, dO, scale: float):
    """fp64 gradients (dQ, dK, dV) [T, d] of the masked attention of one head, given
    dO.  Inputs as for attention(): float32 arrays or uint16 bf16 bit patterns."""
    T, d = Q.shape
    assert T == mask.T and K.shape == (T, d) and V.shape == (T, d) and dO.shape == (T, d)
    if Q.dtype == np.float32:
        dt = 0
    elif Q.dtype == np.uint16:
        dt = 1
    else:
        raise TypeError("inputs must be float32 or uint16 (bf16 bits)")
    assert K.dtype == V.dtype == dO.dtype == Q.dtype
    Q, K, V, dO = (np.ascontiguousarray(x) for x in (Q, K, V, dO))
    dQ = np.zeros((T, d), np.float64)
    dK = np.zeros((T, d), np.float64)
    dV = np.zeros((T, d), np.float64)
    pd = ctypes.POINTER(ctypes.c_double)
    _load().oracle_attention_bwd_head(
        *mask._args(), int(d), dt, Q.ctypes.data, K.ctypes.data, V.ctypes.data,
        dO.ctypes.data, float(scale), dQ.ctypes.data_as(pd), dK.ctypes.data_as(pd),
        dV.ctypes.data_as(pd))
    return dQ, dK, dV


def attention_bwd_dq(mask: Mask, Q, K, V, dO, scale: float, rows):
    """fp64 dQ [len(rows), d] of the listed rows only (each needs only its own set)."""
    T, d = Q.shape
    assert T == mask.T
    dt = 0 if Q.dtype == np.float32 else 1
    Q, K, V, dO = (np.ascontiguousarray(x) for x in (Q, K, V, dO))
    rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rr.size == 0 or (rr.min() >= 0 and rr.max() < T)
    out = np.zeros((rr.size, d), np.float64)
    _load().oracle_attention_bwd_dq_rows(
        *mask._args(), int(d), dt, Q.ctypes.data, K.ctypes.data, V.ctypes.data,
        dO.ctypes.data, float(scale), rr.ctypes.data, int(rr.size),
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def attention_bwd_dkdv(mask: Mask, Q, K, V, dO, scale: float, keys):
    """fp64 (dK, dV), each [len(keys), d], of the listed keys only: every row that
    reads a listed key contributes, with its softmax taken over its whole set."""
    T, d = Q.shape
    assert T == mask.T
    dt = 0 if Q.dtype == np.float32 else 1
    Q, K, V, dO = (np.ascontiguousarray(x) for x in (Q, K, V, dO))
    kk = np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    assert kk.size == 0 or (kk.min() >= 0 and kk.max() < T)
    assert np.unique(kk).size == kk.size, "keys must be distinct"
    dK = np.zeros((kk.size, d), np.float64)
    dV = np.zeros((kk.size, d), np.float64)
    pd = ctypes.POINTER(ctypes.c_double)
    _load().oracle_attention_bwd_dkdv_keys(
        *mask._args(), int(d), dt, Q.ctypes.data, K.ctypes.data, V.ctypes.data,
        dO.ctypes.data, float(scale), kk.ctypes.data, int(kk.size),
        dK.ctypes.data_as(pd), dV.ctypes.data_as(pd))
    return dK, dV


def decode(q, Kc, Vc, t: int, window: int, scale: float):
    """One decode step of one query head against a ring-buffer cache.

    q: [d]; Kc, Vc: [cap, d] (float32, or uint16 bf16 bits); the token at position t
    reads positions max(0, t-window+1) .. t, position p from slot p % cap.
    Returns (out [d] fp64, lse)."""
    cap, d = Kc.shape
    assert Vc.shape == (cap, d) and q.shape == (d,) and 1 <= window <= cap
    dt = 0 if q.dtype == np.float32 else 1
    assert Kc.dtype == Vc.dtype == q.dtype
    q, Kc, Vc = (np.ascontiguousarray(x) for x in (q, Kc, Vc))
    out = np.zeros(d, np.float64)
    lse = ctypes.c_double()
    pd = ctypes.POINTER(ctypes.c_double)
    _load().oracle_decode(int(cap), int(window), int(t), int(d), dt, q.ctypes.data,
                          Kc.ctypes.data, Vc.ctypes.data, float(scale), out.ctypes.data_as(pd),
                          ctypes.byref(lse))
    return out, lse.value


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a torch bf16 tensor (exact; no arithmetic)."""
    import torch
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
