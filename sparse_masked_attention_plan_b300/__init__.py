"""Block-sparse masked attention for B300 (sm_103a): Python binding of libspattn.so.

A thin ctypes layer over the C ABI declared in ``include/spattn.h``.  It only
marshals arguments (torch tensors -> device pointers, streams -> handles); every
step of the computation runs in the library's CUDA kernels.  If the library is
missing, importing the binding's functions raises: there is no fallback path.

    import torch, sparse_masked_attention_plan_b300 as sp
    plan = sp.Plan(T=32768, head_dim=128, causal=1, window=4096)
    o, lse = sp.fwd(plan, q, k, v, scale=128 ** -0.5)      # q, k, v: [B, H, T, d] bf16 cuda
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspattn.so")

OK, ERR_INVALID_SPEC, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_NULL, ERR_CUDA, ERR_TIMEOUT, \
    ERR_UNSUPPORTED = range(9)
BF16, FP32 = 0, 1

# Every symbol include/spattn.h declares.
EXPORTS = ("spattn_mask_validate", "spattn_plan_create", "spattn_plan_info",
           "spattn_plan_copy_tiles", "spattn_plan_copy_columns", "spattn_plan_copy_schedule",
           "spattn_plan_set_walk_counter", "spattn_plan_walk_count", "spattn_fwd",
           "spattn_bwd", "spattn_kv_append", "spattn_decode_workspace_bytes",
           "spattn_decode", "spattn_decode_append", "spattn_decode_check", "spattn_fwd_host",
           "spattn_fwd_static_scratch", "spattn_plan_set_wait_budget",
           "spattn_plan_test_wait_timeout", "spattn_plan_check_device", "spattn_plan_destroy",
           "spattn_last_error", "spattn_version")


class SpattnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"spattn status {status}: {msg}")
        self.status = status


class MaskSpec(ctypes.Structure):
    _fields_ = [("causal", ctypes.c_int32), ("window", ctypes.c_int64),
                ("radius", ctypes.c_int64), ("stride", ctypes.c_int64),
                ("stride_offset", ctypes.c_int64), ("n_global", ctypes.c_int32),
                ("global_pos", ctypes.POINTER(ctypes.c_int32)), ("dilation", ctypes.c_int64),
                ("rand_block", ctypes.c_int32), ("n_rand", ctypes.c_int64),
                ("rand_pairs", ctypes.POINTER(ctypes.c_int32))]


_lib = None
_lock = threading.Lock()
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_vp = ctypes.c_void_p


def lib():
    """The loaded libspattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with "
                                  "`python -m sparse_masked_attention_plan_b300.build_lib`")
            L = ctypes.CDLL(LIB_PATH)
            st = ctypes.c_int
            L.spattn_mask_validate.argtypes = [ctypes.POINTER(MaskSpec), ctypes.c_int64]
            L.spattn_plan_create.argtypes = [ctypes.POINTER(MaskSpec), ctypes.c_int64,
                                             ctypes.c_int32, _vp, ctypes.POINTER(_vp)]
            L.spattn_plan_info.argtypes = [_vp, _i64p, _i64p, _i64p, _i64p, _i32p, _i32p]
            L.spattn_plan_copy_tiles.argtypes = [_vp, _i32p, _i32p, _i32p, _u8p, ctypes.c_int64,
                                                 _i64p]
            L.spattn_plan_copy_columns.argtypes = [_vp, _i32p, ctypes.c_int64, _i64p]
            L.spattn_plan_copy_schedule.argtypes = [_vp, ctypes.c_int32, _i32p, ctypes.c_int64,
                                                    _i64p, _i32p, ctypes.c_int64, _i64p, _i64p]
            L.spattn_plan_set_walk_counter.argtypes = [_vp, ctypes.c_int32]
            L.spattn_plan_walk_count.argtypes = [_vp, _i64p]
            L.spattn_fwd.argtypes = [_vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int, _vp, _vp,
                                     _vp, ctypes.c_float, _vp, _vp, _vp]
            L.spattn_fwd_host.argtypes = [_vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int, _vp,
                                          _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp,
                                          _vp, _vp]
            L.spattn_fwd_static_scratch.argtypes = L.spattn_fwd.argtypes
            L.spattn_kv_append.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                           ctypes.c_int32, ctypes.c_int, _vp, _vp, _vp, _vp,
                                           _vp, _vp]
            L.spattn_decode_workspace_bytes.argtypes = [ctypes.c_int32, ctypes.c_int32,
                                                        ctypes.c_int32, ctypes.c_int64,
                                                        ctypes.c_int32,
                                                        ctypes.POINTER(ctypes.c_size_t)]
            L.spattn_decode.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_int, _vp, _vp, _vp, _vp, ctypes.c_float, _vp,
                                        _vp, _vp, ctypes.c_size_t, _vp]
            L.spattn_decode_append.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                               ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp,
                                               ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t,
                                               _vp]
            L.spattn_decode_check.argtypes = [_vp, _vp]
            L.spattn_bwd.argtypes = [_vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int, _vp,
                                     _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp,
                                     _vp]
            L.spattn_plan_set_wait_budget.argtypes = [_vp, ctypes.c_uint64]
            L.spattn_plan_test_wait_timeout.argtypes = [_vp, ctypes.c_int32]
            L.spattn_plan_check_device.argtypes = [_vp, _vp]
            L.spattn_plan_destroy.argtypes = [_vp]
            L.spattn_plan_destroy.restype = None
            L.spattn_last_error.restype = ctypes.c_char_p
            L.spattn_version.restype = ctypes.c_char_p
            for name in EXPORTS:
                if name not in ("spattn_plan_destroy", "spattn_last_error", "spattn_version"):
                    getattr(L, name).restype = st
            _lib = L
    return _lib


def _check(status: int):
    if status != OK:
        raise SpattnError(status, lib().spattn_last_error().decode())


def make_spec(causal=1, window=0, radius=-1, stride=0, offset=0, global_pos=(), dilation=1,
              rand_block=0, rand_pairs=()):
    """(MaskSpec, keepalive arrays) for the mask fields (see include/spattn.h).
    rand_pairs: (query block, key block) pairs of BigBird random blocks of size
    rand_block."""
    g = np.ascontiguousarray(np.asarray(global_pos, dtype=np.int32))
    r = np.ascontiguousarray(np.asarray(rand_pairs, dtype=np.int32).reshape(-1, 2))
    spec = MaskSpec(int(causal), int(window), int(radius), int(stride), int(offset), len(g),
                    g.ctypes.data_as(_i32p) if len(g) else None, int(dilation),
                    int(rand_block), len(r), r.ctypes.data_as(_i32p) if len(r) else None)
    return spec, (g, r)


def validate(T, **mask) -> int:
    """Host-only spec check: returns the status code (0 = valid)."""
    spec, _keep = make_spec(**mask)
    return lib().spattn_mask_validate(ctypes.byref(spec), int(T))


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """Block-sparse plan of one mask for sequence length T (owns device memory)."""

    def __init__(self, T, head_dim, causal=1, window=0, radius=-1, stride=0, offset=0,
                 global_pos=(), dilation=1, rand_block=0, rand_pairs=(), stream=None):
        self.T = int(T)
        self.head_dim = int(head_dim)
        self.mask = dict(causal=int(causal), window=int(window), radius=int(radius),
                         stride=int(stride), offset=int(offset),
                         global_pos=np.asarray(global_pos, dtype=np.int32),
                         dilation=int(dilation), rand_block=int(rand_block),
                         rand_pairs=np.asarray(rand_pairs, dtype=np.int32).reshape(-1, 2))
        spec, keep = make_spec(causal, window, radius, stride, offset, global_pos, dilation,
                               rand_block, rand_pairs)
        h = _vp()
        _check(lib().spattn_plan_create(ctypes.byref(spec), self.T, self.head_dim,
                                        _stream_handle(stream), ctypes.byref(h)))
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            lib().spattn_plan_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self) -> dict:
        v = [ctypes.c_int64() for _ in range(4)]
        bm, bn = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().spattn_plan_info(self._h, *[ctypes.byref(x) for x in v], ctypes.byref(bm),
                                      ctypes.byref(bn)))
        return dict(pairs_per_head=v[0].value, n_full=v[1].value, n_partial=v[2].value,
                    n_empty=v[3].value, bm=bm.value, bn=bn.value)

    def tiles(self):
        """(qb, kb, cnt, cls) of the non-empty tiles, canonical order."""
        n = ctypes.c_int64()
        lib().spattn_plan_copy_tiles(self._h, None, None, None, None, 0, ctypes.byref(n))
        k = n.value
        qb = np.zeros(k, np.int32)
        kb = np.zeros(k, np.int32)
        cnt = np.zeros(k, np.int32)
        cls = np.zeros(k, np.uint8)
        _check(lib().spattn_plan_copy_tiles(self._h, qb.ctypes.data_as(_i32p),
                                            kb.ctypes.data_as(_i32p), cnt.ctypes.data_as(_i32p),
                                            cls.ctypes.data_as(_u8p), k, ctypes.byref(n)))
        return qb, kb, cnt, cls

    def columns(self) -> np.ndarray:
        n = ctypes.c_int64()
        lib().spattn_plan_copy_columns(self._h, None, 0, ctypes.byref(n))
        out = np.zeros(n.value, np.int32)
        _check(lib().spattn_plan_copy_columns(self._h, out.ctypes.data_as(_i32p), n.value,
                                              ctypes.byref(n)))
        return out

    def schedule(self, which=0):
        """(items [n,4], entries [m,4], tile_products) of the execution schedule."""
        ni, ne, tp = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().spattn_plan_copy_schedule(self._h, int(which), None, 0, ctypes.byref(ni),
                                               None, 0, ctypes.byref(ne), ctypes.byref(tp)))
        items = np.zeros((ni.value, 4), np.int32)
        ents = np.zeros((ne.value, 4), np.int32)
        _check(lib().spattn_plan_copy_schedule(self._h, int(which), items.ctypes.data_as(_i32p),
                                               ni.value, ctypes.byref(ni),
                                               ents.ctypes.data_as(_i32p), ne.value,
                                               ctypes.byref(ne), ctypes.byref(tp)))
        return items, ents, tp.value

    def set_walk_counter(self, enable=True):
        _check(lib().spattn_plan_set_walk_counter(self._h, 1 if enable else 0))

    def walk_count(self) -> int:
        v = ctypes.c_int64()
        _check(lib().spattn_plan_walk_count(self._h, ctypes.byref(v)))
        return v.value

    def set_wait_budget(self, cycles: int):
        _check(lib().spattn_plan_set_wait_budget(self._h, int(cycles)))

    def test_wait_timeout(self, enable=True):
        _check(lib().spattn_plan_test_wait_timeout(self._h, 1 if enable else 0))

    def check_device(self, stream=None):
        _check(lib().spattn_plan_check_device(self._h, _stream_handle(stream)))


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def fwd(plan: Plan, q, k, v, scale: float, out=None, lse=None, stream=None, want_lse=True):
    """Forward pass on device tensors q, k, v: [B, H, T, d] (bf16 or fp32, contiguous).

    Returns (O, LSE); O has q's dtype, LSE is fp32 [B, H, T].  Asynchronous on
    `stream` (default: torch's current stream)."""
    import torch
    B, H, T, d = q.shape
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, H, T, d):
            raise ValueError("q, k, v must be contiguous CUDA tensors of equal shape")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    _check(lib().spattn_fwd(plan.handle, B, H, _dtype_code(q), q.data_ptr(), k.data_ptr(),
                            v.data_ptr(), float(scale), out.data_ptr(),
                            lse.data_ptr() if lse is not None else None,
                            _stream_handle(stream)))
    return out, lse


def bwd(plan: Plan, q, k, v, o, lse, do, scale: float, dq=None, dk=None, dv=None,
        stream=None):
    """Gradients (dQ, dK, dV) of the masked attention given dO, from the forward's
    inputs q, k, v, its output o and LSE (all [B, H, T, d] / [B, H, T] CUDA tensors,
    contiguous, o and do of q's dtype).  Asynchronous on `stream`."""
    import torch
    B, H, T, d = q.shape
    for t in (q, k, v, o, do):
        if (not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, H, T, d)
                or t.dtype != q.dtype):
            raise ValueError("q, k, v, o, do must be contiguous CUDA tensors of equal shape "
                             "and dtype")
    if (not lse.is_cuda or not lse.is_contiguous() or lse.dtype != torch.float32
            or tuple(lse.shape) != (B, H, T)):
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, H, T]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    _check(lib().spattn_bwd(plan.handle, B, H, _dtype_code(q), q.data_ptr(), k.data_ptr(),
                            v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                            float(scale), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                            _stream_handle(stream)))
    return dq, dk, dv


class DecodeCache:
    """A ring-buffer KV cache of one sliding-window layer and its decode workspace.

    K, V: [B, Hkv, cap, d] CUDA tensors (allocated here); position p lives in slot
    p % cap.  append() writes a step's keys/values, step() runs one decode step."""

    def __init__(self, B, Hq, Hkv, cap, head_dim, window=0, dtype=None, device="cuda"):
        import torch
        dtype = torch.bfloat16 if dtype is None else dtype
        self.B, self.Hq, self.Hkv, self.cap, self.d = B, Hq, Hkv, cap, head_dim
        self.window = window
        self.K = torch.zeros(B, Hkv, cap, head_dim, dtype=dtype, device=device)
        self.V = torch.zeros_like(self.K)
        n = ctypes.c_size_t()
        _check(lib().spattn_decode_workspace_bytes(B, Hq, Hkv, cap, head_dim, ctypes.byref(n)))
        self.workspace = torch.zeros(n.value, dtype=torch.uint8, device=device)

    def append(self, k_new, v_new, pos, stream=None):
        """k_new, v_new: [B, Hkv, d]; pos: [B] int64 CUDA tensor."""
        _check(lib().spattn_kv_append(self.B, self.Hkv, self.cap, self.d, _dtype_code(k_new),
                                      self.K.data_ptr(), self.V.data_ptr(), k_new.data_ptr(),
                                      v_new.data_ptr(), pos.data_ptr(), _stream_handle(stream)))

    def step(self, q, pos, scale, out=None, lse=None, stream=None):
        """q: [B, Hq, d]; pos: [B] int64 CUDA tensor.  Returns (out, lse)."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty(self.B, self.Hq, dtype=torch.float32, device=q.device)
        _check(lib().spattn_decode(self.B, self.Hq, self.Hkv, self.cap, self.window, self.d,
                                   _dtype_code(q), q.data_ptr(), self.K.data_ptr(),
                                   self.V.data_ptr(), pos.data_ptr(), float(scale),
                                   out.data_ptr(), lse.data_ptr(), self.workspace.data_ptr(),
                                   self.workspace.numel(), _stream_handle(stream)))
        return out, lse

    def append_step(self, k_new, v_new, q, pos, scale, out=None, lse=None, stream=None):
        """append(k_new, v_new, pos) then step(q, pos, scale) as one call
        (spattn_decode_append).  Returns (out, lse)."""
        import torch
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty(self.B, self.Hq, dtype=torch.float32, device=q.device)
        _check(lib().spattn_decode_append(
            self.B, self.Hq, self.Hkv, self.cap, self.window, self.d, _dtype_code(q),
            q.data_ptr(), self.K.data_ptr(), self.V.data_ptr(), k_new.data_ptr(),
            v_new.data_ptr(), pos.data_ptr(), float(scale), out.data_ptr(), lse.data_ptr(),
            self.workspace.data_ptr(), self.workspace.numel(), _stream_handle(stream)))
        return out, lse

    def check(self, stream=None):
        _check(lib().spattn_decode_check(self.workspace.data_ptr(), _stream_handle(stream)))


def fwd_static_scratch(plan: Plan, q, k, v, scale: float, out=None, lse=None, stream=None):
    """fwd() through spattn_fwd_static_scratch: the packing scratch comes from the
    library's fixed 16 MiB device array, so the call allocates no device memory
    (out / lse are allocated here only when not given)."""
    import torch
    B, H, T, d = q.shape
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, H, T, d):
            raise ValueError("q, k, v must be contiguous CUDA tensors of equal shape")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    _check(lib().spattn_fwd_static_scratch(plan.handle, B, H, _dtype_code(q), q.data_ptr(),
                                           k.data_ptr(), v.data_ptr(), float(scale),
                                           out.data_ptr(), lse.data_ptr(),
                                           _stream_handle(stream)))
    return out, lse


def fwd_host(plan: Plan, q_host, k_host, v_host, scale: float, o_host, lse_host, dev_bufs,
             stream=None):
    """End-to-end call from host tensors (pinned): copies in, computes, copies out.

    dev_bufs = (q_dev, k_dev, v_dev, o_dev, lse_dev) preallocated on the device."""
    B, H, T, d = q_host.shape
    qd, kd, vd, od, ld = dev_bufs
    _check(lib().spattn_fwd_host(plan.handle, B, H, _dtype_code(q_host), q_host.data_ptr(),
                                 k_host.data_ptr(), v_host.data_ptr(), float(scale),
                                 o_host.data_ptr(),
                                 lse_host.data_ptr() if lse_host is not None else None,
                                 qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(),
                                 ld.data_ptr() if ld is not None else None,
                                 _stream_handle(stream)))
    return o_host, lse_host
