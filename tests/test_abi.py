"""The C-ABI library builds, loads and exports every symbol the header declares;
host-side spec validation agrees with the oracle's reading of the mask domain.
No compute call here: these run without a GPU."""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import sparse_masked_attention_plan_b300 as sp
from sparse_masked_attention_plan_b300 import build_lib
from pins import small_specs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spattn.h")


@pytest.fixture(scope="module")
def built():
    build_lib.build()
    return sp.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spattn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(sp.EXPORTS)


def test_library_exports_every_declared_symbol(built):
    out = subprocess.run(["nm", "-D", "--defined-only", sp.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (spattn_\w+)", out))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, f"not exported: {missing}"
    for f in declared_functions():
        assert hasattr(built, f)


def test_library_is_sm_103a_only(built):
    out = subprocess.run(["/usr/local/cuda/bin/cuobjdump", "--list-elf", sp.LIB_PATH],
                         capture_output=True, text=True).stdout
    archs = set(re.findall(r"sm_\d+a?", out))
    assert archs == {"sm_103a"}, archs


def test_version(built):
    assert b"sm_103a" in built.spattn_version()


@pytest.mark.parametrize("seed", [0, 1])
def test_validate_accepts_what_the_oracle_accepts(oracle_mod, built, seed):
    for e in small_specs(seed, n=60):
        m = oracle.Mask(e["T"], e["causal"], e["window"], e["radius"], e["stride"],
                        e["offset"], e["global_pos"], e["dilation"], e.get("rand_block", 0),
                        e.get("rand_pairs", ()))
        assert m.validate() == 0
        st = sp.validate(e["T"], causal=e["causal"], window=e["window"], radius=e["radius"],
                         stride=e["stride"], offset=e["offset"], global_pos=e["global_pos"],
                         dilation=e["dilation"], rand_block=e.get("rand_block", 0),
                         rand_pairs=e.get("rand_pairs", ()))
        assert st == sp.OK, (e, built.spattn_last_error())


INVALID = [
    dict(T=0), dict(T=8, causal=2), dict(T=8, causal=1, window=-1),
    dict(T=8, causal=1, radius=2), dict(T=8, causal=0, radius=-2),
    dict(T=8, causal=0, window=3, radius=1), dict(T=8, stride=-1),
    dict(T=8, stride=4, offset=4), dict(T=8, stride=0, offset=1),
    dict(T=8, global_pos=[8]), dict(T=8, global_pos=[-1]), dict(T=8, global_pos=[3, 3]),
    dict(T=8, dilation=-1),
    dict(T=40, causal=0, radius=2, rand_block=48, rand_pairs=[(0, 0)]),
    dict(T=40, causal=0, radius=2, rand_block=16, rand_pairs=[(0, 3)]),
    dict(T=40, causal=0, radius=2, rand_block=16, rand_pairs=[(0, 1), (0, 1)]),
    dict(T=40, causal=0, radius=2, rand_block=16, rand_pairs=[(-1, 0)]),
]


@pytest.mark.parametrize("case", INVALID, ids=[str(c) for c in INVALID])
def test_validate_rejects_what_the_oracle_rejects(oracle_mod, built, case):
    c = dict(causal=1, window=0, radius=-1, stride=0, offset=0, global_pos=[], dilation=1,
             rand_block=0, rand_pairs=[])
    c.update(case)
    T = c.pop("T")
    m = oracle.Mask(T, c["causal"], c["window"], c["radius"], c["stride"], c["offset"],
                    c["global_pos"], c["dilation"], c["rand_block"], c["rand_pairs"])
    assert m.validate() != 0
    assert sp.validate(T, **c) != sp.OK


def test_validate_accepts_unsorted_globals(built):
    assert sp.validate(10, causal=0, radius=1, global_pos=[7, 2, 5]) == sp.OK


def test_plan_create_rejects_bad_head_dim_without_gpu(built):
    spec, _keep = sp.make_spec(causal=1, window=4)
    import ctypes
    h = ctypes.c_void_p()
    st = built.spattn_plan_create(ctypes.byref(spec), 64, 96, None, ctypes.byref(h))
    assert st == sp.ERR_SHAPE and not h.value


def test_null_arguments_are_rejected(built):
    import ctypes
    assert built.spattn_mask_validate(None, 16) == sp.ERR_NULL
    assert built.spattn_plan_info(None, None, None, None, None, None, None) == sp.ERR_NULL
    assert built.spattn_fwd(None, 1, 1, 0, None, None, None, 1.0, None, None,
                            None) == sp.ERR_NULL
    built.spattn_plan_destroy(None)
    assert built.spattn_last_error()


def test_decode_workspace_bytes_without_gpu(built):
    """The workspace holds a 256-byte header (error word) and one (d + 2)-float partial per
    (batch, query head, split); the split count keeps B * Hkv * splits within 2 * 148
    CTAs, at most 64 splits and one 64-slot sub-chunk per split at least."""
    import ctypes
    n = ctypes.c_size_t()

    def ws(B, Hq, Hkv, cap, d):
        assert built.spattn_decode_workspace_bytes(B, Hq, Hkv, cap, d, ctypes.byref(n)) == sp.OK
        return n.value

    def expect(B, Hq, Hkv, cap, d, splits):
        return 256 + B * Hq * splits * (d + 2) * 4

    assert ws(8, 32, 8, 4096, 128) == expect(8, 32, 8, 4096, 128, 4)      # 296 // 64
    assert ws(32, 32, 8, 4096, 128) == expect(32, 32, 8, 4096, 128, 1)    # 296 // 256
    assert ws(64, 32, 8, 4096, 128) == expect(64, 32, 8, 4096, 128, 1)    # never below 1
    assert ws(1, 8, 1, 100000, 64) == expect(1, 8, 1, 100000, 64, 64)     # at most 64
    assert ws(1, 8, 2, 100, 64) == expect(1, 8, 2, 100, 64, 2)            # ceil(100 / 64)
    assert built.spattn_decode_workspace_bytes(1, 8, 3, 100, 64, ctypes.byref(n)) == sp.ERR_SHAPE
    assert built.spattn_decode_workspace_bytes(1, 8, 2, 100, 64, None) == sp.ERR_NULL
