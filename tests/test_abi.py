"""The C-ABI library builds, loads and exports every symbol include/int8kv.h
declares; host-side validation needs no GPU (CPU only)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from int8_kv_cache_02_gb300 import binding, build
    build.build()
    return binding.lib()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                                txt, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    assert "attn_decode_int8" in names and "kv_quant_append" in names and "kv_pool_create" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_status_strings(L):
    from int8_kv_cache_02_gb300 import binding
    assert binding.int8kv_status_string(0) == "ok"
    for s in range(-1, -10, -1):
        assert binding.int8kv_status_string(s) != "unknown status"


def test_region_bytes_match_the_528_byte_cell(L):
    """One page (64 positions) of a k8v8 pool, 2 kv heads, head_dim 256, 64-value
    groups: (K codes + K scales) / 64 = 528 B per cell (Strata #2698)."""
    from int8_kv_cache_02_gb300 import binding as b
    codes = b.int8kv_pool_region_bytes(1, 2, 256, 64, 64, 1, b.K8V8, 0)
    scales = b.int8kv_pool_region_bytes(1, 2, 256, 64, 64, 1, b.K8V8, 2)
    assert (codes + scales) // 64 == 528
    assert b.int8kv_pool_region_bytes(1, 2, 256, 64, 64, 1, b.K8V16, 3) == 0
    assert b.int8kv_pool_region_bytes(1, 2, 256, 64, 64, 1, b.K8V16, 1) == 64 * 2 * 256 * 2


@pytest.mark.parametrize("args,status", [
    ((1, 2, 256, 48, 64, 1, 0, 0), -4),    # group does not divide head_dim
    ((1, 2, 256, 4, 64, 1, 0, 0), -4),     # group below head_dim / 32
    ((1, 2, 96, 32, 64, 1, 0, 0), -6),     # head_dim not built
    ((1, 2, 128, 128, 48, 1, 0, 0), -6),   # page size not built
    ((0, 2, 128, 128, 64, 1, 0, 0), -1),
    ((1, 2, 128, 128, 64, 1, 7, 0), -1),   # unknown variant
    ((1, 2, 128, 128, 64, 1, 0, 9), -1),   # unknown region
])
def test_region_bytes_validation(L, args, status):
    out = ctypes.c_size_t(0)
    assert L.int8kv_pool_region_bytes(*args, ctypes.byref(out)) == status


def test_pool_create_validation_without_device(L):
    h = ctypes.c_void_p()
    a16 = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    # NULL store / missing scales for an int8 store
    assert L.kv_pool_create(ctypes.byref(h), 1, 2, 128, 128, 64, 4, 0, None, a16, a16, a16, None) == -2
    assert L.kv_pool_create(ctypes.byref(h), 1, 2, 128, 128, 64, 4, 0, a16, a16, None, a16, None) == -2
    # scales given for an fp16 store
    assert L.kv_pool_create(ctypes.byref(h), 1, 2, 128, 128, 64, 4, 1, a16, a16, a16, a16, None) == -1
    # misaligned region
    assert L.kv_pool_create(ctypes.byref(h), 1, 2, 128, 128, 64, 4, 0, odd, a16, a16, a16, None) == -3
    assert L.kv_pool_create(None, 1, 2, 128, 128, 64, 4, 0, a16, a16, a16, a16, None) == -2


def test_decode_and_append_reject_null_pool(L):
    assert L.attn_decode_int8(None, 0, None, 1, 8, None, None, 1, 0, ctypes.c_float(0), 0, None,
                              None, 0, None) == -2
    assert L.kv_quant_append(None, 0, None, None, 1, 1, None, None, 1, None) == -2
    assert L.attn_decode_multi_int8(None, 0, None, 1, 2, 8, None, None, 1, ctypes.c_float(0), 0,
                                    None, None, 0, None) == -2


def test_workspace_bytes(L):
    from int8_kv_cache_02_gb300 import binding as b
    assert b.attn_decode_workspace_bytes(1, 16, 2, 256, 1) == 0
    n = b.attn_decode_workspace_bytes(1, 16, 2, 256, 4)
    assert n >= 16 * 4 * 256 * 4 + 16 * 4 * 8 and n % 256 == 0
    out = ctypes.c_size_t(0)
    assert L.attn_decode_workspace_bytes(1, 16, 2, 256, 0, ctypes.byref(out)) == -1
    assert L.attn_decode_workspace_bytes(1, 16, 2, 256, 100000, ctypes.byref(out)) == -1


def test_pool_image_calls_reject_null_arguments(L):
    out = ctypes.c_size_t(0)
    assert L.kv_pool_image_bytes(None, 1, None, ctypes.byref(out)) == -2
    assert L.kv_pool_save(None, 1, None, None, 1, None, 0, None, 0, None) == -2
    assert L.kv_pool_load(None, None, 0, 1, None, 1, None, 0, None, None) == -2
    from int8_kv_cache_02_gb300 import binding as b
    assert b.int8kv_status_string(-9).startswith("pool image")


def test_k8v4_region_bytes(L):
    """k8v4: K int8 codes + fp16 scales per group; V two 4-bit codes per byte and one
    fp16 scale per 32 values (head_dim 256, 2 kv heads: 512 + 16 B of K and
    256 + 32 B of V per position)."""
    from int8_kv_cache_02_gb300 import binding as b
    r = [b.int8kv_pool_region_bytes(1, 2, 256, 64, 64, 1, b.K8V4, k) for k in range(4)]
    assert r == [64 * 512, 64 * 256, 64 * 16, 64 * 32]
    a16 = ctypes.c_void_p(0x10000)
    h = ctypes.c_void_p()
    # the 4-bit store needs its scales
    assert L.kv_pool_create(ctypes.byref(h), 1, 2, 256, 64, 64, 4, 3, a16, a16, a16, None, None) == -2


def test_q4_0_region_bytes(L):
    """q4_0: K and V both two 4-bit codes per byte and one fp16 scale per 32 values
    (head_dim 128, 2 kv heads: 128 + 16 B per store and position); both scales
    regions are required."""
    from int8_kv_cache_02_gb300 import binding as b
    r = [b.int8kv_pool_region_bytes(1, 2, 128, 128, 64, 1, b.Q4_0, k) for k in range(4)]
    assert r == [64 * 128, 64 * 128, 64 * 16, 64 * 16]
    a16 = ctypes.c_void_p(0x10000)
    h = ctypes.c_void_p()
    assert L.kv_pool_create(ctypes.byref(h), 1, 2, 128, 128, 64, 4, 4, a16, a16, None, a16, None) == -2
    assert L.kv_pool_create(ctypes.byref(h), 1, 2, 128, 128, 64, 4, 4, a16, a16, a16, None, None) == -2
    assert L.kv_pool_create(ctypes.byref(h), 1, 2, 128, 128, 64, 4, 5, a16, a16, a16, a16, None) == -1
