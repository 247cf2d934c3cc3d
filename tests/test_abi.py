"""The C-ABI library, checked without a GPU: it loads, exports every function
that include/pagedattn.h declares, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_230_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    build.build()
    from paged_kv_cache_230_gb300 import pagedattn
    return pagedattn


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pagedattn.h")).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_calls(pa):
    assert declared_functions() == sorted(pa.EXPORTS)
    for name in ("pa_reshape_and_cache", "pa_decode", "pa_decode_split", "pa_decode_split_workspace_size"):
        assert name in declared_functions()


def test_library_exports_every_declared_symbol(pa):
    lib = ctypes.CDLL(build.LIB)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(pa.EXPORTS) == declared_functions()


def test_status_strings_and_version(pa):
    assert pa.status_string(0) == "ok"
    assert "workspace" in pa.status_string(-3)
    assert pa.status_string(-99) == "unknown status"
    assert pa.lib.pa_version() == 100


def test_workspace_size_formula(pa):
    # S * Hq * ceil(maxlen / P) * (D + 2) * 4
    assert pa.decode_split_workspace_size(8, 64, 128, 131072, 512) == 8 * 64 * 256 * 130 * 4
    assert pa.decode_split_workspace_size(3, 4, 64, 513, 512) == 3 * 4 * 2 * 66 * 4
    assert pa.decode_split_workspace_size(3, 4, 64, 0, 512) == 3 * 4 * 1 * 66 * 4
    assert pa.decode_split_workspace_size(3, 4, 64, 10, 0) == 0


def _desc(pa, NB=4, bs=16, Hkv=2, D=128, dt=1):
    return pa.CacheDesc(NB, bs, Hkv, D, dt)


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails its host checks first


def test_host_checks_return_codes_without_a_gpu(pa):
    L = pa.lib
    d = _desc(pa)
    null = ctypes.c_void_p(0)
    # null cache pointer
    assert L.pa_decode(FAKE, FAKE, 1, 1, 4, null, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 1.0, null) == -1
    # head_dim 96, block size 12, bad dtype: unsupported
    for bad in (_desc(pa, D=96), _desc(pa, bs=12), _desc(pa, dt=7)):
        assert L.pa_decode(FAKE, FAKE, 1, 1, 4, FAKE, FAKE, ctypes.byref(bad), FAKE, 4, FAKE, 0.1, 1.0, null) == -2
    # group of 256 query heads per kv head (above 128): unsupported; 5 % 2: invalid
    assert L.pa_decode(FAKE, FAKE, 1, 1, 512, FAKE, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 1.0, null) == -2
    # a group of 32 goes to the tensor-core kernel, which takes scale > 0
    assert L.pa_decode(FAKE, FAKE, 1, 1, 64, FAKE, FAKE, ctypes.byref(d), FAKE, 4, FAKE, -0.1, 1.0, null) == -1
    assert L.pa_decode(FAKE, FAKE, 1, 1, 5, FAKE, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 1.0, null) == -1
    # q dtype f16 with a bf16 cache
    assert L.pa_decode(FAKE, FAKE, 0, 1, 4, FAKE, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 1.0, null) == -2
    # kv_scale must be 1 for 16-bit caches, positive and finite for FP8
    assert L.pa_decode(FAKE, FAKE, 1, 1, 4, FAKE, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 0.5, null) == -1
    d8 = _desc(pa, dt=2)
    assert L.pa_decode(FAKE, FAKE, 1, 1, 4, FAKE, FAKE, ctypes.byref(d8), FAKE, 4, FAKE, 0.1, 0.0, null) == -1
    # misaligned cache
    odd = ctypes.c_void_p(0x1008)
    assert L.pa_decode(FAKE, FAKE, 1, 1, 4, odd, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 1.0, null) == -1
    # split: partition size not a multiple of 64; missing workspace
    assert L.pa_decode_split(FAKE, FAKE, 1, 1, 4, FAKE, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 1.0, 64, 100,
                             FAKE, 1 << 20, null) == -1
    assert L.pa_decode_split(FAKE, FAKE, 1, 1, 4, FAKE, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 1.0, 64, 64,
                             null, 0, null) == -3
    assert L.pa_decode_split(FAKE, FAKE, 1, 1, 4, FAKE, FAKE, ctypes.byref(d), FAKE, 4, FAKE, 0.1, 1.0, 64, 64,
                             FAKE, 16, null) == -3
    # scatter: f16 rows into a bf16 cache; negative token count
    assert L.pa_reshape_and_cache(FAKE, FAKE, 0, 1, FAKE, FAKE, ctypes.byref(d), FAKE, 1.0, null) == -2
    assert L.pa_reshape_and_cache(FAKE, FAKE, 1, -1, FAKE, FAKE, ctypes.byref(d), FAKE, 1.0, null) == -1
    # empty batches succeed without touching the device
    assert L.pa_decode(null, null, 1, 0, 4, FAKE, FAKE, ctypes.byref(d), null, 4, null, 0.1, 1.0, null) == 0
    assert L.pa_reshape_and_cache(null, null, 1, 0, FAKE, FAKE, ctypes.byref(d), null, 1.0, null) == 0
