"""ctypes front end of the C oracle in ``oracle.c``.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The functions take the
library's layouts as numpy arrays of raw bit patterns (uint16 for f16/bf16,
uint8 for E4M3) and return fp64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, E4M3 = 0, 1, 2
_CODES = {"f16": F16, "bf16": BF16, "fp8": E4M3, F16: F16, BF16: BF16, E4M3: E4M3}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles oracle.c with gcc (IEEE arithmetic, no FMA contraction, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float
            L.orc_init.restype = None
            L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_double.restype = f64
            L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_double.restype = f64
            L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_to_double.restype = f64
            L.orc_float_to_e4m3.argtypes = [f32]
            L.orc_float_to_e4m3.restype = ctypes.c_uint8
            L.orc_double_to_f16.argtypes = [f64]
            L.orc_double_to_f16.restype = ctypes.c_uint16
            L.orc_double_to_bf16.argtypes = [f64]
            L.orc_double_to_bf16.restype = ctypes.c_uint16
            L.orc_reshape_and_cache.argtypes = [P, P, i32, i64, i32, i32, P, P, i32, i64, i32, P, f32]
            L.orc_reshape_and_cache.restype = i64
            L.orc_decode.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, i32, i64, i32, P, i32, P,
                                     f64, f64, i32, i32]
            L.orc_decode.restype = i32
            L.orc_attend_range.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, i32, i64, i32, P,
                                           i32, f64, f64, i32, i32, i32, i32]
            L.orc_attend_range.restype = None
            L.orc_decode16_array.argtypes = [P, P, i64, i32]
            L.orc_e4m3_decode_array.argtypes = [P, P, i64]
            L.orc_e4m3_encode_array.argtypes = [P, P, i64]
            L.orc_round_array.argtypes = [P, P, i64, i32]
            L.orc_max_threads.restype = i32
            for fn in ("orc_copy_blocks",):
                getattr(L, fn).argtypes = [P, P, i64, P, i64, i64]
                getattr(L, fn).restype = i64
            L.orc_gather_blocks.argtypes = [P, P, P, i64, P, i64, i64]
            L.orc_gather_blocks.restype = i64
            L.orc_scatter_blocks.argtypes = [P, P, P, i64, P, i64, i64]
            L.orc_scatter_blocks.restype = i64
            L.orc_init()
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(lib().orc_max_threads())


def f16_to_double(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().orc_decode16_array(_ptr(b), _ptr(out), b.size, F16)
    return out


def bf16_to_double(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().orc_decode16_array(_ptr(b), _ptr(out), b.size, BF16)
    return out


def decode16(bits, dtype) -> np.ndarray:
    return f16_to_double(bits) if _CODES[dtype] == F16 else bf16_to_double(bits)


def e4m3_to_double(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def float_to_e4m3(y) -> np.ndarray:
    v = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def round_out(x, dtype) -> np.ndarray:
    """Round fp64 results to f16/bf16 bit patterns (nearest, ties to even)."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_round_array(_ptr(v), _ptr(out), v.size, _CODES[dtype])
    return out


def reshape_and_cache(key, value, in_dtype, k_cache, v_cache, cache_dtype, slot_mapping,
                      kv_scale: float = 1.0) -> int:
    """Scatter in place into ``k_cache``/``v_cache`` ([NB, Hkv, bs, D]).
    Returns the number of tokens skipped because their slot is outside the pool."""
    key = np.ascontiguousarray(key, dtype=np.uint16)
    value = np.ascontiguousarray(value, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = key.shape
    NB, Hc, bs, Dc = k_cache.shape
    assert (Hc, Dc) == (Hkv, D) and v_cache.shape == k_cache.shape and len(slots) == T
    want = np.uint8 if _CODES[cache_dtype] == E4M3 else np.uint16
    assert k_cache.dtype == want and v_cache.dtype == want
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    return int(lib().orc_reshape_and_cache(_ptr(key), _ptr(value), _CODES[in_dtype], T, Hkv, D,
                                           _ptr(k_cache), _ptr(v_cache), _CODES[cache_dtype], NB, bs,
                                           _ptr(slots), ctypes.c_float(kv_scale)))


def decode(q, q_dtype, k_cache, v_cache, cache_dtype, block_tables, context_lens, scale,
           kv_scale: float = 1.0, partition_size: int = 0, num_threads: int | None = None) -> np.ndarray:
    """fp64 decode attention ``[S, Hq, D]``; ``partition_size > 0`` gives the split variant."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, Hq, D = q.shape
    NB, Hkv, bs, Dc = k_cache.shape
    assert Dc == D and Hq % Hkv == 0 and bt.shape[0] == S and cl.shape == (S,)
    out = np.empty((S, Hq, D), np.float64)
    nt = max_threads() if num_threads is None else int(num_threads)
    rc = lib().orc_decode(_ptr(out), _ptr(q), _CODES[q_dtype], S, Hq, Hkv, D,
                          _ptr(np.ascontiguousarray(k_cache)), _ptr(np.ascontiguousarray(v_cache)),
                          _CODES[cache_dtype], NB, bs, _ptr(bt), bt.shape[1], _ptr(cl),
                          float(scale), float(kv_scale), int(partition_size), nt)
    if rc != 0:
        raise ValueError("oracle: context length or block id out of range")
    return out


def attend_range(q, q_dtype, k_cache, v_cache, cache_dtype, block_tables, scale, kv_scale, s, g, t0, t1):
    """Partial (m, l, o) of query head g of sequence s over tokens [t0, t1)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    S, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    m = ctypes.c_double()
    l = ctypes.c_double()
    o = np.empty(D, np.float64)
    lib().orc_attend_range(ctypes.byref(m), ctypes.byref(l), _ptr(o), _ptr(q), _CODES[q_dtype], Hq,
                           Hkv, D, _ptr(np.ascontiguousarray(k_cache)), _ptr(np.ascontiguousarray(v_cache)),
                           _CODES[cache_dtype], NB, bs, _ptr(bt), bt.shape[1], float(scale),
                           float(kv_scale), int(s), int(g), int(t0), int(t1))
    return m.value, l.value, o


def _block_bytes(cache):
    return int(cache[0].nbytes)


def copy_blocks(k_cache, v_cache, pairs) -> int:
    """In place: cache[dst] = cache[src] for each (src, dst) row, in order."""
    pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    return int(lib().orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), _block_bytes(k_cache), _ptr(pairs),
                                     len(pairs), k_cache.shape[0]))


def gather_blocks(k_cache, v_cache, ids) -> np.ndarray:
    """[n, 2, *block] buffer of the named blocks (K then V)."""
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    buf = np.zeros((len(ids), 2) + k_cache.shape[1:], k_cache.dtype)
    lib().orc_gather_blocks(_ptr(buf), _ptr(k_cache), _ptr(v_cache), _block_bytes(k_cache), _ptr(ids), len(ids),
                            k_cache.shape[0])
    return buf


def scatter_blocks(k_cache, v_cache, buf, ids) -> int:
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    buf = np.ascontiguousarray(buf)
    return int(lib().orc_scatter_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(buf), _block_bytes(k_cache), _ptr(ids),
                                        len(ids), k_cache.shape[0]))
