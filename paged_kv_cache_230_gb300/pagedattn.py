"""Python binding of libpagedattn.so (ctypes; argument marshalling only).

Every function here checks tensor devices, dtypes, shapes and contiguity,
then passes raw device pointers and the current CUDA stream to the C ABI
declared in ``include/pagedattn.h``.  All arithmetic runs in the library's
kernels; there is no fallback.  Importing this module loads the library and
raises if it has not been built (``paged_kv_cache_230_gb300.build.build()``).

Tensor conventions (torch, on the GPU):
  q, out              [S, Hq, D]  float16 or bfloat16
  key, value          [T, Hkv, D] float16 or bfloat16
  k_cache, v_cache    [NB, Hkv, bs, D] float16 / bfloat16, or uint8 /
                      float8_e4m3fn holding OCP E4M3 codes
  block_tables        int32 [S, max_blocks_per_seq]
  context_lens        int32 [S]
  slot_mapping        int64 [T]
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported configuration", -3: "workspace",
          -4: "CUDA error", -5: "out-of-range index seen by a kernel", -6: "pipeline wait timed out",
          -7: "not enough free blocks", -8: "unknown or duplicate sequence id"}
DEVERR_BLOCK_ID, DEVERR_CONTEXT_LEN, DEVERR_SLOT, DEVERR_TIMEOUT, DEVERR_LAYOUT = 0x1, 0x2, 0x4, 0x8, 0x10
EXPORTS = ["pa_reshape_and_cache", "pa_decode", "pa_decode_multi", "pa_prefill", "pa_prefill_workspace_size",
           "pa_decode_split_workspace_size",
           "pa_decode_split", "pa_decode_multi_split_workspace_size", "pa_decode_multi_split", "pa_cache_and_decode",
           "pa_decode_split_noalloc", "pa_copy_blocks", "pa_gather_blocks", "pa_scatter_blocks",
           "pa_bm_create", "pa_bm_destroy", "pa_bm_add_sequence", "pa_bm_fork", "pa_bm_append_tokens",
           "pa_bm_free_sequence", "pa_bm_block_table", "pa_bm_num_free_blocks", "pa_bm_refcount",
           "pa_bm_tail_waste", "pa_bm_check", "pa_status_string", "pa_set_check_mode", "pa_get_device_error",
           "pa_selftest_wait_timeout", "pa_probe_l2_read", "pa_version"]


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__("%s failed: %s (%d)" % (fn, STATUS.get(status, "unknown"), status))
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError("libpagedattn.so is not built (%s); run paged_kv_cache_230_gb300.build.build()" % path)
    lib = ctypes.CDLL(path)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.pa_reshape_and_cache.argtypes = [P, P, i32, i32, P, P, ctypes.POINTER(CacheDesc), P, f32, P]
    lib.pa_decode.argtypes = [P, P, i32, i32, i32, P, P, ctypes.POINTER(CacheDesc), P, i32, P, f32, f32, P]
    lib.pa_decode_multi.argtypes = [P, P, i32, i32, i32, i32, P, P, ctypes.POINTER(CacheDesc), P, i32, P, f32, f32,
                                    P]
    lib.pa_prefill.argtypes = [P, P, i32, i32, i32, i32, P, P, ctypes.POINTER(CacheDesc), P, i32, P, f32, f32, P,
                               ctypes.c_size_t, P]
    lib.pa_prefill_workspace_size.argtypes = [i32, i32, ctypes.POINTER(CacheDesc)]
    lib.pa_prefill_workspace_size.restype = ctypes.c_size_t
    lib.pa_prefill.restype = ctypes.c_int
    lib.pa_decode_split_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.pa_decode_split_workspace_size.restype = ctypes.c_size_t
    lib.pa_decode_split.argtypes = [P, P, i32, i32, i32, P, P, ctypes.POINTER(CacheDesc), P, i32, P, f32, f32,
                                    i32, i32, P, ctypes.c_size_t, P]
    lib.pa_decode_multi_split_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.pa_decode_multi_split_workspace_size.restype = ctypes.c_size_t
    lib.pa_decode_multi_split.argtypes = [P, P, i32, i32, i32, i32, P, P, ctypes.POINTER(CacheDesc), P, i32, P, f32,
                                          f32, i32, i32, P, ctypes.c_size_t, P]
    lib.pa_cache_and_decode.argtypes = [P, P, i32, i32, i32, i32, P, P, P, P, P, ctypes.POINTER(CacheDesc), P, i32, P,
                                        f32, f32, i32, i32, P, ctypes.c_size_t, P]
    lib.pa_decode_split_noalloc.argtypes = [P, P, i32, i32, i32, P, P, ctypes.POINTER(CacheDesc), P, i32, P, f32,
                                            f32, i32, i32, P]
    D = ctypes.POINTER(CacheDesc)
    lib.pa_copy_blocks.argtypes = [P, P, D, P, i32, P]
    lib.pa_gather_blocks.argtypes = [P, P, P, D, P, i32, P]
    lib.pa_scatter_blocks.argtypes = [P, P, D, P, P, i32, P]
    lib.pa_bm_create.argtypes = [i64, i32]
    lib.pa_bm_create.restype = P
    lib.pa_bm_destroy.argtypes = [P]
    lib.pa_bm_destroy.restype = None
    lib.pa_bm_add_sequence.argtypes = [P, i64, i64]
    lib.pa_bm_fork.argtypes = [P, i64, i64]
    lib.pa_bm_append_tokens.argtypes = [P, i64, i32, P, P, P]
    lib.pa_bm_free_sequence.argtypes = [P, i64]
    lib.pa_bm_block_table.argtypes = [P, i64, P, i32, P, P]
    lib.pa_bm_num_free_blocks.argtypes = [P]
    lib.pa_bm_num_free_blocks.restype = i64
    lib.pa_bm_refcount.argtypes = [P, i64]
    lib.pa_bm_refcount.restype = i32
    lib.pa_bm_tail_waste.argtypes = [P]
    lib.pa_bm_tail_waste.restype = i64
    lib.pa_bm_check.argtypes = [P]
    lib.pa_bm_check.restype = i64
    for name in ("pa_copy_blocks", "pa_gather_blocks", "pa_scatter_blocks", "pa_bm_add_sequence", "pa_bm_fork",
                 "pa_bm_append_tokens", "pa_bm_free_sequence", "pa_bm_block_table"):
        getattr(lib, name).restype = ctypes.c_int
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_set_check_mode.argtypes = [ctypes.c_int]
    lib.pa_get_device_error.argtypes = []
    lib.pa_selftest_wait_timeout.argtypes = [ctypes.c_void_p]
    lib.pa_probe_l2_read.argtypes = [P, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int32, P,
                                     ctypes.POINTER(ctypes.c_ulonglong), P]
    lib.pa_version.argtypes = []
    for name in ("pa_reshape_and_cache", "pa_decode", "pa_decode_multi", "pa_decode_split", "pa_decode_multi_split",
                 "pa_cache_and_decode",
                 "pa_decode_split_noalloc",
                 "pa_set_check_mode",
                 "pa_get_device_error", "pa_selftest_wait_timeout", "pa_probe_l2_read", "pa_version"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


lib = _load()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float16:
        return PA_F16
    if t == torch.bfloat16:
        return PA_BF16
    if t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return PA_FP8_E4M3
    raise TypeError("unsupported dtype %s" % t)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise PagedAttnError(fn, rc)


def _need(t: torch.Tensor, name: str, dtype=None, ndim=None, device=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError("%s has dtype %s" % (name, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    NB, Hkv, bs, D = k_cache.shape
    return CacheDesc(NB, bs, Hkv, D, _dtype_code(k_cache.dtype))


def _check_caches(k_cache, v_cache):
    _need(k_cache, "k_cache", ndim=4)
    _need(v_cache, "v_cache", ndim=4, device=k_cache.device)
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must match")


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, kv_scale: float = 1.0) -> None:
    """Writes key/value rows [T, Hkv, D] into the cache slots named by slot_mapping."""
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(key, "key", (torch.float16, torch.bfloat16), 3, dev)
    _need(value, "value", key.dtype, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    T = key.shape[0]
    if value.shape != key.shape or slot_mapping.shape[0] != T:
        raise ValueError("key/value/slot_mapping shapes disagree")
    if key.shape[1] != k_cache.shape[1] or key.shape[2] != k_cache.shape[3]:
        raise ValueError("key rows do not match the cache's heads/head_dim")
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_reshape_and_cache(_ptr(key), _ptr(value), _dtype_code(key.dtype), T, _ptr(k_cache),
                                      _ptr(v_cache), ctypes.byref(desc), _ptr(slot_mapping), float(kv_scale),
                                      _stream(dev))
    _check("pa_reshape_and_cache", rc)


def _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens):
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", (torch.float16, torch.bfloat16), 3, dev)
    _need(out, "out", q.dtype, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    S = q.shape[0]
    if out.shape != q.shape or block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("q/out/block_tables/context_lens shapes disagree")
    if q.shape[2] != k_cache.shape[3]:
        raise ValueError("head_dim of q and cache differ")
    return dev


def decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, kv_scale: float = 1.0) -> None:
    """Paged decode attention, one CTA per (sequence, kv head); writes out [S, Hq, D]."""
    dev = _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens)
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_decode(_ptr(out), _ptr(q), _dtype_code(q.dtype), q.shape[0], q.shape[1], _ptr(k_cache),
                           _ptr(v_cache), ctypes.byref(desc), _ptr(block_tables), block_tables.shape[1],
                           _ptr(context_lens), float(scale), float(kv_scale), _stream(dev))
    _check("pa_decode", rc)


def decode_multi(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, kv_scale: float = 1.0) -> None:
    """Decode of k new tokens per sequence, q/out [S, k, Hq, D], causal within the new tokens."""
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", (torch.float16, torch.bfloat16), 4, dev)
    _need(out, "out", q.dtype, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    S, k, Hq, D = q.shape
    if out.shape != q.shape or block_tables.shape[0] != S or context_lens.shape[0] != S or D != k_cache.shape[3]:
        raise ValueError("q/out/block_tables/context_lens shapes disagree")
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_decode_multi(_ptr(out), _ptr(q), _dtype_code(q.dtype), S, k, Hq, _ptr(k_cache), _ptr(v_cache),
                                 ctypes.byref(desc), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                 float(scale), float(kv_scale), _stream(dev))
    _check("pa_decode_multi", rc)


def prefill_workspace_size(num_seqs: int, max_blocks_per_seq: int, k_cache: torch.Tensor) -> int:
    """Bytes of the workspace prefill uses with E4M3 caches (0 for 16-bit caches)."""
    desc = cache_desc(k_cache)
    return int(lib.pa_prefill_workspace_size(num_seqs, max_blocks_per_seq, ctypes.byref(desc)))


def prefill(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
            block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, kv_scale: float = 1.0,
            workspace: Optional[torch.Tensor] = None, widen: bool = True) -> None:
    """Chunked prefill on the tensor cores: q/out [S, C, Hq, D] (D 64 or 128), causal over the paged context.
    With E4M3 caches ``workspace`` (uint8, at least prefill_workspace_size bytes) holds the widened blocks;
    it is allocated with torch when not given.  ``widen=False`` passes no workspace (the packed-group
    kernel, which widens E4M3 tiles in shared memory)."""
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", (torch.float16, torch.bfloat16), 4, dev)
    _need(out, "out", q.dtype, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    S, C, Hq, D = q.shape
    if out.shape != q.shape or block_tables.shape[0] != S or context_lens.shape[0] != S or D != k_cache.shape[3]:
        raise ValueError("q/out/block_tables/context_lens shapes disagree")
    desc = cache_desc(k_cache)
    need = prefill_workspace_size(S, block_tables.shape[1], k_cache) if widen else 0
    if not widen:
        workspace = None
    elif workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", device=dev)
    with torch.cuda.device(dev):
        rc = lib.pa_prefill(_ptr(out), _ptr(q), _dtype_code(q.dtype), S, C, Hq, _ptr(k_cache), _ptr(v_cache),
                            ctypes.byref(desc), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                            float(scale), float(kv_scale), None if workspace is None else _ptr(workspace),
                            0 if workspace is None else workspace.numel() * workspace.element_size(), _stream(dev))
    _check("pa_prefill", rc)


def decode_split_workspace_size(num_seqs: int, num_q_heads: int, head_dim: int, max_context_len: int,
                                partition_size: int) -> int:
    return int(lib.pa_decode_split_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len,
                                                  partition_size))


def decode_split(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, kv_scale: float,
                 max_context_len: int, partition_size: int = 512,
                 workspace: Optional[torch.Tensor] = None) -> None:
    """Split-context decode: per-partition partials merged by log-sum-exp.
    ``workspace`` (uint8, at least decode_split_workspace_size bytes) is
    allocated with torch when not given."""
    dev = _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens)
    need = decode_split_workspace_size(q.shape[0], q.shape[1], q.shape[2], max_context_len, partition_size)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", device=dev)
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_decode_split(_ptr(out), _ptr(q), _dtype_code(q.dtype), q.shape[0], q.shape[1],
                                 _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(block_tables),
                                 block_tables.shape[1], _ptr(context_lens), float(scale), float(kv_scale),
                                 int(max_context_len), int(partition_size), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(dev))
    _check("pa_decode_split", rc)


def decode_multi_split_workspace_size(num_seqs: int, num_q_tokens: int, num_q_heads: int, head_dim: int,
                                      max_context_len: int, partition_size: int) -> int:
    return int(lib.pa_decode_multi_split_workspace_size(num_seqs, num_q_tokens, num_q_heads, head_dim,
                                                        max_context_len, partition_size))


def decode_multi_split(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, kv_scale: float,
                       max_context_len: int, partition_size: int = 512,
                       workspace: Optional[torch.Tensor] = None) -> None:
    """Multi-token decode (q/out [S, k, Hq, D]) split into partitions merged by
    log-sum-exp.  ``workspace`` (uint8, at least
    decode_multi_split_workspace_size bytes) is allocated with torch when not
    given."""
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", (torch.float16, torch.bfloat16), 4, dev)
    _need(out, "out", q.dtype, 4, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    S, k, Hq, D = q.shape
    if out.shape != q.shape or block_tables.shape[0] != S or context_lens.shape[0] != S or D != k_cache.shape[3]:
        raise ValueError("q/out/block_tables/context_lens shapes disagree")
    need = decode_multi_split_workspace_size(S, k, Hq, D, max_context_len, partition_size)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", device=dev)
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_decode_multi_split(_ptr(out), _ptr(q), _dtype_code(q.dtype), S, k, Hq, _ptr(k_cache),
                                       _ptr(v_cache), ctypes.byref(desc), _ptr(block_tables), block_tables.shape[1],
                                       _ptr(context_lens), float(scale), float(kv_scale), int(max_context_len),
                                       int(partition_size), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(dev))
    _check("pa_decode_multi_split", rc)


def cache_and_decode(out: torch.Tensor, q: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                     slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, kv_scale: float = 1.0,
                     max_context_len: int = 0, partition_size: int = 0,
                     workspace: Optional[torch.Tensor] = None) -> None:
    """One launch doing reshape_and_cache of the new rows and the decode (one
    pass, or split when partition_size > 0).  q/out [S, Hq, D] (one new token)
    or [S, k, Hq, D]; key/value [S * k, Hkv, D]; slot_mapping [S * k]."""
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(q, "q", (torch.float16, torch.bfloat16), None, dev)
    if q.dim() not in (3, 4):
        raise ValueError("q must have 3 or 4 dims")
    _need(out, "out", q.dtype, q.dim(), dev)
    _need(key, "key", q.dtype, 3, dev)
    _need(value, "value", q.dtype, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    S = q.shape[0]
    k = q.shape[1] if q.dim() == 4 else 1
    Hq, D = q.shape[-2], q.shape[-1]
    if out.shape != q.shape or block_tables.shape[0] != S or context_lens.shape[0] != S or D != k_cache.shape[3]:
        raise ValueError("q/out/block_tables/context_lens shapes disagree")
    if key.shape != value.shape or key.shape[0] != S * k or slot_mapping.shape[0] != S * k:
        raise ValueError("key/value/slot_mapping must have num_seqs * num_q_tokens rows")
    if key.shape[1] != k_cache.shape[1] or key.shape[2] != D:
        raise ValueError("key rows do not match the cache's heads/head_dim")
    ws_ptr, ws_bytes = None, 0
    if partition_size > 0:
        need = decode_multi_split_workspace_size(S, k, Hq, D, max_context_len, partition_size)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", device=dev)
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_cache_and_decode(_ptr(out), _ptr(q), _dtype_code(q.dtype), S, k, Hq, _ptr(key), _ptr(value),
                                     _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
                                     _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), float(scale),
                                     float(kv_scale), int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
                                     _stream(dev))
    _check("pa_cache_and_decode", rc)


def set_check_mode(enable: bool) -> bool:
    return bool(lib.pa_set_check_mode(1 if enable else 0))


def selftest_wait_timeout() -> None:
    """Enqueue, on torch's current stream, a kernel whose bounded mbarrier
    wait runs out (nothing arrives): after about one second it records
    DEVERR_TIMEOUT in the device error word and returns (read it with
    get_device_error())."""
    _check("pa_selftest_wait_timeout", lib.pa_selftest_wait_timeout(_stream(torch.device("cuda", torch.cuda.current_device()))))


def probe_l2_read(buf: torch.Tensor, mode: int, iters: int, sink: torch.Tensor) -> int:
    """Enqueue, on torch's current stream, the L2 read-rate probe over the
    bytes of `buf` (a contiguous CUDA tensor; mode 0: plain 16-byte loads,
    `iters` passes over the buffer; mode 1: TMA boxes of 16 x 128 bytes,
    `iters` 32 KB stages per SM).  `sink` is a CUDA tensor of at least 4 bytes.
    Returns the bytes the launch reads."""
    if not buf.is_cuda or not buf.is_contiguous() or not sink.is_cuda or sink.numel() * sink.element_size() < 4:
        raise ValueError("probe_l2_read wants a contiguous CUDA buffer and a CUDA sink of at least 4 bytes")
    n = ctypes.c_ulonglong(0)
    _check("pa_probe_l2_read", lib.pa_probe_l2_read(_ptr(buf), buf.numel() * buf.element_size(), int(mode),
                                                      int(iters), _ptr(sink), ctypes.byref(n), _stream(buf.device)))
    return int(n.value)


def get_device_error() -> int:
    rc = int(lib.pa_get_device_error())
    if rc < 0:
        raise PagedAttnError("pa_get_device_error", rc)
    return rc


def status_string(status: int) -> str:
    return lib.pa_status_string(status).decode()


# ---------------------------------------------------------------------------
# whole-block moves
# ---------------------------------------------------------------------------

def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs: torch.Tensor) -> None:
    """k/v_cache[dst] = k/v_cache[src] for each row (src, dst) of int64 pairs [n, 2]."""
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(pairs, "pairs", torch.int64, 2, dev)
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(pairs), pairs.shape[0],
                                _stream(dev))
    _check("pa_copy_blocks", rc)


def _check_buf(buf: torch.Tensor, k_cache: torch.Tensor, n: int):
    if not buf.is_contiguous():
        raise ValueError("buffer must be contiguous")
    need = n * 2 * k_cache[0].numel() * k_cache.element_size()
    if buf.numel() * buf.element_size() < need:
        raise ValueError("buffer holds %d bytes, %d needed" % (buf.numel() * buf.element_size(), need))
    if not (buf.is_cuda or buf.is_pinned()):
        raise ValueError("buffer must be device memory or pinned host memory")


def gather_blocks(dst: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, ids: torch.Tensor) -> None:
    """dst[i] = (k_cache[ids[i]], v_cache[ids[i]]); dst is device memory or pinned host memory."""
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(ids, "ids", torch.int64, 1, dev)
    _check_buf(dst, k_cache, ids.shape[0])
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_gather_blocks(_ptr(dst), _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(ids),
                                  ids.shape[0], _stream(dev))
    _check("pa_gather_blocks", rc)


def scatter_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src: torch.Tensor, ids: torch.Tensor) -> None:
    """(k_cache[ids[i]], v_cache[ids[i]]) = src[i]; src is device memory or pinned host memory."""
    _check_caches(k_cache, v_cache)
    dev = k_cache.device
    _need(ids, "ids", torch.int64, 1, dev)
    _check_buf(src, k_cache, ids.shape[0])
    desc = cache_desc(k_cache)
    with torch.cuda.device(dev):
        rc = lib.pa_scatter_blocks(_ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(src), _ptr(ids),
                                   ids.shape[0], _stream(dev))
    _check("pa_scatter_blocks", rc)


# ---------------------------------------------------------------------------
# host block manager
# ---------------------------------------------------------------------------

class BlockManager:
    """Owner of a pool's free list, block tables and reference counts (the
    native manager in the library; no device work)."""

    def __init__(self, num_blocks: int, block_size: int):
        self._h = lib.pa_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError("bad pool size")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.pa_bm_destroy(h)
            self._h = None

    def add_sequence(self, seq_id: int, num_tokens: int) -> None:
        _check("pa_bm_add_sequence", lib.pa_bm_add_sequence(self._h, seq_id, num_tokens))

    def fork(self, parent: int, child: int) -> None:
        _check("pa_bm_fork", lib.pa_bm_fork(self._h, parent, child))

    def append_tokens(self, seq_id: int, n: int):
        """Returns (slots [n], copy-on-write pair (src, dst) or None)."""
        slots = (ctypes.c_int64 * max(n, 1))()
        pair = (ctypes.c_int64 * 2)()
        ncow = ctypes.c_int32()
        _check("pa_bm_append_tokens", lib.pa_bm_append_tokens(self._h, seq_id, n, slots, pair, ctypes.byref(ncow)))
        return [slots[i] for i in range(n)], ((pair[0], pair[1]) if ncow.value else None)

    def free_sequence(self, seq_id: int) -> None:
        _check("pa_bm_free_sequence", lib.pa_bm_free_sequence(self._h, seq_id))

    def block_table(self, seq_id: int):
        """(list of physical block ids, number of tokens)."""
        nb, nt = ctypes.c_int32(), ctypes.c_int64()
        rc = lib.pa_bm_block_table(self._h, seq_id, None, 0, ctypes.byref(nb), ctypes.byref(nt))
        if rc == -8:
            _check("pa_bm_block_table", rc)
        buf = (ctypes.c_int32 * max(nb.value, 1))()
        _check("pa_bm_block_table", lib.pa_bm_block_table(self._h, seq_id, buf, nb.value, ctypes.byref(nb),
                                                          ctypes.byref(nt)))
        return [buf[i] for i in range(nb.value)], nt.value

    def num_free_blocks(self) -> int:
        return int(lib.pa_bm_num_free_blocks(self._h))

    def refcount(self, block: int) -> int:
        return int(lib.pa_bm_refcount(self._h, block))

    def tail_waste(self) -> int:
        return int(lib.pa_bm_tail_waste(self._h))

    def check(self) -> int:
        return int(lib.pa_bm_check(self._h))
