"""pa_decode_split_noalloc: split decode whose scratch is compiled into the
library, for callers that cannot allocate device memory at call time (for
example a serving process whose KV-cache pool already reserved nearly all of
HBM, or a host framework that owns every device allocation of its
plug-ins).  Called through the C ABI, its output must be bit-identical to
pa_decode_split with a caller-provided workspace (the same kernels, partition
runs and merge order run on the same bytes), call after call, and within
tolerance of the oracle's split evaluation.

This file is named to be collected last: it also passes on its own in a fresh
process."""
import ctypes

import pytest
import torch

import oracle
from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # the limit stated in include/pagedattn.h


def _call(pa, b, out, P, max_context_len=None, num_seqs=None):
    wl = b.wl
    desc = pa.cache_desc(b.k_cache)
    mcl = wl.max_context_len if max_context_len is None else max_context_len
    S = wl.S if num_seqs is None else num_seqs
    return pa.lib.pa_decode_split_noalloc(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(b.q.data_ptr()), pa._dtype_code(b.q.dtype), S, wl.Hq,
        ctypes.c_void_p(b.k_cache.data_ptr()), ctypes.c_void_p(b.v_cache.data_ptr()), ctypes.byref(desc),
        ctypes.c_void_p(b.block_tables.data_ptr()), wl.max_blocks, ctypes.c_void_p(b.context_lens.data_ptr()),
        float(wl.scale), float(wl.kv_scale), int(mcl), int(P),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _oracle_split(b, P):
    wl = b.wl
    if wl.kv_dtype == "fp8":
        kc, vc = b.k_cache.cpu().numpy(), b.v_cache.cpu().numpy()
    else:
        kc, vc = _gpu.host16(b.k_cache), _gpu.host16(b.v_cache)
    return oracle.decode(wl.q, wl.q_dtype, kc, vc, wl.kv_dtype, wl.block_tables, wl.context_lens, wl.scale,
                         wl.kv_scale, partition_size=P)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_noalloc_split_matches_workspace_split_twice(kv_dtype):
    pa = _gpu.lib()
    from paged_kv_cache_230_gb300.device import DeviceBatch
    P = 128
    wl = W.make_workload(name="t", seed=21, context_lens=[1, 64, 129, 700, 2049, 513, 3000, 40], Hq=32, Hkv=8,
                         D=128, bs=16, q_dtype="bf16", kv_dtype=kv_dtype)
    assert pa.decode_split_workspace_size(wl.S, wl.Hq, wl.D, wl.max_context_len, P) <= SCRATCH_BYTES
    b = DeviceBatch(wl, "cuda", partition_size=P)
    want = b.step().clone()  # existing entry point, caller-provided workspace
    torch.cuda.synchronize()
    ref = _oracle_split(b, P)
    # a larger batch with another layout in between: the second small call
    # reads scratch that different partial rows last wrote
    big = W.make_workload(name="t2", seed=23, context_lens=[4000 + 37 * i for i in range(24)], Hq=32, Hkv=8,
                          D=128, bs=16, q_dtype="bf16", kv_dtype=kv_dtype)
    assert pa.decode_split_workspace_size(big.S, big.Hq, big.D, big.max_context_len, 64) <= SCRATCH_BYTES
    bb = DeviceBatch(big, "cuda", partition_size=64)
    bb.scatter()
    big_want = bb.decode().clone()
    for i in range(2):
        out = torch.full_like(b.q, float("nan"))
        assert _call(pa, b, out, P) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, want), "call %d differs from pa_decode_split" % i
        assert _gpu.max_err(out, ref) <= _gpu.tolerance(wl)
        if i == 0:
            big_out = torch.full_like(bb.q, float("nan"))
            assert _call(pa, bb, big_out, 64) == 0
            torch.cuda.synchronize()
            assert torch.equal(big_out, big_want)


def test_noalloc_rejects_batches_beyond_its_scratch():
    pa = _gpu.lib()
    from paged_kv_cache_230_gb300.device import DeviceBatch
    wl = W.make_workload(name="t", seed=22, context_lens=[5, 9], Hq=8, Hkv=8, D=128, bs=16, q_dtype="f16",
                         kv_dtype="f16")
    b = DeviceBatch(wl, "cuda", partition_size=0)
    out = torch.zeros_like(b.q)
    huge = 1 << 30  # a context bound whose partials would need far more than 32 MiB
    assert pa.decode_split_workspace_size(wl.S, wl.Hq, wl.D, huge, 64) > SCRATCH_BYTES
    assert _call(pa, b, out, 64, max_context_len=huge) == -3
    # argument errors come first, as in pa_decode_split: a partition size
    # that is not a multiple of 64 is invalid whatever the batch's size
    assert _call(pa, b, out, 100, max_context_len=huge) == -1
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    # an empty batch is a no-op, as for pa_decode_split
    assert _call(pa, b, out, 64, num_seqs=0) == 0
