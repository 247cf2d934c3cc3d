"""The five named workloads at full size, in the launch configuration the
benchmark times: the whole pool after the scatter is compared byte for byte
with the oracle's, and EVERY output of the batch is compared with the
oracle's fp64 decode, for both launch forms — the single-pass fused step and
the split fused step (partitions merged by log-sum-exp), the latter against
the oracle's own split evaluation with the same partition size."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4], ids=W.CONFIG_NAMES)
def test_full_size_workload(idx):
    from paged_kv_cache_230_gb300.device import DeviceBatch
    wl = W.make_config(idx)
    b = DeviceBatch(wl, "cuda")
    out = b.step().clone()
    torch.cuda.synchronize()
    kc, vc = _gpu.oracle_pool(wl)
    if wl.kv_dtype == W.FP8:
        gk, gv = b.k_cache.cpu().numpy(), b.v_cache.cpu().numpy()
    else:
        gk, gv = _gpu.host16(b.k_cache), _gpu.host16(b.v_cache)
    assert np.array_equal(gk, kc), "K pool differs from the oracle's"
    assert np.array_equal(gv, vc), "V pool differs from the oracle's"
    del gk, gv
    tol = _gpu.tolerance(wl)
    # the launch form the benchmark times (split for the long-context
    # workload, single pass otherwise), every sequence
    want = oracle.decode(wl.q, wl.q_dtype, kc, vc, wl.kv_dtype, wl.block_tables, wl.context_lens, wl.scale,
                         wl.kv_scale, partition_size=wl.partition_size)
    err = _gpu.max_err(out, want)
    # the other launch form: split with 512-token partitions where the
    # workload runs single pass, single pass where it runs split; the pool
    # already holds this step's rows, and the fused write stores the same bytes
    P2 = 0 if wl.partition_size else 512
    b2 = DeviceBatch(wl, "cuda", partition_size=P2)
    out2 = b2.step()
    torch.cuda.synchronize()
    want2 = oracle.decode(wl.q, wl.q_dtype, kc, vc, wl.kv_dtype, wl.block_tables, wl.context_lens, wl.scale,
                          wl.kv_scale, partition_size=P2)
    err2 = _gpu.max_err(out2, want2)
    print("%s: max|gpu - oracle| = %.3g (partition %d), %.3g (partition %d), %d outputs each, tolerance %g"
          % (wl.name, err, wl.partition_size, err2, P2, want.size, tol))
    assert err <= tol, err
    assert err2 <= tol, err2
