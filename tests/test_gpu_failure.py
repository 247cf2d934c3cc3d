"""Failure detection without a GPU fault: a pipeline wait that runs out
gives up after about a second, the kernel records the timeout in the device
error word and returns, and the context keeps working."""
import time

import pytest

from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_reports_and_context_stays_usable():
    lib = _gpu.lib()
    lib.get_device_error()  # clears earlier bits
    t0 = time.perf_counter()
    lib.selftest_wait_timeout()
    bits = lib.get_device_error()  # synchronises the device
    dt = time.perf_counter() - t0
    assert bits == lib.DEVERR_TIMEOUT
    assert 0.5 < dt < 30.0, dt
    assert lib.get_device_error() == 0  # read and cleared
    # the same context still runs the decode path correctly
    wl = W.make_workload(name="t", seed=5, context_lens=[1, 17, 200, 513], Hq=8, Hkv=2, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16")
    g = _gpu.OnGpu(wl)
    g.scatter()
    out = g.decode()
    assert lib.get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    err = _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc))
    assert err <= _gpu.tolerance(wl), err
