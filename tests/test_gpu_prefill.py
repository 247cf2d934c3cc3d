"""Chunked prefill on the tensor cores (pa_prefill) against the oracle: each
of the C new tokens is decoded by the oracle over the context prefix ending
at its own position (causal), through the same block table."""
import numpy as np
import pytest
import torch

from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

CASES = [
    # (Hq, Hkv, q/kv dtype, bs, C, context lengths)
    (4, 4, "bf16", 16, 128, [128, 200, 700]),
    (8, 2, "bf16", 16, 256, [256, 300, 1000, 129]),
    (4, 1, "f16", 8, 192, [192, 450, 64]),
    (2, 2, "bf16", 32, 320, [320, 333, 1500]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "Hq%d-Hkv%d-%s-bs%d-C%d" % c[:5])
def test_prefill_matches_oracle(case):
    Hq, Hkv, dt, bs, C, lens = case
    wl = W.make_workload(name="t", seed=41, context_lens=lens, Hq=Hq, Hkv=Hkv, D=128, bs=bs, q_dtype=dt,
                         kv_dtype=dt, qlen=C)
    g = _gpu.OnGpu(wl)
    g.scatter()
    out = torch.full_like(g.q, float("nan"))
    _gpu.lib().prefill(out, g.q, g.kc, g.vc, g.bt, g.cl, wl.scale)
    torch.cuda.synchronize()
    assert _gpu.lib().get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    want = _gpu.oracle_out(wl, kc, vc)
    err = _gpu.max_err(out, want)
    assert err <= _gpu.tolerance(wl), err
    # rows whose position is negative (C > L) are zero
    for s, L in enumerate(lens):
        for j in range(max(0, C - L)):
            assert torch.all(out[s, j] == 0)
