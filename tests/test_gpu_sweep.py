"""A seeded sweep over the supported space, beside the hand-picked cases:
group sizes 1 to 16, head_dim 64 or 128, block size 8, 16 or 32, every q and
cache dtype pairing, 1 to 4 new tokens per sequence (group size x tokens up
to 16), one pass or split into 64- or 256-token partitions, and the fused
launch or the scatter and the decode as two calls.  In every case the pool
after the step equals the oracle's scatter bit for bit and the attention is
within the dtype's tolerance of the oracle."""
import numpy as np
import pytest
import torch

from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

DTYPES = [("f16", "f16"), ("bf16", "bf16"), ("bf16", "fp8"), ("f16", "fp8")]


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    while True:
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.integers(1, 17))
        k = int(rng.integers(1, 5))
        if G * k <= 16:
            break
    qd, kd = DTYPES[int(rng.integers(0, len(DTYPES)))]
    S = int(rng.integers(1, 7))
    return dict(Hq=G * Hkv, Hkv=Hkv, D=int(rng.choice([64, 128])), bs=int(rng.choice([8, 16, 32])), q_dtype=qd,
                kv_dtype=kd, qlen=k, lens=[int(x) for x in rng.integers(k, 1500, size=S)],
                P=int(rng.choice([0, 64, 256])), fused=bool(rng.integers(0, 2)), seed=2000 + i)


CASES = [_draw(i) for i in range(32)]


def _id(c):
    return "Hq%d-Hkv%d-D%d-bs%d-%s-%s-k%d-P%d-%s" % (c["Hq"], c["Hkv"], c["D"], c["bs"], c["q_dtype"], c["kv_dtype"],
                                                    c["qlen"], c["P"], "fused" if c["fused"] else "two")


@pytest.mark.parametrize("c", CASES, ids=_id)
def test_sweep_scatter_bit_exact_and_attention_within_tolerance(c):
    wl = W.make_workload(name="t", seed=c["seed"], context_lens=c["lens"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"],
                         bs=c["bs"], q_dtype=c["q_dtype"], kv_dtype=c["kv_dtype"], qlen=c["qlen"])
    pa = _gpu.lib()
    assert pa.get_device_error() == 0
    g = _gpu.OnGpu(wl)
    if c["fused"]:
        out = torch.full_like(g.q, float("nan"))
        pa.cache_and_decode(out, g.q, g.key, g.value, g.slots, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale,
                            max_context_len=wl.max_context_len, partition_size=c["P"])
    else:
        out = g.step(partition_size=c["P"])
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    gk, gv = g.caches_host()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc), "scatter differs from the oracle"
    err = _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc, partition_size=c["P"]))
    assert err <= _gpu.tolerance(wl), err
