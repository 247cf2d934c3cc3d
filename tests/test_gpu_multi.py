"""Multi-token decode (k new tokens per sequence, causal among them) against
the oracle: the scatter of the k rows is bit-exact and every output is within
tolerance; tokens whose position is negative (k > L) give zeros."""
import numpy as np
import pytest
import torch

from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

CASES = [
    # (Hq, Hkv, D, q_dtype, kv_dtype, k)
    (32, 8, 128, "bf16", "bf16", 4),   # 16 columns
    (64, 8, 128, "bf16", "bf16", 2),   # 16 columns
    (32, 32, 128, "f16", "f16", 4),    # MHA: 4 columns
    (8, 8, 64, "f16", "f16", 8),       # 8 columns
    (32, 8, 128, "bf16", "fp8", 2),    # FP8 KV
    (32, 8, 128, "bf16", "fp8", 4),    # FP8 KV, 16 columns
    (16, 4, 64, "f16", "fp8", 4),      # FP8 rows of 64 bytes, 16 columns
    (12, 4, 128, "bf16", "bf16", 5),   # 15 columns (padded to 16)
]
LENS = [1, 3, 4, 5, 15, 16, 17, 64, 65, 511, 513, 1000, 2049]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "Hq%d-Hkv%d-D%d-%s-%s-k%d" % c)
def test_multi_token_decode(case):
    Hq, Hkv, D, qd, kd, k = case
    wl = W.make_workload(name="t", seed=31, context_lens=LENS, Hq=Hq, Hkv=Hkv, D=D, bs=16, q_dtype=qd,
                         kv_dtype=kd, qlen=k)
    g = _gpu.OnGpu(wl)
    out = g.step()
    torch.cuda.synchronize()
    kc, vc = _gpu.oracle_pool(wl)
    gk, gv = g.caches_host()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    want = _gpu.oracle_out(wl, kc, vc)
    assert _gpu.max_err(out, want) <= _gpu.tolerance(wl)
    # tokens before the start of the context attend to nothing
    L = wl.context_lens
    for s in range(wl.S):
        for j in range(k):
            if L[s] - k + j < 0:
                assert torch.all(out[s, j] == 0)
    # deterministic
    out2 = g.decode().clone()
    assert torch.equal(out2, out)


def test_single_token_through_multi_matches_decode():
    wl = W.make_workload(name="t", seed=32, context_lens=[5, 700, 33, 1500], Hq=32, Hkv=8, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16")
    g = _gpu.OnGpu(wl)
    base = g.step().clone()
    out = torch.empty_like(g.q).unsqueeze(1)
    _gpu.lib().decode_multi(out, g.q.unsqueeze(1).contiguous(), g.kc, g.vc, g.bt, g.cl, wl.scale)
    assert torch.equal(out[:, 0], base)


@pytest.mark.parametrize("P", [64, 512])
@pytest.mark.parametrize("case", [CASES[0], CASES[4], CASES[5], CASES[6]],
                         ids=lambda c: "Hq%d-Hkv%d-D%d-%s-%s-k%d" % c)
def test_multi_token_split_decode(case, P):
    """pa_decode_multi_split: the same causal result, per partition and
    merged by log-sum-exp; a partition wholly after a new token's position
    (L = 65 or 513 with k > 1) contributes nothing to it."""
    Hq, Hkv, D, qd, kd, k = case
    wl = W.make_workload(name="t", seed=33, context_lens=LENS, Hq=Hq, Hkv=Hkv, D=D, bs=16, q_dtype=qd,
                         kv_dtype=kd, qlen=k)
    g = _gpu.OnGpu(wl)
    out = g.step(partition_size=P).clone()
    torch.cuda.synchronize()
    kc, vc = _gpu.oracle_pool(wl)
    want = _gpu.oracle_out(wl, kc, vc, partition_size=P)
    assert _gpu.max_err(out, want) <= _gpu.tolerance(wl)
    L = wl.context_lens
    for s in range(wl.S):
        for j in range(k):
            if L[s] - k + j < 0:
                assert torch.all(out[s, j] == 0)
    assert torch.equal(g.decode(partition_size=P), out)  # deterministic
    one_pass = g.decode().clone()
    assert _gpu.max_err(one_pass, want) <= _gpu.tolerance(wl)


@pytest.mark.parametrize("kd", ["bf16", "fp8"])
def test_sixteen_columns_never_read_nan_in_unused_slots(kd):
    """16 query columns (G = 4, k = 4) over contexts whose last sub-tile is
    ragged, with every slot outside the contexts holding NaN codes: masked
    tokens must not reach the output, on the variant with separate K and V
    stage barriers (16-bit caches) and on the E4M3 one."""
    wl = W.make_workload(name="t", seed=37, context_lens=[1, 17, 33, 100, 513], Hq=32, Hkv=8, D=128, bs=16,
                         q_dtype="bf16", kv_dtype=kd, qlen=4, fill_unused="nan")
    g = _gpu.OnGpu(wl)
    out = g.step()
    torch.cuda.synchronize()
    kc, vc = _gpu.oracle_pool(wl)
    want = _gpu.oracle_out(wl, kc, vc)
    assert torch.isfinite(out).all()
    assert _gpu.max_err(out, want) <= _gpu.tolerance(wl)
    # the split variant: 64-token partitions end inside the ragged tails too
    out = g.decode(partition_size=64)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert _gpu.max_err(out, want) <= _gpu.tolerance(wl)
