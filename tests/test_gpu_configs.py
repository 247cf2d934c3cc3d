"""The five named workloads at full size, in the launch configuration the
benchmark times: the whole pool after the scatter is compared byte for byte
with the oracle's, and sampled sequences (always including the shortest and
the longest) are decoded by the oracle and compared within tolerance."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

SAMPLES = {0: 4, 1: 12, 2: 16, 3: 2, 4: 12}


def _sample(wl, k, seed):
    L = wl.context_lens
    pick = {int(np.argmin(L)), int(np.argmax(L))}
    rng = np.random.default_rng(seed)
    rest = [i for i in rng.permutation(wl.S) if int(i) not in pick]
    for i in rest[:max(0, k - len(pick))]:
        pick.add(int(i))
    return np.array(sorted(pick))


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4], ids=W.CONFIG_NAMES)
def test_full_size_workload(idx):
    from paged_kv_cache_230_gb300.device import DeviceBatch
    wl = W.make_config(idx)
    b = DeviceBatch(wl, "cuda")
    out = b.step()
    torch.cuda.synchronize()
    kc, vc = _gpu.oracle_pool(wl)
    if wl.kv_dtype == W.FP8:
        gk, gv = b.k_cache.cpu().numpy(), b.v_cache.cpu().numpy()
    else:
        gk, gv = _gpu.host16(b.k_cache), _gpu.host16(b.v_cache)
    assert np.array_equal(gk, kc), "K pool differs from the oracle's"
    assert np.array_equal(gv, vc), "V pool differs from the oracle's"
    del gk, gv
    seqs = _sample(wl, SAMPLES[idx], idx)
    sub = W.subset(wl, seqs)
    want = oracle.decode(sub.q, sub.q_dtype, kc, vc, sub.kv_dtype, sub.block_tables, sub.context_lens, sub.scale,
                         sub.kv_scale)
    got = out[torch.from_numpy(seqs).cuda()]
    err = _gpu.max_err(got, want)
    assert err <= _gpu.tolerance(wl), err
    # whole-batch properties at any size: finite outputs, and the single-pass
    # and split paths agree within the same tolerance
    assert torch.isfinite(out.float()).all()
    if wl.partition_size:
        b2 = DeviceBatch(wl, "cuda", partition_size=0)
        out2 = b2.step()
    else:
        b2 = DeviceBatch(wl, "cuda", partition_size=512)
        out2 = b2.step()
    diff = (out.float() - out2.float()).abs().max().item()
    assert diff <= 2 * _gpu.tolerance(wl), diff
