"""pa_cache_and_decode (the scatter of the new rows and the decode in one
launch) against the two separate calls and the oracle: the pool bytes after
the call are the oracle's scatter exactly, and every output bit equals the
separate path's (the same bytes go through the same arithmetic)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

CASES = [
    # (Hq, Hkv, D, q_dtype, kv_dtype, new tokens per sequence)
    (32, 8, 128, "bf16", "bf16", 1),
    (32, 32, 128, "f16", "f16", 1),
    (32, 8, 128, "bf16", "fp8", 1),
    (8, 8, 64, "f16", "fp8", 1),
    (32, 8, 128, "bf16", "bf16", 4),
    (6, 2, 64, "bf16", "bf16", 1),
]
LENS = [1, 15, 16, 17, 64, 65, 511, 513, 1000, 2049]


def _id(c):
    return "Hq%d-Hkv%d-D%d-%s-%s-k%d" % c


def _fused(wl, P=0):
    """A fresh pool (before this step's scatter) and one fused call."""
    pa = _gpu.lib()
    g = _gpu.OnGpu(wl)
    out = torch.full_like(g.q, float("nan"))
    pa.cache_and_decode(out, g.q, g.key, g.value, g.slots, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale,
                        max_context_len=wl.max_context_len, partition_size=P)
    torch.cuda.synchronize()
    return g, out


@pytest.mark.parametrize("P", [0, 64, 512])
@pytest.mark.parametrize("case", CASES, ids=_id)
def test_fused_equals_scatter_then_decode(case, P):
    Hq, Hkv, D, qd, kd, k = case
    wl = W.make_workload(name="t", seed=51, context_lens=LENS, Hq=Hq, Hkv=Hkv, D=D, bs=16, q_dtype=qd,
                         kv_dtype=kd, qlen=k)
    pa = _gpu.lib()
    assert pa.get_device_error() == 0
    g, out = _fused(wl, P)
    assert pa.get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    gk, gv = g.caches_host()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    ref = _gpu.OnGpu(wl)
    want = ref.step(partition_size=P).clone()
    assert torch.equal(out, want)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc, partition_size=P)) <= _gpu.tolerance(wl)


def test_slot_outside_the_sequences_table_is_flagged():
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=52, context_lens=[40, 100, 7], Hq=8, Hkv=2, D=128, bs=16, q_dtype="bf16",
                         kv_dtype="bf16")
    g = _gpu.OnGpu(wl)
    assert pa.get_device_error() == 0
    slots = g.slots.clone()
    slots[1] = slots[0]  # sequence 1's new row aimed at sequence 0's slot
    out = torch.empty_like(g.q)
    pa.cache_and_decode(out, g.q, g.key, g.value, slots, g.kc, g.vc, g.bt, g.cl, wl.scale)
    assert pa.get_device_error() & pa.DEVERR_SLOT
    slots = g.slots.clone()
    slots[2] = wl.NB * wl.bs + 5  # outside the pool: skipped and flagged
    pa.cache_and_decode(out, g.q, g.key, g.value, slots, g.kc, g.vc, g.bt, g.cl, wl.scale)
    assert pa.get_device_error() & pa.DEVERR_SLOT
    assert torch.isfinite(out.float()).all()
    # consistent slots: nothing flagged
    pa.cache_and_decode(out, g.q, g.key, g.value, g.slots, g.kc, g.vc, g.bt, g.cl, wl.scale)
    assert pa.get_device_error() == 0


@pytest.mark.parametrize("P", [0, 64])
def test_check_mode_flags_a_write_into_a_block_another_table_names(P):
    """Copy-on-write skipped: sequence 1 shares sequence 0's first three
    blocks, including the partially filled one that sequence 0's new row goes
    to.  Without check mode the write goes through unreported (the slot is in
    sequence 0's own table); check mode scans the other tables and reports it."""
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=53, context_lens=[40, 50, 20], Hq=8, Hkv=2, D=128, bs=16, q_dtype="bf16",
                         kv_dtype="bf16")
    g = _gpu.OnGpu(wl)
    out = torch.empty_like(g.q)
    assert pa.get_device_error() == 0
    prev = pa.set_check_mode(True)
    try:
        # private tables: nothing to report
        pa.cache_and_decode(out, g.q, g.key, g.value, g.slots, g.kc, g.vc, g.bt, g.cl, wl.scale,
                            max_context_len=wl.max_context_len, partition_size=P)
        bt = g.bt.clone()
        bt[1, :3] = bt[0, :3]  # blocks of tokens 0-47 of sequence 1 = sequence 0's blocks 0-2
        slots = g.slots.clone()  # row 0 goes to position 39, in block bt[0, 2]
        with pytest.raises(pa.PagedAttnError) as e:
            pa.cache_and_decode(out, g.q, g.key, g.value, slots, g.kc, g.vc, bt, g.cl, wl.scale,
                                max_context_len=wl.max_context_len, partition_size=P)
        assert e.value.status == -5
        # the shared block is not the new row's once sequence 1 keeps only the
        # full blocks 0-1 in common (block 2 private again): nothing reported
        bt[1, 2] = g.bt[1, 2]
        pa.cache_and_decode(out, g.q, g.key, g.value, slots, g.kc, g.vc, bt, g.cl, wl.scale,
                            max_context_len=wl.max_context_len, partition_size=P)
    finally:
        pa.set_check_mode(prev)
    assert pa.get_device_error() == 0
