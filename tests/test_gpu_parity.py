"""GPU parity: the CUDA path against the fp64 oracle on the same seeded bytes.

Scatter and block-table handling must be bit-exact; attention must stay within
max |gpu - oracle| <= 2e-3 (fp16 out), 1.6e-2 (bf16 out), 5e-2 (FP8 KV)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 15, 16, 17, 63, 64, 65, 127, 511, 512, 513, 1000, 2049]

CASES = [
    # (Hq, Hkv, D, q_dtype, kv_dtype)
    (8, 8, 64, "f16", "f16"),     # MHA, warp-shuffle path
    (32, 32, 128, "f16", "f16"),
    (32, 8, 128, "bf16", "bf16"),  # G = 4, MMA path
    (64, 8, 128, "bf16", "bf16"),  # G = 8
    (16, 1, 128, "f16", "f16"),    # G = 16
    (6, 2, 64, "bf16", "bf16"),    # G = 3, warp-shuffle path
    (4, 2, 128, "f16", "f16"),     # G = 2
    (32, 8, 128, "bf16", "fp8"),   # FP8 KV, MMA path
    (8, 8, 128, "bf16", "fp8"),    # FP8 KV, warp-shuffle path
    (16, 2, 64, "f16", "fp8"),     # FP8 rows of 64 bytes, MMA path
    (2, 2, 64, "bf16", "fp8"),     # FP8 rows of 64 bytes, warp-shuffle path
    (20, 4, 64, "f16", "f16"),     # G = 5 (padded to 8)
]


def _id(c):
    return "Hq%d-Hkv%d-D%d-%s-%s" % c


def _workload(case, bs=16, lens=EDGE_LENS, seed=0, **kw):
    Hq, Hkv, D, qd, kd = case
    return W.make_workload(name="t", seed=seed, context_lens=lens, Hq=Hq, Hkv=Hkv, D=D, bs=bs, q_dtype=qd,
                           kv_dtype=kd, **kw)


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_scatter_bit_exact_and_decode_within_tolerance(case):
    wl = _workload(case)
    g = _gpu.OnGpu(wl)
    out = g.step()
    torch.cuda.synchronize()
    kc, vc = _gpu.oracle_pool(wl)
    gk, gv = g.caches_host()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc), "scatter differs from the oracle"
    want = _gpu.oracle_out(wl, kc, vc)
    err = _gpu.max_err(out, want)
    assert err <= _gpu.tolerance(wl), err


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[7], CASES[10]], ids=_id)
def test_other_block_sizes(case, bs):
    wl = _workload(case, bs=bs, lens=[1, 7, 8, 9, 31, 32, 33, 100, 700])
    g = _gpu.OnGpu(wl)
    out = g.step()
    kc, vc = _gpu.oracle_pool(wl)
    gk, gv = g.caches_host()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)


@pytest.mark.parametrize("P", [64, 128, 512])
@pytest.mark.parametrize("case", [CASES[1], CASES[2], CASES[3], CASES[7], CASES[5]], ids=_id)
def test_split_within_tolerance(case, P):
    wl = _workload(case, lens=[1, 64, 65, 511, 512, 513, 1500, 3000])
    g = _gpu.OnGpu(wl)
    out = g.step(partition_size=P)
    kc, vc = _gpu.oracle_pool(wl)
    want = _gpu.oracle_out(wl, kc, vc, partition_size=P)
    assert _gpu.max_err(out, want) <= _gpu.tolerance(wl)


@pytest.mark.parametrize("case", [CASES[1], CASES[2], CASES[7], CASES[5]], ids=_id)
def test_block_placement_is_bit_invariant(case):
    """Moving blocks to other physical ids, or giving each sequence private
    copies of shared blocks, must not change a single output bit."""
    wl = _workload(case, lens=[300, 1, 77, 1024, 513])
    g = _gpu.OnGpu(wl)
    base = g.step().clone()
    # run to run
    assert torch.equal(g.decode(), base)
    # physical permutation of the pool
    perm = torch.from_numpy(np.random.default_rng(1).permutation(wl.NB)).cuda()
    kc2 = torch.empty_like(g.kc)
    vc2 = torch.empty_like(g.vc)
    kc2[perm] = g.kc
    vc2[perm] = g.vc
    bt2 = torch.where(g.bt >= 0, perm[g.bt.clamp(min=0).long()].int(), g.bt)
    out2 = torch.empty_like(base)
    _gpu.lib().decode(out2, g.q, kc2, vc2, bt2, g.cl, wl.scale, wl.kv_scale)
    assert torch.equal(out2, base)
    # split with one partition covering every context takes the same arithmetic
    assert torch.equal(g.decode(partition_size=4096), base)


def test_shared_prefix_equals_private_copies():
    lens = [256 + 1 + t for t in (0, 5, 17, 40, 3, 9, 100, 250)]
    for kd in ("bf16", "fp8"):
        wl = W.make_workload(name="t", seed=4, context_lens=lens, Hq=32, Hkv=8, D=128, bs=16, q_dtype="bf16",
                             kv_dtype=kd, shared_prefix=(2, 256))
        g = _gpu.OnGpu(wl)
        base = g.step().clone()
        nshared = 256 // 16
        extra = wl.S * nshared
        kc2 = torch.cat([g.kc, torch.empty((extra,) + tuple(g.kc.shape[1:]), dtype=g.kc.dtype, device="cuda")])
        vc2 = torch.cat([g.vc, torch.empty((extra,) + tuple(g.vc.shape[1:]), dtype=g.vc.dtype, device="cuda")])
        bt2 = g.bt.clone()
        nxt = wl.NB
        for s in range(wl.S):
            for j in range(nshared):
                b = int(wl.block_tables[s, j])
                kc2[nxt] = g.kc[b]
                vc2[nxt] = g.vc[b]
                bt2[s, j] = nxt
                nxt += 1
        out2 = torch.empty_like(base)
        _gpu.lib().decode(out2, g.q, kc2, vc2, bt2, g.cl, wl.scale, wl.kv_scale)
        assert torch.equal(out2, base)
        kc, vc = _gpu.oracle_pool(wl)
        assert _gpu.max_err(base, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)


@pytest.mark.parametrize("case", [CASES[1], CASES[2], CASES[7], CASES[5]], ids=_id)
def test_unused_slots_holding_nan_are_never_read(case):
    wl = _workload(case, lens=[1, 17, 33, 100, 513], fill_unused="nan")
    g = _gpu.OnGpu(wl)
    out = g.step()
    kc, vc = _gpu.oracle_pool(wl)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)
    out = g.decode(partition_size=64)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)


def test_zero_length_context_and_padding_slot():
    case = CASES[2]
    wl = _workload(case, lens=[0, 5, 0, 40])
    g = _gpu.OnGpu(wl)
    before_k = g.kc.clone()
    g.slots[:] = torch.where(g.cl > 0, g.slots, torch.full_like(g.slots, -1))
    out = g.step()
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    kc, vc = _gpu.oracle_pool(wl)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)
    # a padding slot (-1) writes nothing
    g2 = _gpu.OnGpu(wl)
    g2.slots.fill_(-1)
    g2.scatter()
    assert torch.equal(g2.kc, before_k)
    out = g.decode(partition_size=64)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)


def test_empty_batch_is_a_no_op():
    pa = _gpu.lib()
    kc = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    cl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    pa.decode(q.clone(), q, kc, kc, bt, cl, 0.1)
    key = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    pa.reshape_and_cache(key, key, kc, kc.clone(), torch.zeros((0,), dtype=torch.int64, device="cuda"))


@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_fp8_scatter_every_input_pattern(in_dtype):
    """All 65536 16-bit inputs, several per-tensor scales: every code equals the
    oracle's (IEEE float32 division, then nearest-even E4M3 with saturation);
    NaN inputs give a NaN code."""
    pa = _gpu.lib()
    D, Hkv = 128, 1
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(-1, Hkv, D)  # 512 tokens
    T = bits.shape[0]
    NB, bs = T // 16, 16
    slots = np.random.default_rng(0).permutation(NB * bs)[:T].astype(np.int64)
    dec = oracle.decode16(bits.reshape(-1), in_dtype)
    nan_in = np.isnan(dec).reshape(T, D)
    for kv_scale in (1.0, 0.0123, 2.0 ** -4, 3.7, 1e-3, 448.0 / 3.0):
        kc = np.zeros((NB, Hkv, bs, D), np.uint8)
        vc = np.zeros_like(kc)
        oracle.reshape_and_cache(bits, bits, in_dtype, kc, vc, "fp8", slots, kv_scale)
        gk = torch.zeros((NB, Hkv, bs, D), dtype=torch.uint8, device="cuda")
        gv = torch.zeros_like(gk)
        x = _gpu.dev16(bits, in_dtype)
        pa.reshape_and_cache(x, x, gk, gv, torch.from_numpy(slots).cuda(), kv_scale)
        got = gk.cpu().numpy()
        want = kc
        rows_got = got[slots // bs, 0, slots % bs, :]
        rows_want = want[slots // bs, 0, slots % bs, :]
        assert np.array_equal(rows_got[~nan_in], rows_want[~nan_in]), kv_scale
        assert np.all((rows_got[nan_in] & 0x7F) == 0x7F)
        assert np.array_equal(gv.cpu().numpy(), got)


def test_out_of_range_indices_are_contained_and_reported():
    pa = _gpu.lib()
    case = CASES[2]
    wl = _workload(case, lens=[40, 100])
    g = _gpu.OnGpu(wl)
    assert pa.get_device_error() == 0
    prev = pa.set_check_mode(True)
    try:
        g.step()  # valid input: no error
        bad = g.bt.clone()
        bad[1, 2] = wl.NB + 7  # block id outside the pool
        out = torch.empty_like(g.q)
        with pytest.raises(pa.PagedAttnError) as e:
            pa.decode(out, g.q, g.kc, g.vc, bad, g.cl, wl.scale)
        assert e.value.status == -5
        assert torch.isfinite(out.float()).all()
        cl = g.cl.clone()
        cl[0] = wl.max_blocks * wl.bs + 1  # longer than its table
        with pytest.raises(pa.PagedAttnError):
            pa.decode(out, g.q, g.kc, g.vc, g.bt, cl, wl.scale)
        slots = g.slots.clone()
        slots[0] = wl.NB * wl.bs + 3
        kc_before = g.kc.clone()
        with pytest.raises(pa.PagedAttnError):
            pa.reshape_and_cache(g.key, g.value, g.kc, g.vc, slots)
        # the in-range token was written, the out-of-range one was not
        # only the in-range token's row changed
        sl = int(wl.slot_mapping[1])
        expect = kc_before.clone()
        expect[sl // 16, :, sl % 16] = g.key[1]
        assert torch.equal(g.kc, expect)
    finally:
        pa.set_check_mode(prev)
    # outside check mode the same event is recorded and readable later
    pa.decode(out, g.q, g.kc, g.vc, bad, g.cl, wl.scale)
    assert pa.get_device_error() & pa.DEVERR_BLOCK_ID
    assert pa.get_device_error() == 0


def test_host_side_argument_errors_launch_nothing():
    pa = _gpu.lib()
    kc = torch.zeros((4, 2, 16, 96), dtype=torch.bfloat16, device="cuda")  # head_dim 96: not built
    q = torch.zeros((1, 4, 96), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    cl = torch.ones((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.decode(q.clone(), q, kc, kc, bt, cl, 0.1)
    assert e.value.status == -2
    kc = torch.zeros((4, 3, 16, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")  # 4 % 3 != 0
    with pytest.raises(pa.PagedAttnError) as e:
        pa.decode(q.clone(), q, kc, kc, bt, cl, 0.1)
    assert e.value.status == -1
    kc = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:  # 16-bit caches take kv_scale 1
        pa.decode(q.clone(), q, kc, kc, bt, cl, 0.1, kv_scale=0.5)
    assert e.value.status == -1
    small = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.decode_split(q.clone(), q, kc, kc, bt, cl, 0.1, 1.0, 64, 64, small)
    assert e.value.status == -3
    with pytest.raises(pa.PagedAttnError) as e:  # partition size must be a multiple of 64
        pa.decode_split(q.clone(), q, kc, kc, bt, cl, 0.1, 1.0, 64, 100)
    assert e.value.status == -1
    assert pa.get_device_error() == 0
