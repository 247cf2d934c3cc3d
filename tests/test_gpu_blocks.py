"""Whole-block moves on the GPU against the oracle (bit-exact), swapping
through pinned host memory, and a decode step driven by the native block
manager: prompts, forks that share their blocks, appends that trigger
copy-on-write, the block copy, the scatter of the new rows and the decode --
every step mirrored by the oracle on host arrays."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu


def _pool(NB, Hkv, bs, D, dt, seed):
    if dt == "fp8":
        rng = np.random.default_rng(seed)
        return (rng.integers(0, 256, size=(NB, Hkv, bs, D), dtype=np.uint8),
                rng.integers(0, 256, size=(NB, Hkv, bs, D), dtype=np.uint8))
    ss = np.random.SeedSequence(seed)
    a, b = ss.spawn(2)
    return W.normal_bits(a, (NB, Hkv, bs, D), dt), W.normal_bits(b, (NB, Hkv, bs, D), dt)


def _dev(a, dt):
    return torch.from_numpy(a).cuda() if dt == "fp8" else _gpu.dev16(a, dt)


def _host(t, dt):
    return t.cpu().numpy() if dt == "fp8" else _gpu.host16(t)


@pytest.mark.parametrize("dt,D,bs", [("bf16", 128, 16), ("f16", 64, 8), ("fp8", 128, 32), ("fp8", 64, 16)])
def test_copy_gather_scatter_bit_exact(dt, D, bs):
    pa = _gpu.lib()
    NB, Hkv = 64, 4
    kc, vc = _pool(NB, Hkv, bs, D, dt, 5)
    gk, gv = _dev(kc, dt), _dev(vc, dt)
    rng = np.random.default_rng(1)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:20], perm[20:40]], axis=1).astype(np.int64)  # sources and destinations disjoint
    pa.copy_blocks(gk, gv, torch.from_numpy(pairs).cuda())
    oracle.copy_blocks(kc, vc, pairs)
    assert np.array_equal(_host(gk, dt), kc) and np.array_equal(_host(gv, dt), vc)
    ids = rng.permutation(NB)[:25].astype(np.int64)
    buf = torch.empty((25, 2) + tuple(gk.shape[1:]), dtype=gk.dtype, device="cuda")
    pa.gather_blocks(buf, gk, gv, torch.from_numpy(ids).cuda())
    want = oracle.gather_blocks(kc, vc, ids)
    assert np.array_equal(_host(buf, dt), want)
    # scatter into a zeroed pool
    zk, zv = torch.zeros_like(gk), torch.zeros_like(gv)
    pa.scatter_blocks(zk, zv, buf, torch.from_numpy(ids).cuda())
    ok_, ov = np.zeros_like(kc), np.zeros_like(vc)
    oracle.scatter_blocks(ok_, ov, want, ids)
    assert np.array_equal(_host(zk, dt), ok_) and np.array_equal(_host(zv, dt), ov)


def test_swap_out_to_pinned_host_and_back():
    pa = _gpu.lib()
    NB, Hkv, bs, D = 128, 8, 16, 128
    kc, vc = _pool(NB, Hkv, bs, D, "bf16", 6)
    gk, gv = _dev(kc, "bf16"), _dev(vc, "bf16")
    ids = torch.from_numpy(np.random.default_rng(2).permutation(NB)[:40].astype(np.int64)).cuda()
    host = torch.empty((40, 2, Hkv, bs, D), dtype=torch.bfloat16, pin_memory=True)
    pa.gather_blocks(host, gk, gv, ids)  # swap out: device pool -> pinned host memory
    torch.cuda.synchronize()
    assert np.array_equal(_gpu.host16(host), oracle.gather_blocks(kc, vc, ids.cpu().numpy()))
    gk.zero_()
    gv.zero_()
    pa.scatter_blocks(gk, gv, host, ids)  # swap in
    idn = ids.cpu().numpy()
    assert np.array_equal(_gpu.host16(gk)[idn], kc[idn]) and np.array_equal(_gpu.host16(gv)[idn], vc[idn])


def test_block_ids_outside_the_pool_are_skipped_and_reported():
    pa = _gpu.lib()
    kc, vc = _pool(8, 2, 16, 64, "f16", 7)
    gk, gv = _dev(kc, "f16"), _dev(vc, "f16")
    prev = pa.set_check_mode(True)
    try:
        with pytest.raises(pa.PagedAttnError) as e:
            pa.copy_blocks(gk, gv, torch.tensor([[1, 2], [3, 99]], dtype=torch.int64, device="cuda"))
        assert e.value.status == -5
    finally:
        pa.set_check_mode(prev)
    want_k = kc.copy()
    want_k[2] = kc[1]
    assert np.array_equal(_gpu.host16(gk), want_k)


def test_block_manager_drives_a_decode_step_with_copy_on_write():
    pa = _gpu.lib()
    NB, Hkv, Hq, bs, D = 96, 4, 16, 16, 128
    dt = "bf16"
    bm = pa.BlockManager(NB, bs)
    kc = np.zeros((NB, Hkv, bs, D), np.uint16)
    vc = np.zeros_like(kc)
    gk, gv = _dev(kc, dt), _dev(vc, dt)
    ss = np.random.SeedSequence(11)
    rows = iter(ss.spawn(64))

    def write(slots):
        key = W.normal_bits(next(rows), (len(slots), Hkv, D), dt)
        val = W.normal_bits(next(rows), (len(slots), Hkv, D), dt)
        sl = np.array(slots, np.int64)
        oracle.reshape_and_cache(key, val, dt, kc, vc, dt, sl)
        pa.reshape_and_cache(_gpu.dev16(key, dt), _gpu.dev16(val, dt), gk, gv, torch.from_numpy(sl).cuda())

    # two prompts whose last blocks are partially filled, each forked into 3 samples
    seqs = []
    for pid, n in ((0, 40), (1, 70)):
        bm.add_sequence(pid * 10, 0)
        slots, cow = bm.append_tokens(pid * 10, n)
        assert cow is None
        write(slots)
        for c in (1, 2):
            bm.fork(pid * 10, pid * 10 + c)
        seqs += [pid * 10, pid * 10 + 1, pid * 10 + 2]
    assert bm.check() == 0
    # one decode step: every sequence appends one token; the first writers into
    # a shared partial block get a private copy first
    pairs, new_slots = [], []
    for s in seqs:
        slots, cow = bm.append_tokens(s, 1)
        if cow:
            pairs.append(cow)
        new_slots += slots
    assert len(pairs) == 4  # in each family the last block stays with the last writer
    p = np.array(pairs, np.int64)
    oracle.copy_blocks(kc, vc, p)
    pa.copy_blocks(gk, gv, torch.from_numpy(p).cuda())
    write(new_slots)
    assert bm.check() == 0
    tabs = [bm.block_table(s) for s in seqs]
    maxb = max(len(t) for t, _ in tabs)
    bt = np.full((len(seqs), maxb), -1, np.int32)
    for i, (t, _) in enumerate(tabs):
        bt[i, :len(t)] = t
    cl = np.array([n for _, n in tabs], np.int32)
    q = W.normal_bits(next(rows), (len(seqs), Hq, D), dt)
    out = torch.empty((len(seqs), Hq, D), dtype=torch.bfloat16, device="cuda")
    pa.decode(out, _gpu.dev16(q, dt), gk, gv, torch.from_numpy(bt).cuda(), torch.from_numpy(cl).cuda(), 0.088)
    assert np.array_equal(_gpu.host16(gk), kc) and np.array_equal(_gpu.host16(gv), vc)
    want = oracle.decode(q, dt, kc, vc, dt, bt, cl, 0.088)
    assert _gpu.max_err(out, want) <= _gpu.TOL["bf16"]
    # samples of one prompt share all full prefix blocks
    t0, t1 = tabs[0][0], tabs[1][0]
    assert t0[:2] == t1[:2] and t0[2] != t1[2]


def test_pageable_host_buffers_are_refused_before_launch():
    import ctypes
    pa = _gpu.lib()
    gk = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device="cuda")
    gv = torch.zeros_like(gk)
    ids = torch.tensor([0, 1], dtype=torch.int64, device="cuda")
    pageable = np.zeros(2 * 2 * gk[0].numel() * 2 + 64, np.uint8)
    addr = (pageable.ctypes.data + 15) // 16 * 16
    desc = pa.cache_desc(gk)
    rc = pa.lib.pa_gather_blocks(ctypes.c_void_p(addr), ctypes.c_void_p(gk.data_ptr()), ctypes.c_void_p(gv.data_ptr()),
                                 ctypes.byref(desc), ctypes.c_void_p(ids.data_ptr()), 2, None)
    assert rc == -1
    host_ids = np.array([0, 1], np.int64)
    rc = pa.lib.pa_copy_blocks(ctypes.c_void_p(gk.data_ptr()), ctypes.c_void_p(gv.data_ptr()), ctypes.byref(desc),
                               ctypes.c_void_p(host_ids.ctypes.data), 1, None)
    assert rc == -1
    assert pa.get_device_error() == 0
