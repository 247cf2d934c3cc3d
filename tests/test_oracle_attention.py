"""Pins the oracle's attention and scatter against facts that do not come from
the oracle itself: hand-worked cases (tests/golden), dense softmax attention
computed with scipy on an unpaged copy, and invariants the paging scheme must
keep (physical placement and shared prefixes do not change results)."""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_kv_cache_230_gb300 import workloads as W
from tests import _golden


# --------------------------------------------------------------------------
# hand-worked cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", [c["name"] for c in _golden.load()["cases"]])
def test_golden_cases(name):
    c = next(c for c in _golden.load()["cases"] if c["name"] == name)
    a = _golden.case_arrays(c)
    got = oracle.decode(a["q"], c["dtype"], a["k_cache"], a["v_cache"], c["kv_dtype"],
                        a["block_tables"], a["context_lens"], a["scale"], a["kv_scale"])
    np.testing.assert_allclose(got, a["expected"], rtol=0, atol=1e-12)
    if "split" in c:
        P = c["split"]["partition_size"]
        got2 = oracle.decode(a["q"], c["dtype"], a["k_cache"], a["v_cache"], c["kv_dtype"],
                             a["block_tables"], a["context_lens"], a["scale"], a["kv_scale"],
                             partition_size=P)
        np.testing.assert_allclose(got2, a["expected"], rtol=0, atol=1e-12)
        for p, want in enumerate(c["split"]["partials"]):
            L = int(a["context_lens"][0])
            m, l, o = oracle.attend_range(a["q"], c["dtype"], a["k_cache"], a["v_cache"], c["kv_dtype"],
                                          a["block_tables"], a["scale"], a["kv_scale"], 0, 0,
                                          p * P, min(L, (p + 1) * P))
            assert abs(m - _golden.scalar(want["m"])) < 1e-12
            assert abs(l - _golden.scalar(want["l"])) < 1e-12
            np.testing.assert_allclose(o, [_golden.scalar(x) for x in want["o"]], atol=1e-12)


def test_golden_scatter():
    sc = _golden.load()["scatter"]
    key = _golden.enc16(np.array(sc["key"], np.float64), sc["in_dtype"])
    value = key.copy()
    NB, bs, Hkv, D = sc["num_blocks"], sc["block_size"], sc["num_kv_heads"], sc["head_dim"]
    kc = np.full((NB, Hkv, bs, D), 0xAA, np.uint8)
    vc = kc.copy()
    bad = oracle.reshape_and_cache(key, value, sc["in_dtype"], kc, vc, "fp8",
                                   np.array(sc["slot_mapping"], np.int64), sc["kv_scale"])
    assert bad == 0
    want = np.array([int(x, 16) for x in sc["expected_codes"]], np.uint8)
    assert np.array_equal(kc[sc["expected_block"], 0, sc["expected_offset"]], want)
    assert np.array_equal(vc[sc["expected_block"], 0, sc["expected_offset"]], want)
    untouched = np.ones(kc.shape, bool)
    untouched[sc["expected_block"], 0, sc["expected_offset"]] = False
    assert np.all(kc[untouched] == 0xAA) and np.all(vc[untouched] == 0xAA)


# --------------------------------------------------------------------------
# dense brute force on an unpaged copy
# --------------------------------------------------------------------------

def dense_reference(wl, k_cache, v_cache):
    """softmax(scale q K^T) V per (sequence, query head), computed with scipy on
    K/V rows gathered into a dense [L, D] array per sequence (numpy indexing,
    float64), with query head g on kv head g // G."""
    if wl.kv_dtype == "fp8":
        kd = torch.from_numpy(k_cache).view(torch.float8_e4m3fn).double().numpy() * wl.kv_scale
        vd = torch.from_numpy(v_cache).view(torch.float8_e4m3fn).double().numpy() * wl.kv_scale
    else:
        kd = W.bits_to_f32(k_cache, wl.kv_dtype).astype(np.float64)
        vd = W.bits_to_f32(v_cache, wl.kv_dtype).astype(np.float64)
    q = W.bits_to_f32(wl.q, wl.q_dtype).astype(np.float64)
    out = np.zeros((wl.S, wl.Hq, wl.D))
    for s in range(wl.S):
        L = int(wl.context_lens[s])
        if L == 0:
            continue
        i = np.arange(L)
        phys = wl.block_tables[s, i // wl.bs]
        for g in range(wl.Hq):
            h = g // wl.G
            K = kd[phys, h, i % wl.bs, :]
            V = vd[phys, h, i % wl.bs, :]
            p = scipy.special.softmax(wl.scale * (K @ q[s, g]))
            out[s, g] = p @ V
    return out


def _filled(wl):
    """Pool contents after this step's scatter, via the oracle."""
    if wl.kv_dtype == "fp8":
        kc = np.zeros(wl.cache_shape(), np.uint8)
        vc = np.zeros(wl.cache_shape(), np.uint8)
        oracle.reshape_and_cache(wl.prefill_key, wl.prefill_value, wl.q_dtype, kc, vc, "fp8",
                                 wl.prefill_slots, wl.kv_scale)
    else:
        kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.reshape_and_cache(wl.key, wl.value, wl.q_dtype, kc, vc, wl.kv_dtype, wl.slot_mapping, wl.kv_scale)
    return kc, vc


def _decode(wl, kc, vc, P=0):
    return oracle.decode(wl.q, wl.q_dtype, kc, vc, wl.kv_dtype, wl.block_tables, wl.context_lens,
                         wl.scale, wl.kv_scale, partition_size=P)


SMALL = [
    dict(Hq=4, Hkv=4, D=64, q_dtype="f16", kv_dtype="f16", lens=[1, 15, 16, 17, 40]),
    dict(Hq=8, Hkv=2, D=64, q_dtype="bf16", kv_dtype="bf16", lens=[33, 7, 64, 2]),
    dict(Hq=4, Hkv=1, D=32, q_dtype="bf16", kv_dtype="fp8", lens=[5, 50, 31]),
    dict(Hq=6, Hkv=2, D=16, q_dtype="f16", kv_dtype="fp8", lens=[3, 48]),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: "%s-%s-G%d" % (c["q_dtype"], c["kv_dtype"], c["Hq"] // c["Hkv"]))
@pytest.mark.parametrize("bs", [8, 16])
def test_paged_equals_dense_bruteforce(cfg, bs):
    wl = W.make_workload(name="t", seed=11, context_lens=cfg["lens"], Hq=cfg["Hq"], Hkv=cfg["Hkv"],
                         D=cfg["D"], bs=bs, q_dtype=cfg["q_dtype"], kv_dtype=cfg["kv_dtype"])
    kc, vc = _filled(wl)
    got = _decode(wl, kc, vc)
    want = dense_reference(wl, kc, vc)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_contiguous_table_equals_dense_without_any_indexing():
    """Identity block table: token i is row i of a [L, D] array reshaped straight
    out of the pool, no block-table lookup on the reference side."""
    rng = np.random.default_rng(5)
    D, bs, L = 32, 16, 80
    nb = L // bs
    kf = rng.standard_normal((nb, 1, bs, D)).astype(np.float16)
    vf = rng.standard_normal((nb, 1, bs, D)).astype(np.float16)
    q = rng.standard_normal((1, 1, D)).astype(np.float16)
    bt = np.arange(nb, dtype=np.int32)[None]
    got = oracle.decode(q.view(np.uint16), "f16", kf.view(np.uint16), vf.view(np.uint16), "f16", bt,
                        np.array([L], np.int32), 0.3)
    K = kf.astype(np.float64).reshape(L, D)
    V = vf.astype(np.float64).reshape(L, D)
    p = scipy.special.softmax(0.3 * K @ q.astype(np.float64)[0, 0])
    np.testing.assert_allclose(got[0, 0], p @ V, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------
# invariants of the paging scheme
# --------------------------------------------------------------------------

def test_physical_permutation_is_bit_invariant():
    wl = W.make_workload(name="t", seed=3, context_lens=[100, 1, 37, 64], Hq=8, Hkv=2, D=32, bs=16,
                         q_dtype="bf16", kv_dtype="bf16")
    kc, vc = _filled(wl)
    base = _decode(wl, kc, vc)
    perm = np.random.default_rng(9).permutation(wl.NB)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    got = oracle.decode(wl.q, wl.q_dtype, kc2, vc2, wl.kv_dtype, bt2, wl.context_lens, wl.scale)
    assert np.array_equal(got, base)


def test_shared_prefix_equals_unshared_copies():
    lens = [2048 // 8 + 1 + t for t in (0, 5, 17, 40, 3, 9)]
    wl = W.make_workload(name="t", seed=4, context_lens=lens, Hq=4, Hkv=2, D=16, bs=8, q_dtype="bf16",
                         kv_dtype="fp8", shared_prefix=(2, 256))
    counts = W.check_block_table_invariant(wl.block_tables, wl.context_lens, wl.bs, wl.NB)
    assert counts.max() == 3  # each prompt's blocks are shared by its 3 sequences
    kc, vc = _filled(wl)
    base = _decode(wl, kc, vc)
    # give every sequence private copies of the blocks it shares
    NB2 = wl.NB + int((wl.block_tables >= 0).sum())
    kc2 = np.zeros((NB2,) + kc.shape[1:], kc.dtype)
    vc2 = np.zeros_like(kc2)
    kc2[:wl.NB], vc2[:wl.NB] = kc, vc
    bt2 = wl.block_tables.copy()
    nxt = wl.NB
    for s in range(wl.S):
        for j in range(256 // wl.bs):
            b = wl.block_tables[s, j]
            kc2[nxt], vc2[nxt] = kc[b], vc[b]
            bt2[s, j] = nxt
            nxt += 1
    assert W.check_block_table_invariant(bt2, wl.context_lens, wl.bs, NB2).max() == 1
    got = oracle.decode(wl.q, wl.q_dtype, kc2, vc2, wl.kv_dtype, bt2, wl.context_lens, wl.scale, wl.kv_scale)
    assert np.array_equal(got, base)


def test_single_token_context_returns_its_value():
    wl = W.make_workload(name="t", seed=6, context_lens=[1, 1, 1], Hq=4, Hkv=2, D=32, bs=16,
                         q_dtype="f16", kv_dtype="f16")
    kc, vc = _filled(wl)
    got = _decode(wl, kc, vc)
    for s in range(wl.S):
        b = wl.block_tables[s, 0]
        for g in range(wl.Hq):
            want = W.bits_to_f32(vc[b, g // wl.G, 0], "f16").astype(np.float64)
            assert np.array_equal(got[s, g], want)


def test_zero_query_and_constant_keys_give_mean_of_values():
    wl = W.make_workload(name="t", seed=7, context_lens=[70, 5, 129], Hq=4, Hkv=4, D=32, bs=16,
                         q_dtype="bf16", kv_dtype="bf16")
    kc, vc = _filled(wl)
    vals = []
    for s in range(wl.S):
        L = int(wl.context_lens[s])
        i = np.arange(L)
        V = W.bits_to_f32(vc[wl.block_tables[s, i // 16], :, i % 16, :], "bf16").astype(np.float64)
        vals.append(V.mean(axis=0))  # [Hkv, D]
    zq = np.zeros_like(wl.q)
    got = oracle.decode(zq, "bf16", kc, vc, "bf16", wl.block_tables, wl.context_lens, wl.scale)
    for s in range(wl.S):
        np.testing.assert_allclose(got[s], vals[s], rtol=1e-13, atol=1e-15)
    # every key row equal (a constant row), any query: scores are equal, output is the mean
    kconst = np.broadcast_to(kc[:1, :, :1, :], kc.shape).copy()
    got2 = oracle.decode(wl.q, "bf16", kconst, vc, "bf16", wl.block_tables, wl.context_lens, wl.scale)
    for s in range(wl.S):
        np.testing.assert_allclose(got2[s], vals[s], rtol=1e-13, atol=1e-15)


def test_gqa_equals_mha_with_replicated_kv_heads():
    wl = W.make_workload(name="t", seed=8, context_lens=[50, 17, 90], Hq=8, Hkv=2, D=32, bs=16,
                         q_dtype="bf16", kv_dtype="bf16")
    kc, vc = _filled(wl)
    gqa = _decode(wl, kc, vc)
    rep_k = np.ascontiguousarray(np.repeat(kc, wl.G, axis=1))
    rep_v = np.ascontiguousarray(np.repeat(vc, wl.G, axis=1))
    mha = oracle.decode(wl.q, "bf16", rep_k, rep_v, "bf16", wl.block_tables, wl.context_lens, wl.scale)
    assert np.array_equal(gqa, mha)
    # and the kv heads really differ, so a wrong head mapping would be caught
    assert not np.allclose(gqa[:, 0], gqa[:, wl.G])


def test_split_equals_unsplit():
    wl = W.make_workload(name="t", seed=10, context_lens=[1, 511, 512, 513, 2000, 64], Hq=4, Hkv=2, D=32,
                         bs=16, q_dtype="bf16", kv_dtype="bf16")
    kc, vc = _filled(wl)
    base = _decode(wl, kc, vc)
    for P in (64, 512):
        got = _decode(wl, kc, vc, P)
        np.testing.assert_allclose(got, base, rtol=1e-12, atol=1e-14)
    # one partition that covers every context is the unsplit computation exactly
    assert np.array_equal(_decode(wl, kc, vc, 4096), base)


def test_lse_merge_is_order_invariant():
    wl = W.make_workload(name="t", seed=12, context_lens=[777], Hq=2, Hkv=1, D=16, bs=16,
                         q_dtype="bf16", kv_dtype="bf16")
    kc, vc = _filled(wl)
    P = 64
    L = 777
    parts = [oracle.attend_range(wl.q, "bf16", kc, vc, "bf16", wl.block_tables, wl.scale, 1.0, 0, 1,
                                 t, min(L, t + P)) for t in range(0, L, P)]
    want = _decode(wl, kc, vc, P)[0, 1]
    for seed in range(4):
        order = np.random.default_rng(seed).permutation(len(parts))
        M = max(parts[i][0] for i in order)
        num = sum(parts[i][2] * math.exp(parts[i][0] - M) for i in order)
        den = sum(parts[i][1] * math.exp(parts[i][0] - M) for i in order)
        np.testing.assert_allclose(num / den, want, rtol=1e-12)


def test_scatter_copies_and_skips():
    wl = W.make_workload(name="t", seed=13, context_lens=[5, 16, 33], Hq=4, Hkv=2, D=16, bs=8,
                         q_dtype="f16", kv_dtype="f16")
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    slots = wl.slot_mapping.copy()
    slots[1] = -1
    bad = oracle.reshape_and_cache(wl.key, wl.value, "f16", kc, vc, "f16", slots)
    assert bad == 0
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        assert np.array_equal(kc[sl // 8, :, sl % 8, :], wl.key[t])
        assert np.array_equal(vc[sl // 8, :, sl % 8, :], wl.value[t])
    changed = (kc != wl.k_cache).any(axis=(1, 3))  # [NB, bs]
    assert changed.sum() <= 2
    # a slot outside the pool is counted and skipped
    kc3, vc3 = wl.k_cache.copy(), wl.v_cache.copy()
    bad = oracle.reshape_and_cache(wl.key, wl.value, "f16", kc3, vc3, "f16",
                                   np.array([wl.NB * 8, -5, wl.NB * 8 + 100], np.int64))
    assert bad == 2 and np.array_equal(kc3, wl.k_cache)


def test_fp8_scatter_matches_torch_quantisation():
    wl = W.make_workload(name="t", seed=14, context_lens=[9, 40], Hq=4, Hkv=2, D=32, bs=16,
                         q_dtype="bf16", kv_dtype="fp8")
    kc = np.zeros(wl.cache_shape(), np.uint8)
    vc = np.zeros(wl.cache_shape(), np.uint8)
    oracle.reshape_and_cache(wl.key, wl.value, "bf16", kc, vc, "fp8", wl.slot_mapping, wl.kv_scale)
    x = W.bits_to_f32(wl.key, "bf16")
    y = (x / np.float32(wl.kv_scale)).astype(np.float32)  # float32 division, as stated
    assert np.abs(y).max() < 448  # the per-tensor scale keeps values in range
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t, sl in enumerate(wl.slot_mapping):
        assert np.array_equal(kc[sl // 16, :, sl % 16, :], want[t])


def test_configs_satisfy_block_table_invariant():
    for idx in (0, 1, 4):
        wl = W.make_config(idx)
        counts = W.check_block_table_invariant(wl.block_tables, wl.context_lens, wl.bs, wl.NB)
        if idx == 4:
            assert counts.max() == 16  # 16 sequences fork from each prompt
        else:
            assert counts.max() == 1
        assert np.all(wl.slot_mapping // wl.bs == wl.block_tables[np.arange(wl.S), (wl.context_lens - 1) // wl.bs])
    L = W.config_lengths(2, 2)
    assert len(L) == 256 and L.min() >= 16 and L.max() <= 8192
    assert 600 < np.median(L) < 1600
    L = W.config_lengths(3, 3)
    assert len(L) == 8 and L.min() >= 32768 and L.max() <= 131072


def test_fp8_config_scale_covers_every_value():
    wl = W.make_config(4)
    amax = max(np.abs(W.bits_to_f32(a, "bf16")).max() for a in (wl.prefill_key, wl.prefill_value, wl.key, wl.value))
    assert wl.kv_scale == float(np.float32(amax) / np.float32(448.0))


def test_multi_token_reading_is_causal_dense_attention():
    """The tests' oracle for k new tokens (each new token decoded over the
    context prefix ending at its own position) equals dense causal attention
    computed with scipy on the unpaged rows."""
    from tests import _gpu
    k = 3
    wl = W.make_workload(name="t", seed=15, context_lens=[2, 9, 40], Hq=4, Hkv=2, D=16, bs=8, q_dtype="bf16",
                         kv_dtype="bf16", qlen=k)
    kc, vc = _filled(wl)
    got = _gpu.oracle_out(wl, kc, vc)
    q = W.bits_to_f32(wl.q, "bf16").astype(np.float64)  # [S, k, Hq, D]
    kd = W.bits_to_f32(kc, "bf16").astype(np.float64)
    vd = W.bits_to_f32(vc, "bf16").astype(np.float64)
    for s in range(wl.S):
        L = int(wl.context_lens[s])
        i = np.arange(L)
        phys = wl.block_tables[s, i // wl.bs]
        for j in range(k):
            pos = L - k + j
            for g in range(wl.Hq):
                if pos < 0:
                    assert np.all(got[s, j, g] == 0)
                    continue
                K = kd[phys, g // wl.G, i % wl.bs, :][: pos + 1]
                V = vd[phys, g // wl.G, i % wl.bs, :][: pos + 1]
                p = scipy.special.softmax(wl.scale * (K @ q[s, j, g]))
                np.testing.assert_allclose(got[s, j, g], p @ V, rtol=1e-12, atol=1e-13)
    # the scatter writes the k new rows at positions L - k .. L - 1
    for s in range(wl.S):
        for j in range(k):
            pos = int(wl.context_lens[s]) - k + j
            sl = wl.slot_mapping[s * k + j]
            if pos < 0:
                assert sl == -1
            else:
                assert sl == wl.block_tables[s, pos // wl.bs] * wl.bs + pos % wl.bs
