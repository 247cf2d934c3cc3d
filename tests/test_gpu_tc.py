"""The tensor-core attention path against the oracle: chunked prefill with
head_dim 64 and 128 and every kind of query group (the group's heads packed
into the MMA rows, including group sizes that do not divide the 128 rows),
and multi-token decode whose query group is wider than the warp-MMA decode
kernel serves (G x k > 16 columns: speculative verification of 4-16 draft
tokens, and single-token decode with G > 16), one pass or split into runs of
partitions merged by log-sum-exp, with the new rows written by the fused
call or by a separate scatter."""
import numpy as np
import pytest
import torch

from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

LENS = [1, 3, 8, 15, 16, 17, 64, 65, 127, 128, 129, 511, 513, 1000, 2049]


def _check_zero_rows(out, wl):
    """New tokens whose position is negative (k > L) attend to nothing."""
    L = wl.context_lens
    for s in range(wl.S):
        for j in range(wl.qlen):
            if L[s] - wl.qlen + j < 0:
                assert torch.all(out[s, j] == 0)


PREFILL = [
    # (Hq, Hkv, D, dtype, bs, C, context lengths).  16-bit caches: an even
    # group takes the head-pair kernel (head_dim 64 or 128), an odd one the
    # one-head kernel (head_dim 128) or the packed-group kernel (head_dim 64)
    (8, 2, 64, "bf16", 16, 256, [256, 300, 1000, 129]),  # G = 4, two pairs
    (4, 4, 64, "f16", 8, 200, [200, 201, 777]),          # G = 1, packed
    (12, 4, 128, "bf16", 16, 300, [300, 650, 1200]),    # G = 3, one head per item
    (24, 4, 64, "f16", 32, 100, [100, 400]),            # G = 6, three pairs
    (64, 4, 128, "bf16", 16, 70, [70, 500, 1300]),      # G = 16, eight pairs
    (32, 1, 128, "f16", 16, 40, [40, 333]),             # G = 32 (MQA)
    (128, 1, 64, "bf16", 8, 9, [9, 100, 257]),          # G = 128, 64 pairs
    (12, 4, 64, "bf16", 16, 130, [130, 700]),           # G = 3, packed
]


def _prefill_case(Hq, Hkv, D, dt, bs, C, lens, kv_dtype=None, seed=61):
    kd = dt if kv_dtype is None else kv_dtype
    wl = W.make_workload(name="t", seed=seed, context_lens=lens, Hq=Hq, Hkv=Hkv, D=D, bs=bs, q_dtype=dt,
                         kv_dtype=kd, qlen=C)
    pa = _gpu.lib()
    g = _gpu.OnGpu(wl)
    g.scatter()
    out = torch.full_like(g.q, float("nan"))
    pa.prefill(out, g.q, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    gk, gv = g.caches_host()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    err = _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc))
    assert err <= _gpu.tolerance(wl), err
    _check_zero_rows(out, wl)
    out2 = torch.full_like(g.q, float("nan"))
    pa.prefill(out2, g.q, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale)
    assert torch.equal(out, out2)  # deterministic


@pytest.mark.parametrize("case", PREFILL, ids=lambda c: "Hq%d-Hkv%d-D%d-%s-bs%d-C%d" % c[:6])
def test_prefill_packed_groups_and_head_dims(case):
    _prefill_case(*case)


PREFILL_FP8 = [
    # (Hq, Hkv, D, q dtype, bs, C, context lengths): E4M3 caches with a per-tensor scale
    (32, 8, 128, "bf16", 16, 256, [256, 300, 1000, 129]),
    (8, 2, 64, "bf16", 16, 200, [200, 777]),
    (4, 4, 128, "f16", 8, 150, [150, 151, 600]),
    (12, 4, 64, "f16", 32, 90, [90, 400, 1100]),
    (64, 8, 128, "bf16", 16, 40, [40, 2100]),
]


@pytest.mark.parametrize("case", PREFILL_FP8, ids=lambda c: "Hq%d-Hkv%d-D%d-%s-bs%d-C%d-fp8" % c[:6])
def test_prefill_fp8_caches(case):
    _prefill_case(*case, kv_dtype="fp8", seed=65)


WIDE = [
    # (Hq, Hkv, D, dtype, k)
    (32, 8, 128, "bf16", 8),    # 32 columns: the GQA-8B shape verifying 8 draft tokens
    (64, 8, 128, "bf16", 4),    # 32 columns: the long-context shape verifying 4
    (64, 4, 128, "bf16", 4),    # G = 16: 64 columns
    (32, 1, 128, "f16", 1),     # MQA, one token: 32 columns
    (12, 4, 64, "f16", 7),      # G = 3: 21 columns
    (16, 8, 64, "bf16", 16),    # G = 2, 16 tokens: 32 columns
    (256, 2, 64, "bf16", 1),    # G = 128
]
WIDE_FP8 = [
    # (Hq, Hkv, D, q dtype, k): E4M3 caches
    (32, 8, 128, "bf16", 8),
    (64, 8, 128, "bf16", 4),
    (16, 4, 64, "f16", 6),
]


def _wide_id(c):
    return "Hq%d-Hkv%d-D%d-%s-k%d" % c


def _wide_case(case, P, fused, kv_dtype=None):
    Hq, Hkv, D, dt, k = case
    wl = W.make_workload(name="t", seed=62, context_lens=LENS, Hq=Hq, Hkv=Hkv, D=D, bs=16, q_dtype=dt,
                         kv_dtype=dt if kv_dtype is None else kv_dtype, qlen=k)
    pa = _gpu.lib()
    assert pa.get_device_error() == 0
    g = _gpu.OnGpu(wl)
    if fused:
        out = torch.full_like(g.q, float("nan"))
        pa.cache_and_decode(out, g.q, g.key, g.value, g.slots, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale,
                            max_context_len=wl.max_context_len, partition_size=P)
    else:
        out = g.step(partition_size=P).clone()
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    gk, gv = g.caches_host()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    err = _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc, partition_size=P))
    assert err <= _gpu.tolerance(wl), err
    _check_zero_rows(out, wl)
    assert torch.equal(g.decode(partition_size=P), out)  # deterministic


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two"])
@pytest.mark.parametrize("P", [0, 64, 512])
@pytest.mark.parametrize("case", WIDE, ids=_wide_id)
def test_wide_group_decode(case, P, fused):
    _wide_case(case, P, fused)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two"])
@pytest.mark.parametrize("P", [0, 128])
@pytest.mark.parametrize("case", WIDE_FP8, ids=lambda c: _wide_id(c) + "-fp8")
def test_wide_group_decode_fp8(case, P, fused):
    _wide_case(case, P, fused, kv_dtype="fp8")


def _draw(i):
    rng = np.random.default_rng(5000 + i)
    while True:
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.integers(1, 33))
        k = int(rng.integers(1, 17))
        if 16 < G * k <= 160:
            break
    dt = ["f16", "bf16"][int(rng.integers(0, 2))]
    kd = dt if rng.integers(0, 3) else "fp8"
    S = int(rng.integers(1, 6))
    return dict(Hq=G * Hkv, Hkv=Hkv, D=int(rng.choice([64, 128])), bs=int(rng.choice([8, 16, 32])), dt=dt, kd=kd, k=k,
                lens=[int(x) for x in rng.integers(1, 2500, size=S)], P=int(rng.choice([0, 64, 128, 512])),
                fused=bool(rng.integers(0, 2)), seed=6000 + i)


SWEEP = [_draw(i) for i in range(24)]


@pytest.mark.parametrize("c", SWEEP, ids=lambda c: "Hq%d-Hkv%d-D%d-bs%d-%s-%s-k%d-P%d-%s" % (
    c["Hq"], c["Hkv"], c["D"], c["bs"], c["dt"], c["kd"], c["k"], c["P"], "fused" if c["fused"] else "two"))
def test_wide_group_sweep(c):
    """Seeded draws of group size (1-32), new tokens (1-16, G x k from 17 to
    160 columns), head_dim, block size, q and cache dtype (a third E4M3),
    partition size and launch form."""
    wl = W.make_workload(name="t", seed=c["seed"], context_lens=c["lens"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"],
                         bs=c["bs"], q_dtype=c["dt"], kv_dtype=c["kd"], qlen=c["k"])
    pa = _gpu.lib()
    g = _gpu.OnGpu(wl)
    if c["fused"]:
        out = torch.full_like(g.q, float("nan"))
        pa.cache_and_decode(out, g.q, g.key, g.value, g.slots, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale,
                            max_context_len=wl.max_context_len, partition_size=c["P"])
    else:
        out = g.step(partition_size=c["P"]).clone()
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    gk, gv = g.caches_host()
    assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc, partition_size=c["P"])) <= _gpu.tolerance(wl)
    _check_zero_rows(out, wl)


def test_nan_in_unused_pool_slots_is_never_read():
    wl = W.make_workload(name="t", seed=63, context_lens=[130, 300, 17, 1000, 5], Hq=32, Hkv=8, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16", qlen=8, fill_unused="nan")
    g = _gpu.OnGpu(wl)
    out = g.step().clone()
    kc, vc = _gpu.oracle_pool(wl)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)
    out = g.step(partition_size=64).clone()
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc, partition_size=64)) <= _gpu.tolerance(wl)


@pytest.mark.parametrize("k", [8, 4])
def test_full_size_multi_token_workloads(k):
    """The benchmark's multi-token lines at full size, every output against
    the oracle: the GQA-8B batch (256 sequences) verifying 8 draft tokens (32
    columns per kv head) one pass, and the long-context batch (8 sequences,
    64/8 heads, 32K-128K tokens) verifying 4 (32 columns), split into
    512-token partitions."""
    from paged_kv_cache_230_gb300.device import DeviceBatch
    wl = W.make_config(2 if k == 8 else 3, qlen=k)
    b = DeviceBatch(wl, "cuda")
    out = b.step().clone()
    torch.cuda.synchronize()
    assert _gpu.lib().get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    err = _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc, partition_size=wl.partition_size))
    print("%s k=%d: max|gpu - oracle| = %.3g over %d outputs" % (wl.name, k, err, out.numel()))
    assert err <= _gpu.tolerance(wl), err


def test_bad_block_ids_and_context_lengths_are_contained_and_reported():
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=64, context_lens=[200, 300], Hq=32, Hkv=8, D=128, bs=16, q_dtype="bf16",
                         kv_dtype="bf16", qlen=8)
    g = _gpu.OnGpu(wl)
    g.scatter()
    assert pa.get_device_error() == 0
    base = g.decode().clone()
    bad = g.bt.clone()
    bad[1, 3] = wl.NB + 5
    out = torch.empty_like(g.q)
    pa.decode_multi(out, g.q, g.kc, g.vc, bad, g.cl, wl.scale)
    assert pa.get_device_error() & pa.DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out[0], base[0])
    cl = g.cl.clone()
    cl[0] = wl.max_blocks * wl.bs + 100  # past the table: clamped and reported
    pa.decode_multi(out, g.q, g.kc, g.vc, g.bt, cl, wl.scale)
    assert pa.get_device_error() & pa.DEVERR_CONTEXT_LEN
    assert torch.isfinite(out.float()).all()
    assert pa.get_device_error() == 0


def test_scale_must_be_positive_on_the_tensor_core_path():
    pa = _gpu.lib()
    q = torch.zeros((1, 8, 32, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    cl = torch.full((1,), 10, dtype=torch.int32, device="cuda")
    for bad in (0.0, -0.1):
        with pytest.raises(pa.PagedAttnError) as e:
            pa.decode_multi(q.clone(), q, kc, kc, bt, cl, bad)
        assert e.value.status == -1


@pytest.mark.parametrize("P", [0, 512])
def test_graph_captured_launch_replays_the_oracle_result(P):
    """The tensor-core path captured into a CUDA graph (tensor maps and
    parameters baked into the graph, the split workspace allocated before
    capture): replays give the eager launch's bits, within the oracle's
    tolerance, and agree with each other."""
    wl = W.make_workload(name="t", seed=66, context_lens=LENS + [3000, 4097], Hq=32, Hkv=8, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16", qlen=8)
    pa = _gpu.lib()
    g = _gpu.OnGpu(wl)
    g.scatter()
    eager = g.decode(partition_size=P).clone()
    torch.cuda.synchronize()
    kc, vc = _gpu.oracle_pool(wl)
    want = _gpu.oracle_out(wl, kc, vc, partition_size=P)
    assert _gpu.max_err(eager, want) <= _gpu.tolerance(wl)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g.decode(partition_size=P)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.decode(partition_size=P)
    for _ in range(2):
        g.out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        assert torch.equal(g.out, eager)
    _check_zero_rows(g.out, wl)


def test_concurrent_launches_on_many_streams_agree():
    """Launches on 80 streams at once (the kernel keeps no state between
    launches) all give the single-stream result bit for bit."""
    wl = W.make_workload(name="t", seed=67, context_lens=[700, 33, 1500], Hq=32, Hkv=8, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16", qlen=8)
    pa = _gpu.lib()
    g = _gpu.OnGpu(wl)
    g.scatter()
    ref = g.decode().clone()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(80)]
    outs = [torch.empty_like(g.q) for _ in streams]
    for s, o in zip(streams, outs):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            pa.decode_multi(o, g.q, g.kc, g.vc, g.bt, g.cl, wl.scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    for o in outs:
        assert torch.equal(o, ref)


NARROW_EDGES = [
    # (Hq, Hkv, G x k rows): the narrow instantiation serves groups of at most
    # 96 rows, its softmax warps with no live row (rows 32 w .. 32 w + 31 all
    # past the group) skipping the arithmetic
    (32, 8, 8),    # G = 4, k = 8: 32 rows, warps 1-3 of each half without a live row
    (33, 1, 1),    # G = 33, k = 1: 33 rows, one live row in the second quarter
    (16, 1, 4),    # G = 16, k = 4: 64 rows
    (32, 1, 3),    # G = 32, k = 3: 96 rows, the largest narrow group
    (97, 1, 1),    # G = 97: 97 rows, the smallest group past the narrow instantiation
]


@pytest.mark.parametrize("P", [0, 128])
@pytest.mark.parametrize("case", NARROW_EDGES, ids=lambda c: "Hq%d-Hkv%d-k%d" % c)
def test_narrow_group_edges(case, P):
    Hq, Hkv, k = case
    wl = W.make_workload(name="t", seed=68, context_lens=[1, 5, 129, 700, 1500], Hq=Hq, Hkv=Hkv, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16", qlen=k)
    pa = _gpu.lib()
    g = _gpu.OnGpu(wl)
    out = g.step(partition_size=P).clone()
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc, partition_size=P)) <= _gpu.tolerance(wl)
    _check_zero_rows(out, wl)
