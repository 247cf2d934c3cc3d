"""Chunked prefill on the tensor cores (pa_prefill) against the oracle: each
of the C new tokens is decoded by the oracle over the context prefix ending
at its own position (causal), through the same block table."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

CASES = [
    # (Hq, Hkv, q/kv dtype, bs, C, context lengths)
    (4, 4, "bf16", 16, 128, [128, 200, 700]),
    (8, 2, "bf16", 16, 256, [256, 300, 1000, 129]),
    (4, 1, "f16", 8, 192, [192, 450, 64]),
    (2, 2, "bf16", 32, 320, [320, 333, 1500]),
    # even groups take the two-head kernel: G = 2 (one pair) and G = 8 (four
    # pairs), several query tiles, a ragged last tile
    (4, 2, "bf16", 16, 640, [640, 700, 2000]),
    (16, 2, "f16", 32, 200, [1500, 201]),
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


def _draw(i):
    rng = np.random.default_rng(3000 + i)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.integers(1, 7))
    S = int(rng.integers(1, 4))
    C = int(rng.integers(1, 401))
    lens = [int(C + x) for x in rng.integers(0, 900, size=S)]
    return (G * Hkv, Hkv, ["f16", "bf16"][int(rng.integers(0, 2))], int(rng.choice([8, 16, 32])), C, lens)


SWEEP = [_draw(i) for i in range(12)]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: "Hq%d-Hkv%d-%s-bs%d-C%d" % c[:5])
def test_prefill_sweep_matches_oracle(case):
    """Seeded draws of group size, heads, dtype, block size, chunk length
    (ragged against the 128-row tiles) and contexts."""
    test_prefill_matches_oracle(case)


def _prefill(g, wl, bt=None, kc=None, vc=None, cl=None):
    out = torch.full_like(g.q, float("nan"))
    _gpu.lib().prefill(out, g.q, g.kc if kc is None else kc, g.vc if vc is None else vc,
                       g.bt if bt is None else bt, g.cl if cl is None else cl, wl.scale)
    torch.cuda.synchronize()
    return out


def test_full_size_bench_batch_on_sampled_rows():
    """The batch bench.py times (16 x 2048 new tokens at context 4096, 32/8
    heads, bf16, block size 16), in the same launch, checked on sampled query
    rows that the oracle evaluates one by one; every output is finite."""
    wl = W.make_prefill_workload()
    g = _gpu.OnGpu(wl)
    g.scatter()
    out = _prefill(g, wl)
    assert _gpu.lib().get_device_error() == 0
    assert torch.isfinite(out.float()).all()
    S, C = wl.S, wl.qlen
    rng = np.random.default_rng(11)
    s_idx = np.concatenate([rng.integers(0, S, 60), [0, S - 1, 5, 5, 9]])
    j_idx = np.concatenate([rng.integers(0, C, 60), [0, C - 1, 127, 128, 1919]])
    kc, vc = _gpu.oracle_pool(wl)
    q_sub = np.ascontiguousarray(wl.q[s_idx, j_idx])  # [n, Hq, D]
    L_sub = (wl.context_lens[s_idx] - C + 1 + j_idx).astype(np.int32)
    want = oracle.decode(q_sub, wl.q_dtype, kc, vc, wl.kv_dtype, np.ascontiguousarray(wl.block_tables[s_idx]),
                         L_sub, wl.scale, wl.kv_scale)
    got = out[torch.from_numpy(s_idx).cuda(), torch.from_numpy(j_idx).cuda()]
    assert _gpu.max_err(got, want) <= _gpu.tolerance(wl)


def test_unused_slots_holding_nan_are_never_read():
    """Pool slots past every context hold NaN: the last K/V tile reaches into
    them, and neither scores nor P.V may pick them up."""
    wl = W.make_workload(name="t", seed=43, context_lens=[130, 300, 17, 1000], Hq=8, Hkv=2, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16", qlen=130, fill_unused="nan")
    g = _gpu.OnGpu(wl)
    g.scatter()
    out = _prefill(g, wl)
    kc, vc = _gpu.oracle_pool(wl)
    assert _gpu.max_err(out, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)


def test_block_placement_is_bit_invariant():
    """Moving every block to another physical id changes no output bit, and
    the result is the same from run to run."""
    wl = W.make_workload(name="t", seed=44, context_lens=[256, 700, 129], Hq=8, Hkv=2, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16", qlen=256)
    g = _gpu.OnGpu(wl)
    g.scatter()
    base = _prefill(g, wl)
    assert torch.equal(_prefill(g, wl), base)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(wl.NB)).cuda()
    kc2 = torch.empty_like(g.kc)
    vc2 = torch.empty_like(g.vc)
    kc2[perm] = g.kc
    vc2[perm] = g.vc
    bt2 = torch.where(g.bt >= 0, perm[g.bt.clamp(min=0).long()].int(), g.bt)
    assert torch.equal(_prefill(g, wl, bt=bt2, kc=kc2, vc=vc2), base)


def test_single_new_token_and_empty_batch():
    wl = W.make_workload(name="t", seed=45, context_lens=[1, 64, 129], Hq=4, Hkv=2, D=128, bs=16,
                         q_dtype="f16", kv_dtype="f16", qlen=1)
    g = _gpu.OnGpu(wl)
    g.scatter()
    q = g.q.unsqueeze(1).contiguous()  # one new token: [S, 1, Hq, D]
    out = torch.full_like(q, float("nan"))
    _gpu.lib().prefill(out, q, g.kc, g.vc, g.bt, g.cl, wl.scale)
    torch.cuda.synchronize()
    kc, vc = _gpu.oracle_pool(wl)
    assert _gpu.max_err(out[:, 0], _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)
    empty = torch.empty((0, 4, 4, 128), dtype=torch.float16, device="cuda")
    _gpu.lib().prefill(empty, empty, g.kc, g.vc, g.bt[:0], g.cl[:0], wl.scale)


def test_unsupported_and_invalid_arguments_launch_nothing():
    pa = _gpu.lib()
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    cl = torch.full((1,), 4, dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 4, 2, 96), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 2, 16, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:  # head_dim 96: not built
        pa.prefill(q.clone(), q, kc, kc, bt, cl, 0.1)
    assert e.value.status == -2
    q = torch.zeros((1, 4, 2, 128), dtype=torch.bfloat16, device="cuda")
    k8 = torch.zeros((4, 2, 16, 128), dtype=torch.uint8, device="cuda")
    for bad in (0.0, -2.0, float("inf")):  # FP8 caches need a positive finite kv_scale
        with pytest.raises(pa.PagedAttnError) as e:
            pa.prefill(q.clone(), q, k8, k8, bt, cl, 0.1, kv_scale=bad)
        assert e.value.status == -1
    f16 = torch.zeros((4, 2, 16, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:  # a 16-bit cache of another dtype than q
        pa.prefill(q.clone(), q, f16, f16, bt, cl, 0.1)
    assert e.value.status == -2
    kc = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:  # 16-bit caches take kv_scale 1
        pa.prefill(q.clone(), q, kc, kc, bt, cl, 0.1, kv_scale=0.5)
    assert e.value.status == -1
    for bad in (0.0, -1.0, float("nan")):
        with pytest.raises(pa.PagedAttnError) as e:
            pa.prefill(q.clone(), q, kc, kc, bt, cl, bad)
        assert e.value.status == -1


def test_out_of_range_block_ids_are_contained_and_reported():
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=46, context_lens=[200, 300], Hq=4, Hkv=2, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16", qlen=128)
    g = _gpu.OnGpu(wl)
    g.scatter()
    assert pa.get_device_error() == 0
    bad = g.bt.clone()
    bad[1, 3] = wl.NB + 5
    out = _prefill(g, wl, bt=bad)
    assert pa.get_device_error() & pa.DEVERR_BLOCK_ID
    assert pa.get_device_error() == 0  # reading clears it
    assert torch.isfinite(out.float()).all()
    # the sequence that never touches the bad entry is unaffected
    base = _prefill(g, wl)
    assert torch.equal(out[0], base[0])


def _prefill_fp8(g, wl, bt=None):
    out = torch.full_like(g.q, float("nan"))
    _gpu.lib().prefill(out, g.q, g.kc, g.vc, g.bt if bt is None else bt, g.cl, wl.scale, wl.kv_scale)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("Hq", [8, 6], ids=["G4", "G3"])
def test_fp8_widened_blocks_with_nan_slots_and_bad_ids(Hq):
    """E4M3 caches through the widening pass (head_dim 128, an even and an odd
    group): pool slots past every context hold the E4M3 NaN code, a block id
    out of range is contained and reported, and a sequence that never touches
    it is unaffected."""
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=47, context_lens=[200, 300, 17], Hq=Hq, Hkv=2, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="fp8", qlen=130, fill_unused="nan")
    g = _gpu.OnGpu(wl)
    g.scatter()
    assert pa.get_device_error() == 0
    base = _prefill_fp8(g, wl)
    assert pa.get_device_error() == 0
    kc, vc = _gpu.oracle_pool(wl)
    assert _gpu.max_err(base, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)
    bad = g.bt.clone()
    bad[1, 3] = wl.NB + 5
    out = _prefill_fp8(g, wl, bt=bad)
    assert pa.get_device_error() & pa.DEVERR_BLOCK_ID
    assert pa.get_device_error() == 0  # reading clears it
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out[0], base[0]) and torch.equal(out[2], base[2])


def test_fp8_prefill_captured_in_a_graph_replays_the_eager_bits():
    """The E4M3 prefill path (the widening pass into a workspace allocated
    before capture, then the head-pair kernel) captured into a CUDA graph
    replays the eager launch's bits."""
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=48, context_lens=[300, 129, 700], Hq=8, Hkv=2, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="fp8", qlen=128)
    g = _gpu.OnGpu(wl)
    g.scatter()
    out = torch.full_like(g.q, float("nan"))
    ws = torch.empty(pa.prefill_workspace_size(wl.S, g.bt.shape[1], g.kc), dtype=torch.uint8, device="cuda")

    def run():
        pa.prefill(out, g.q, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale, workspace=ws)

    run()
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    eager = out.clone()
    kc, vc = _gpu.oracle_pool(wl)
    assert _gpu.max_err(eager, _gpu.oracle_out(wl, kc, vc)) <= _gpu.tolerance(wl)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        assert torch.equal(out, eager)


def test_fp8_workspace_contract():
    """With E4M3 caches: no workspace takes the packed-group kernel (in-kernel
    widening), a workspace the widening pass; both match the oracle.  A
    workspace below pa_prefill_workspace_size, or misaligned, is refused
    before any launch."""
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=49, context_lens=[256, 700], Hq=8, Hkv=2, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="fp8", qlen=256)
    g = _gpu.OnGpu(wl)
    g.scatter()
    kc, vc = _gpu.oracle_pool(wl)
    want = _gpu.oracle_out(wl, kc, vc)
    need = pa.prefill_workspace_size(wl.S, g.bt.shape[1], g.kc)
    assert need == wl.S * g.bt.shape[1] * (4 * wl.Hkv * wl.bs * wl.D + 4)
    assert pa.prefill_workspace_size(wl.S, g.bt.shape[1], g.q.new_empty((1, 1, 1, 1))) == 0  # 16-bit caches
    outs = []
    for kwargs in ({"widen": False}, {"workspace": torch.empty(need, dtype=torch.uint8, device="cuda")}):
        out = torch.full_like(g.q, float("nan"))
        pa.prefill(out, g.q, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale, **kwargs)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        assert _gpu.max_err(out, want) <= _gpu.tolerance(wl)
        outs.append(out)
    out = torch.full_like(g.q, 7.0)
    for bad in (torch.empty(need - 16, dtype=torch.uint8, device="cuda"),
                torch.empty(need + 32, dtype=torch.uint8, device="cuda")[1:need + 1]):
        with pytest.raises(pa.PagedAttnError) as e:
            pa.prefill(out, g.q, g.kc, g.vc, g.bt, g.cl, wl.scale, wl.kv_scale, workspace=bad)
        assert e.value.status == -3
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
