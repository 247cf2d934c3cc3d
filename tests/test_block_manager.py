"""The native host block manager against the paging rules the pages state:
the block invariant (review §8: every physical block is free, owned by one
logical block, or shared with a positive reference count), the waste bound
(review §11: at most block_size - 1 unused slots per sequence), fork as a
pointer update (no data copied, no block used), and copy-on-write of a shared,
partially filled last block.  Also the oracle's whole-block moves against
numpy indexing.  No GPU needed."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_230_gb300 import build

build.build()
from paged_kv_cache_230_gb300 import pagedattn as pa  # noqa: E402


def tables(bm, ids):
    return {s: bm.block_table(s) for s in ids}


def refcounts_from_tables(bm, ids):
    rc = np.zeros(bm.num_blocks, np.int64)
    for s in ids:
        for b in bm.block_table(s)[0]:
            rc[b] += 1
    return rc


def test_add_fork_append_free():
    bm = pa.BlockManager(32, 16)
    bm.add_sequence(1, 40)  # 3 blocks, last holds 8 tokens
    t1, n1 = bm.block_table(1)
    assert len(t1) == 3 and n1 == 40 and bm.num_free_blocks() == 29
    free_before = bm.num_free_blocks()
    bm.fork(1, 2)
    bm.fork(1, 3)
    assert bm.num_free_blocks() == free_before  # fork moves no data and takes no block
    assert bm.block_table(2) == (t1, 40) and all(bm.refcount(b) == 3 for b in t1)
    # appending into the shared, partially filled last block: copy-on-write
    slots, cow = bm.append_tokens(2, 1)
    t2, _ = bm.block_table(2)
    assert cow == (t1[2], t2[2]) and t2[:2] == t1[:2] and t2[2] != t1[2]
    assert slots == [t2[2] * 16 + 8]
    assert bm.refcount(t1[2]) == 2 and bm.refcount(t2[2]) == 1
    assert bm.block_table(1) == (t1, 40) and bm.block_table(3) == (t1, 40)
    # appending again to the now private block needs no copy
    slots, cow = bm.append_tokens(2, 3)
    assert cow is None and slots == [t2[2] * 16 + 9 + i for i in range(3)]
    assert bm.check() == 0
    bm.free_sequence(1)
    bm.free_sequence(3)
    assert all(bm.refcount(b) == 0 for b in [t1[2]])
    assert bm.refcount(t1[0]) == 1  # still held by sequence 2
    bm.free_sequence(2)
    assert bm.num_free_blocks() == 32 and bm.check() == 0


def test_full_shared_block_is_never_copied():
    bm = pa.BlockManager(16, 16)
    bm.add_sequence(7, 32)  # two full blocks
    bm.fork(7, 8)
    t, _ = bm.block_table(7)
    slots, cow = bm.append_tokens(8, 1)
    t8, _ = bm.block_table(8)
    assert cow is None and t8[:2] == t and len(t8) == 3 and slots == [t8[2] * 16]
    assert bm.refcount(t[0]) == 2 and bm.refcount(t[1]) == 2


def test_out_of_blocks_changes_nothing():
    bm = pa.BlockManager(4, 8)
    bm.add_sequence(1, 20)  # 3 blocks
    bm.fork(1, 2)
    before = (tables(bm, [1, 2]), bm.num_free_blocks())
    with pytest.raises(pa.PagedAttnError) as e:
        bm.append_tokens(2, 20)  # needs a copy plus 2 fresh blocks, only 1 free
    assert e.value.status == -7
    assert (tables(bm, [1, 2]), bm.num_free_blocks()) == before
    with pytest.raises(pa.PagedAttnError) as e:
        bm.add_sequence(3, 17)
    assert e.value.status == -7 and bm.check() == 0
    with pytest.raises(pa.PagedAttnError) as e:
        bm.add_sequence(1, 1)  # id in use
    assert e.value.status == -8
    with pytest.raises(pa.PagedAttnError) as e:
        bm.fork(99, 5)
    assert e.value.status == -8


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_random_operations_keep_the_invariant(bs):
    rng = np.random.default_rng(bs)
    NB = 400
    bm = pa.BlockManager(NB, bs)
    live, next_id = [], 0
    for step in range(1500):
        op = rng.integers(0, 10)
        try:
            if op < 3 or not live:
                bm.add_sequence(next_id, int(rng.integers(0, 120)))
                live.append(next_id)
                next_id += 1
            elif op < 5:
                parent = live[rng.integers(len(live))]
                bm.fork(parent, next_id)
                live.append(next_id)
                next_id += 1
            elif op < 9:
                s = live[rng.integers(len(live))]
                tb, n0 = bm.block_table(s)
                k = int(rng.integers(1, 20))
                shared_partial = n0 % bs != 0 and bm.refcount(tb[-1]) > 1
                slots, cow = bm.append_tokens(s, k)
                tb2, n1 = bm.block_table(s)
                assert n1 == n0 + k
                assert (cow is not None) == shared_partial
                if cow:
                    assert cow[0] == tb[-1] and cow[1] == tb2[len(tb) - 1]
                assert slots == [tb2[p // bs] * bs + p % bs for p in range(n0, n1)]
            else:
                s = live.pop(rng.integers(len(live)))
                bm.free_sequence(s)
        except pa.PagedAttnError as e:
            assert e.status == -7  # only running out of blocks is expected
        assert bm.check() == 0
        if step % 50 == 0:
            rc = refcounts_from_tables(bm, live)
            assert all(bm.refcount(b) == rc[b] for b in range(NB))
            assert bm.num_free_blocks() == int((rc == 0).sum())
            waste = 0
            for s in live:
                tb, n = bm.block_table(s)
                assert len(tb) == -(-n // bs)
                assert len(tb) * bs - n <= bs - 1  # at most block_size - 1 unused slots
                waste += len(tb) * bs - n
            assert bm.tail_waste() == waste


def test_oracle_block_moves_match_numpy_indexing():
    rng = np.random.default_rng(3)
    kc = rng.integers(0, 256, size=(10, 2, 4, 8), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(10, 2, 4, 8), dtype=np.uint8)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[1, 5], [2, 6], [9, 0]])
    assert oracle.copy_blocks(kc, vc, pairs) == 0
    for s, d in pairs:
        assert np.array_equal(kc[d], k0[s]) and np.array_equal(vc[d], v0[s])
    ids = np.array([3, 0, 7])
    buf = oracle.gather_blocks(kc, vc, ids)
    assert np.array_equal(buf[:, 0], kc[ids]) and np.array_equal(buf[:, 1], vc[ids])
    kz, vz = np.zeros_like(kc), np.zeros_like(vc)
    assert oracle.scatter_blocks(kz, vz, buf, ids) == 0
    assert np.array_equal(kz[ids], kc[ids]) and np.array_equal(vz[ids], vc[ids])
    assert oracle.copy_blocks(kc, vc, np.array([[11, 0]])) == 1


def fragmentation(bm, ids):
    """Unused slots at the ends of the sequences' last blocks over all slots of
    the blocks the sequences hold (shared blocks counted once)."""
    held = set()
    for s in ids:
        held.update(bm.block_table(s)[0])
    return bm.tail_waste() / (len(held) * bm.block_size)


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_fragmentation_on_the_workload_length_mixes_is_below_four_percent(idx):
    """Paging allocates per token: the review (§3 Q3, §9 "Memory Management",
    §10 table) puts the waste below 4 %, and §11 bounds it by block_size - 1
    slots per sequence.  Checked on each decode workload's length mix, with the
    shared-prefix mix built by forking prompts and appending private tails."""
    from paged_kv_cache_230_gb300 import workloads as W
    L = W.config_lengths(idx, idx)
    bs = 16
    bm = pa.BlockManager(int(sum(-(-int(n) // bs) for n in L)) + 64, bs)
    if idx == 4:
        for p in range(8):
            bm.add_sequence(10_000 + p, 2048)
        for s, n in enumerate(L):
            bm.fork(10_000 + s % 8, s)
            bm.append_tokens(s, int(n) - 2048)
        for p in range(8):
            bm.free_sequence(10_000 + p)
    else:
        for s, n in enumerate(L):
            bm.add_sequence(s, int(n))
    ids = list(range(len(L)))
    for s in ids:
        tb, n = bm.block_table(s)
        assert n == L[s] and len(tb) * bs - n <= bs - 1
    assert bm.check() == 0
    assert fragmentation(bm, ids) < 0.04
