"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays out block tables; it holds none
of the attention or quantisation arithmetic.  Both the CPU oracle tests and the
CUDA path take their inputs from here, so the two sides always see the same
bytes.

What the inputs model (vLLM web pages, "vllm-project-vllm" review, §3 Q2 and
§6 "KV Cache Block Tables"): a pool of fixed-size physical KV blocks, a per
sequence block table mapping logical block j to a physical block id, blocks
allocated without contiguity, blocks shared between sequences that fork from
one prompt, and one new token per sequence per decode step.

Value recipe: every K, V and q element is a standard normal draw, stored as
fp16 (numpy round-to-nearest cast) or bf16 (upper 16 bits of the float32
draw).  The draws come from numpy PCG64 streams spawned from one
``SeedSequence(seed)`` in fixed 1 Mi-element chunks, so the bytes depend only
on the seed and the shapes, never on the thread count.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

F16, BF16, FP8 = "f16", "bf16", "fp8"
DTYPE_CODE = {F16: 0, BF16: 1, FP8: 2}
ELEM_BYTES = {F16: 2, BF16: 2, FP8: 1}
E4M3_MAX = 448.0  # largest finite OCP FP8 E4M3 value

_CHUNK = 1 << 20


def _normal_f32(seed_seq: np.random.SeedSequence, n: int) -> np.ndarray:
    """n standard-normal float32 draws, chunked so the stream is thread-count independent."""
    out = np.empty(n, dtype=np.float32)
    nchunks = max(1, (n + _CHUNK - 1) // _CHUNK)
    kids = seed_seq.spawn(nchunks)

    def fill(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        if lo < hi:
            g = np.random.Generator(np.random.PCG64(kids[i]))
            g.standard_normal(out=out[lo:hi], dtype=np.float32)

    workers = min(16, os.cpu_count() or 1, nchunks)
    if workers <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def normal_bits(seed_seq: np.random.SeedSequence, shape, dtype: str) -> np.ndarray:
    """Standard-normal values as raw 16-bit patterns of ``dtype`` (f16 or bf16)."""
    n = int(np.prod(shape))
    x = _normal_f32(seed_seq, n)
    if dtype == F16:
        bits = x.astype(np.float16).view(np.uint16)
    elif dtype == BF16:
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    else:
        raise ValueError(dtype)
    return bits.reshape(shape)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of f16/bf16 bit patterns to float32 (a format change, no arithmetic)."""
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


@dataclass
class Workload:
    """One decode step's inputs in the library's layouts (all host numpy arrays).

    Layouts: q ``[S, Hq, D]`` (``[S, qlen, Hq, D]`` when qlen > 1); key/value
    (this step's tokens) ``[S * qlen, Hkv, D]``;
    caches ``[NB, Hkv, bs, D]``; block_tables ``int32 [S, max_blocks]``
    (entries past ceil(L/bs) are -1); context_lens ``int32 [S]`` (includes this
    step's tokens); slot_mapping ``int64 [S * qlen]`` (token j of sequence s at
    position L - qlen + j; -1 where that position is negative).

    For 16-bit caches ``k_cache``/``v_cache`` hold the full pool contents.  For
    FP8 caches they are None and the pool is filled by scattering
    ``prefill_key``/``prefill_value`` (16-bit, ``[Tp, Hkv, D]``) into
    ``prefill_slots`` with each implementation's own reshape_and_cache.
    """

    name: str
    S: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    NB: int
    q_dtype: str
    kv_dtype: str
    q: np.ndarray
    key: np.ndarray
    value: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    slot_mapping: np.ndarray
    scale: float
    kv_scale: float = 1.0
    k_cache: Optional[np.ndarray] = None
    v_cache: Optional[np.ndarray] = None
    prefill_key: Optional[np.ndarray] = None
    prefill_value: Optional[np.ndarray] = None
    prefill_slots: Optional[np.ndarray] = None
    partition_size: int = 0
    qlen: int = 1
    notes: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def in_dtype(self) -> str:
        """dtype of the new key/value rows (the q dtype)."""
        return self.q_dtype

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.S else 0

    def cache_shape(self):
        return (self.NB, self.Hkv, self.bs, self.D)

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one decode call reads: every context token's K and V
        row of each kv head, once (shared by the G query heads)."""
        return int(self.context_lens.astype(np.int64).sum()) * self.Hkv * self.D * 2 * ELEM_BYTES[self.kv_dtype]

    def algorithmic_bytes(self) -> int:
        """KV bytes + q in + out + block-table entries used + context lengths."""
        nblk = int(((self.context_lens.astype(np.int64) + self.bs - 1) // self.bs).sum())
        return self.kv_bytes() + self.S * self.qlen * self.Hq * self.D * 2 * 2 + nblk * 4 + self.S * 4

    def scatter_bytes(self) -> int:
        """reshape_and_cache bytes: new K/V rows read + cache rows written + slot ids."""
        rows = int((self.slot_mapping >= 0).sum()) * self.Hkv * self.D
        return rows * 2 * 2 + rows * 2 * ELEM_BYTES[self.kv_dtype] + len(self.slot_mapping) * 8


# ---------------------------------------------------------------------------
# block tables
# ---------------------------------------------------------------------------

def check_block_table_invariant(block_tables, context_lens, bs, NB, refcount=None):
    """Checks the pool invariant stated for vLLM's block manager (web page
    "vllm-project-vllm", §8): every physical block is free, owned by exactly one
    logical block, or shared with a positive reference count.  Also checks the
    waste bound of §11 step 2 (at most bs-1 unused slots per sequence): each
    sequence uses exactly ceil(L/bs) blocks.  Returns the per-block refcount."""
    S = len(context_lens)
    counts = np.zeros(NB, dtype=np.int64)
    for s in range(S):
        L = int(context_lens[s])
        nb = (L + bs - 1) // bs
        assert nb * bs - L <= bs - 1
        row = block_tables[s, :nb]
        assert np.all((row >= 0) & (row < NB)), "block id out of pool"
        assert len(set(row.tolist())) == nb, "a sequence maps two logical blocks to one physical block"
        np.add.at(counts, row, 1)
        assert np.all(block_tables[s, nb:] == -1)
    if refcount is not None:
        assert np.array_equal(counts, refcount)
    return counts


def _slots_for_last_tokens(block_tables, context_lens, bs, qlen=1):
    """Slots of the last qlen positions of every context, [S * qlen] (-1 where
    the position is negative)."""
    L = context_lens.astype(np.int64)
    S = len(L)
    pos = L[:, None] - qlen + np.arange(qlen)[None, :]  # [S, qlen]
    posc = np.maximum(pos, 0)
    phys = block_tables[np.arange(S)[:, None], posc // bs].astype(np.int64)
    return np.where(pos >= 0, phys * bs + posc % bs, -1).reshape(-1)


def make_workload(
    *,
    name: str,
    seed: int,
    context_lens,
    Hq: int,
    Hkv: int,
    D: int,
    bs: int = 16,
    q_dtype: str = BF16,
    kv_dtype: str = BF16,
    max_blocks: Optional[int] = None,
    NB: Optional[int] = None,
    spare: float = 0.05,
    shared_prefix: Optional[tuple] = None,
    scale: Optional[float] = None,
    partition_size: int = 0,
    fill_unused: str = "normal",
    qlen: int = 1,
) -> Workload:
    """Builds a seeded workload.

    ``shared_prefix=(n_prompts, prefix_tokens)`` makes sequence s fork from
    prompt ``s % n_prompts`` (consecutive groups when S is a multiple): the
    prompt's ``prefix_tokens // bs`` whole blocks are shared by every sequence
    of that prompt; the rest of each context is private.  ``fill_unused``
    chooses what the pool holds outside live tokens: "normal" draws or "nan"
    (all-ones bit patterns) to prove they are never read into a result.
    """
    ss = np.random.SeedSequence(seed)
    s_tab, s_q, s_kv, s_new, s_pre = ss.spawn(5)
    rng = np.random.Generator(np.random.PCG64(s_tab))
    L = np.asarray(context_lens, dtype=np.int32)
    S = len(L)
    assert Hq % Hkv == 0
    if kv_dtype != FP8:
        assert kv_dtype == q_dtype, "16-bit caches hold the q dtype"
    nblk = (L.astype(np.int64) + bs - 1) // bs
    if max_blocks is None:
        max_blocks = int(nblk.max()) if S else 1
    assert S == 0 or int(nblk.max()) <= max_blocks

    # logical -> physical assignment
    shared_blocks = 0
    owner_prompt = None
    if shared_prefix is not None:
        n_prompts, prefix_tokens = shared_prefix
        assert prefix_tokens % bs == 0
        shared_blocks = prefix_tokens // bs
        per = max(1, S // n_prompts)
        owner_prompt = np.minimum(np.arange(S) // per, n_prompts - 1)
        assert np.all(nblk >= shared_blocks)
        unique = n_prompts * shared_blocks + int((nblk - shared_blocks).sum())
    else:
        unique = int(nblk.sum())
    if NB is None:
        NB = max(1, int(math.ceil(unique * (1.0 + spare))))
    assert NB >= unique
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((S, max_blocks), -1, dtype=np.int32)
    nxt = 0
    if shared_prefix is not None:
        prompt_blocks = []
        for p in range(shared_prefix[0]):
            prompt_blocks.append(perm[nxt:nxt + shared_blocks])
            nxt += shared_blocks
        for s in range(S):
            bt[s, :shared_blocks] = prompt_blocks[owner_prompt[s]]
            k = int(nblk[s]) - shared_blocks
            bt[s, shared_blocks:shared_blocks + k] = perm[nxt:nxt + k]
            nxt += k
    else:
        for s in range(S):
            k = int(nblk[s])
            bt[s, :k] = perm[nxt:nxt + k]
            nxt += k

    slot_mapping = _slots_for_last_tokens(bt, L, bs, qlen) if S else np.zeros(0, np.int64)
    q = normal_bits(s_q, (S, Hq, D) if qlen == 1 else (S, qlen, Hq, D), q_dtype)
    s_key, s_value = s_new.spawn(2)
    key = normal_bits(s_key, (S * qlen, Hkv, D), q_dtype)
    value = normal_bits(s_value, (S * qlen, Hkv, D), q_dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(D)

    wl = Workload(name=name, S=S, Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, q_dtype=q_dtype,
                  kv_dtype=kv_dtype, q=q, key=key, value=value, block_tables=bt,
                  context_lens=L, slot_mapping=slot_mapping.astype(np.int64), scale=float(scale),
                  partition_size=partition_size, qlen=qlen)

    if kv_dtype != FP8:
        shape = (NB, Hkv, bs, D)
        if fill_unused == "nan":
            kc = np.full(shape, 0xFFFF, dtype=np.uint16)
            vc = np.full(shape, 0xFFFF, dtype=np.uint16)
            # live tokens only (all but the one this step writes)
            live = _live_slots(bt, L - qlen, bs)
            s_k, s_v = s_kv.spawn(2)
            kd = normal_bits(s_k, (len(live), Hkv, D), kv_dtype)
            vd = normal_bits(s_v, (len(live), Hkv, D), kv_dtype)
            blk, off = live // bs, live % bs
            kc[blk, :, off, :] = kd
            vc[blk, :, off, :] = vd
        else:
            kv = s_kv.spawn(2)
            kc = normal_bits(kv[0], shape, kv_dtype)
            vc = normal_bits(kv[1], shape, kv_dtype)
        wl.k_cache, wl.v_cache = kc, vc
        wl.kv_scale = 1.0
    else:
        # Every live token (all but the one this step writes) gets 16-bit K/V
        # draws that are scattered into the FP8 pool before the step.
        live = _live_slots(bt, L - qlen, bs)
        s_k, s_v = s_pre.spawn(2)
        pk = normal_bits(s_k, (len(live), Hkv, D), q_dtype)
        pv = normal_bits(s_v, (len(live), Hkv, D), q_dtype)
        wl.prefill_key, wl.prefill_value, wl.prefill_slots = pk, pv, live.astype(np.int64)
        # Per-tensor scale: the largest magnitude over every K and V value that
        # will be stored, divided by the largest E4M3 value, in float32.
        amax = np.float32(0.0)
        for arr in (pk, pv, key, value):
            if arr.size:
                amax = max(amax, np.abs(bits_to_f32(arr, q_dtype)).max())
        wl.kv_scale = float(np.float32(amax) / np.float32(E4M3_MAX)) if amax > 0 else 1.0
        if fill_unused == "nan":
            wl.notes["fill_unused"] = "nan"
    wl.notes["unique_blocks"] = unique
    return wl


def _live_slots(bt, n_tokens, bs):
    """Distinct physical slots holding tokens [0, n_tokens[s]) of every sequence."""
    slots = []
    for s in range(bt.shape[0]):
        n = int(n_tokens[s])
        if n <= 0:
            continue
        i = np.arange(n, dtype=np.int64)
        slots.append(bt[s, i // bs].astype(np.int64) * bs + i % bs)
    if not slots:
        return np.zeros(0, np.int64)
    return np.unique(np.concatenate(slots))


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

CONFIG_NAMES = ["tiny", "mha7b", "gqa8b", "long_split", "prefix_fp8"]


def config_lengths(idx: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1000 + idx])))
    if idx == 0:
        return rng.integers(1, 200, size=4, endpoint=True).astype(np.int32)
    if idx == 1:
        return rng.integers(512, 2048, size=64, endpoint=True).astype(np.int32)
    if idx == 2:
        x = np.exp(rng.normal(math.log(1000.0), 1.0, size=256))
        return np.clip(np.rint(x), 16, 8192).astype(np.int32)
    if idx == 3:
        return rng.integers(32768, 131072, size=8, endpoint=True).astype(np.int32)
    if idx == 4:
        tails = rng.integers(0, 512, size=128, endpoint=True)
        return (2048 + tails + 1).astype(np.int32)
    raise ValueError(idx)


def make_config(idx: int, seed: Optional[int] = None, fill_unused: str = "normal", qlen: int = 1) -> Workload:
    """The five decode workloads:

    0 tiny: 4 seqs, 8/8 heads, D 64, fp16, L ~ U{1..200}, pool of 64 blocks.
    1 mha7b: 64 seqs, 32/32 heads, D 128, fp16, L ~ U{512..2048}, pool 8192.
    2 gqa8b: 256 seqs, 32/8 heads, D 128, bf16, L ~ lognormal(ln 1000, 1) clipped [16, 8192].
    3 long_split: 8 seqs, 64/8 heads, D 128, bf16, L ~ U{32768..131072}, 512-token partitions.
    4 prefix_fp8: 128 seqs forked from 8 prompts of 2048 shared tokens, private
      tails U{0..512} plus the new token, 32/8 heads, D 128, E4M3 KV, bf16 q.
    """
    seed = idx if seed is None else seed
    L = config_lengths(idx, seed)
    common = dict(name=CONFIG_NAMES[idx] if qlen == 1 else "%s_q%d" % (CONFIG_NAMES[idx], qlen), seed=seed,
                  context_lens=L, bs=16, fill_unused=fill_unused, qlen=qlen)
    if idx == 0:
        return make_workload(Hq=8, Hkv=8, D=64, q_dtype=F16, kv_dtype=F16, max_blocks=13, NB=64, **common)
    if idx == 1:
        return make_workload(Hq=32, Hkv=32, D=128, q_dtype=F16, kv_dtype=F16, max_blocks=128, NB=8192, **common)
    if idx == 2:
        return make_workload(Hq=32, Hkv=8, D=128, q_dtype=BF16, kv_dtype=BF16, max_blocks=512, **common)
    if idx == 3:
        return make_workload(Hq=64, Hkv=8, D=128, q_dtype=BF16, kv_dtype=BF16, max_blocks=8192,
                             partition_size=512, **common)
    if idx == 4:
        return make_workload(Hq=32, Hkv=8, D=128, q_dtype=BF16, kv_dtype=FP8, max_blocks=161,
                             shared_prefix=(8, 2048), **common)
    raise ValueError(idx)


def make_prefill_workload(S: int = 16, C: int = 2048, bs: int = 16, seed: int = 7,
                          fill_unused: str = "normal", kv_dtype: str = BF16, D: int = 128) -> Workload:
    """The chunked-prefill batch: S sequences, each with a chunk of C new
    tokens at the end of a context of 2C (so every query attends to between
    C + 1 and 2C tokens), GQA-8B heads (32 query / 8 kv heads), head_dim D
    (128 by default), bf16 q, bf16 or E4M3 caches, block size bs."""
    name = "prefill_gqa8b" + ("_fp8" if kv_dtype == FP8 else "") + ("" if D == 128 else "_d%d" % D)
    return make_workload(name=name, seed=seed, context_lens=[2 * C] * S, Hq=32, Hkv=8, D=D, bs=bs,
                         q_dtype=BF16, kv_dtype=kv_dtype, qlen=C, fill_unused=fill_unused)


def subset(wl: Workload, seqs) -> Workload:
    """The same pool with only the chosen sequences (for sampled oracle checks)."""
    seqs = np.asarray(seqs, dtype=np.int64)
    out = Workload(**{k: getattr(wl, k) for k in wl.__dataclass_fields__})
    out.S = len(seqs)
    out.q = np.ascontiguousarray(wl.q[seqs])
    tok = (seqs[:, None] * wl.qlen + np.arange(wl.qlen)[None, :]).reshape(-1)
    out.key = np.ascontiguousarray(wl.key[tok])
    out.value = np.ascontiguousarray(wl.value[tok])
    out.block_tables = np.ascontiguousarray(wl.block_tables[seqs])
    out.context_lens = np.ascontiguousarray(wl.context_lens[seqs])
    out.slot_mapping = np.ascontiguousarray(wl.slot_mapping[tok])
    return out
