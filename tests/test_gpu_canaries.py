"""No kernel writes outside its buffers: every buffer the library writes (the
outputs, the KV pool, the split workspace, the pinned swap buffer) sits inside
a larger allocation whose guard bytes on both sides are checked after each
call, with valid inputs and with out-of-range block ids and slots."""
import numpy as np
import pytest
import torch

from paged_kv_cache_230_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side (keeps every buffer 16-byte aligned)
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` / `dtype` with guard bytes before and after it."""

    def __init__(self, like: torch.Tensor, pinned_host: bool = False):
        n = like.numel() * like.element_size()
        self.n = n
        if pinned_host:
            self.raw = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, pin_memory=True)
        else:
            self.raw = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(like.dtype).view(like.shape)
        self.t.copy_(like)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return bool(torch.all(self.raw[:GUARD] == PATTERN)) and bool(torch.all(self.raw[GUARD + self.n:] == PATTERN))


def _guarded_batch(wl):
    g = _gpu.OnGpu(wl)
    names = ("q", "key", "value", "kc", "vc", "bt", "cl", "slots", "out")
    return g, {n: Guarded(getattr(g, n)) for n in names}


@pytest.mark.parametrize("bad_indices", [False, True], ids=["valid", "out-of-range"])
def test_writes_stay_inside_their_buffers(bad_indices):
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=61, context_lens=[1, 17, 200, 513, 1000], Hq=32, Hkv=8, D=128, bs=16,
                         q_dtype="bf16", kv_dtype="bf16", qlen=1)
    g, b = _guarded_batch(wl)
    if bad_indices:
        b["bt"].t[2, 3] = wl.NB + 9
        b["slots"].t[4] = wl.NB * wl.bs + 1
    q, out, kc, vc, bt, cl, sl = (b[n].t for n in ("q", "out", "kc", "vc", "bt", "cl", "slots"))
    P = 64
    need = pa.decode_split_workspace_size(wl.S, wl.Hq, wl.D, wl.max_context_len, P)
    ws = Guarded(torch.zeros(need, dtype=torch.uint8, device="cuda"))
    pa.reshape_and_cache(b["key"].t, b["value"].t, kc, vc, sl)
    pa.decode(out, q, kc, vc, bt, cl, wl.scale)
    pa.decode_split(out, q, kc, vc, bt, cl, wl.scale, 1.0, wl.max_context_len, P, ws.t)
    pa.cache_and_decode(out, q, b["key"].t, b["value"].t, sl, kc, vc, bt, cl, wl.scale)
    pa.cache_and_decode(out, q, b["key"].t, b["value"].t, sl, kc, vc, bt, cl, wl.scale, 1.0, wl.max_context_len, P,
                        ws.t)
    pa.get_device_error()  # clear the expected flags of the out-of-range case
    for name, t in list(b.items()) + [("workspace", ws)]:
        assert t.intact(), name


def test_prefill_and_block_moves_stay_inside_their_buffers():
    pa = _gpu.lib()
    wl = W.make_workload(name="t", seed=62, context_lens=[130, 300], Hq=8, Hkv=2, D=128, bs=16, q_dtype="bf16",
                         kv_dtype="bf16", qlen=130)
    g, b = _guarded_batch(wl)
    q, out, kc, vc, bt, cl = (b[n].t for n in ("q", "out", "kc", "vc", "bt", "cl"))
    pa.prefill(out, q, kc, vc, bt, cl, wl.scale)
    n = 8
    ids = torch.from_numpy(np.random.default_rng(5).permutation(wl.NB)[:2 * n]).cuda()
    pairs = Guarded(torch.stack([ids[:n], ids[n:]], dim=1).contiguous())
    pa.copy_blocks(kc, vc, pairs.t)
    host = Guarded(torch.zeros((n, 2) + tuple(kc.shape[1:]), dtype=kc.dtype), pinned_host=True)
    pa.gather_blocks(host.t, kc, vc, ids[:n].contiguous())
    pa.scatter_blocks(kc, vc, host.t, ids[n:].contiguous())
    for name, t in list(b.items()) + [("pairs", pairs), ("host", host)]:
        assert t.intact(), name
