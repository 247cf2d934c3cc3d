"""Shared helpers of the GPU parity tests: move a seeded workload to the GPU,
run one decode step through the library, and compute the oracle's answer on
the same bytes."""
import numpy as np
import torch

import oracle
from paged_kv_cache_230_gb300 import workloads as W

TOL = {"f16": 2e-3, "bf16": 1.6e-2, "fp8": 5e-2}  # max |gpu - oracle fp64|


def tolerance(wl):
    return TOL["fp8"] if wl.kv_dtype == "fp8" else TOL[wl.q_dtype]


def lib():
    from paged_kv_cache_230_gb300 import build
    build.build()
    from paged_kv_cache_230_gb300 import pagedattn
    return pagedattn


def dev16(bits: np.ndarray, dtype: str, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def host16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class OnGpu:
    """The workload's arrays on the GPU, with the pool filled (FP8 pools by the
    library's own scatter of the prefill rows)."""

    def __init__(self, wl: W.Workload, device="cuda"):
        pa = lib()
        self.wl = wl
        self.q = dev16(wl.q, wl.q_dtype, device)
        self.key = dev16(wl.key, wl.q_dtype, device)
        self.value = dev16(wl.value, wl.q_dtype, device)
        self.bt = torch.from_numpy(wl.block_tables).to(device)
        self.cl = torch.from_numpy(wl.context_lens).to(device)
        self.slots = torch.from_numpy(wl.slot_mapping).to(device)
        if wl.kv_dtype == "fp8":
            fill = 0xFF if wl.notes.get("fill_unused") == "nan" else 0
            self.kc = torch.full(wl.cache_shape(), fill, dtype=torch.uint8, device=device)
            self.vc = torch.full(wl.cache_shape(), fill, dtype=torch.uint8, device=device)
            if len(wl.prefill_slots):
                pa.reshape_and_cache(dev16(wl.prefill_key, wl.q_dtype, device),
                                     dev16(wl.prefill_value, wl.q_dtype, device), self.kc, self.vc,
                                     torch.from_numpy(wl.prefill_slots).to(device), wl.kv_scale)
        else:
            self.kc = dev16(wl.k_cache, wl.kv_dtype, device)
            self.vc = dev16(wl.v_cache, wl.kv_dtype, device)
        self.out = torch.empty_like(self.q)
        self.ws = None

    def scatter(self):
        lib().reshape_and_cache(self.key, self.value, self.kc, self.vc, self.slots, self.wl.kv_scale)

    def decode(self, partition_size: int = 0):
        pa = lib()
        wl = self.wl
        if partition_size:
            mcl = wl.max_context_len
            need = pa.decode_multi_split_workspace_size(wl.S, wl.qlen, wl.Hq, wl.D, mcl, partition_size)
            if self.ws is None or self.ws.numel() < need:
                self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=self.q.device)
            if wl.qlen > 1:
                pa.decode_multi_split(self.out, self.q, self.kc, self.vc, self.bt, self.cl, wl.scale, wl.kv_scale,
                                      mcl, partition_size, self.ws)
            else:
                pa.decode_split(self.out, self.q, self.kc, self.vc, self.bt, self.cl, wl.scale, wl.kv_scale, mcl,
                                partition_size, self.ws)
        elif wl.qlen > 1:
            pa.decode_multi(self.out, self.q, self.kc, self.vc, self.bt, self.cl, wl.scale, wl.kv_scale)
        else:
            pa.decode(self.out, self.q, self.kc, self.vc, self.bt, self.cl, wl.scale, wl.kv_scale)
        return self.out

    def step(self, partition_size: int = 0):
        self.scatter()
        return self.decode(partition_size)

    def caches_host(self):
        if self.wl.kv_dtype == "fp8":
            return self.kc.cpu().numpy(), self.vc.cpu().numpy()
        return host16(self.kc), host16(self.vc)


def oracle_pool(wl: W.Workload):
    """Pool contents after this step's scatter, computed by the oracle."""
    if wl.kv_dtype == "fp8":
        fill = 0xFF if wl.notes.get("fill_unused") == "nan" else 0
        kc = np.full(wl.cache_shape(), fill, np.uint8)
        vc = np.full(wl.cache_shape(), fill, np.uint8)
        if len(wl.prefill_slots):
            oracle.reshape_and_cache(wl.prefill_key, wl.prefill_value, wl.q_dtype, kc, vc, "fp8",
                                     wl.prefill_slots, wl.kv_scale)
    else:
        kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.reshape_and_cache(wl.key, wl.value, wl.q_dtype, kc, vc, wl.kv_dtype, wl.slot_mapping, wl.kv_scale)
    return kc, vc


def oracle_out(wl: W.Workload, kc, vc, partition_size: int = 0):
    """Oracle output in the workload's q layout.  With k new tokens per
    sequence, new token j of sequence s is decoded by the oracle as its own
    query over the context prefix ending at its position L - k + j (the
    causal rule), through the same block-table row."""
    if wl.qlen == 1:
        return oracle.decode(wl.q, wl.q_dtype, kc, vc, wl.kv_dtype, wl.block_tables, wl.context_lens, wl.scale,
                             wl.kv_scale, partition_size=partition_size)
    k = wl.qlen
    q = wl.q.reshape(wl.S * k, wl.Hq, wl.D)
    bt = np.repeat(wl.block_tables, k, axis=0)
    L = (wl.context_lens[:, None] - k + 1 + np.arange(k)[None, :]).reshape(-1)
    Lc = np.maximum(L, 0).astype(np.int32)
    out = oracle.decode(q, wl.q_dtype, kc, vc, wl.kv_dtype, bt, Lc, wl.scale, wl.kv_scale,
                        partition_size=partition_size)
    return out.reshape(wl.S, k, wl.Hq, wl.D)


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.double().cpu().numpy()


def max_err(got: torch.Tensor, want: np.ndarray) -> float:
    g = out_f64(got)
    assert np.all(np.isfinite(g)), "non-finite output"
    return float(np.abs(g - want).max()) if want.size else 0.0
