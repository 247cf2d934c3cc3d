"""A decode batch resident on the GPU.

``DeviceBatch`` holds one workload's q, new K/V rows, block tables, context
lengths, slot mapping and KV pool as torch tensors on a CUDA device (torch is
used for memory only) and runs one decode step through the library: the
scatter of the new rows, then decode attention (single pass or split).
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import pagedattn as pa
from .workloads import FP8, Workload


def to_device16(bits: np.ndarray, dtype: str, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def from_device16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceBatch:
    def __init__(self, wl: Workload, device="cuda", partition_size: Optional[int] = None, fused: bool = True):
        self.wl = wl
        self.fused = fused  # step() = one pa_cache_and_decode launch instead of scatter + decode
        self.device = torch.device(device)
        self.partition_size = wl.partition_size if partition_size is None else partition_size
        d = self.device
        self.q = to_device16(wl.q, wl.q_dtype, d)
        self.key = to_device16(wl.key, wl.q_dtype, d)
        self.value = to_device16(wl.value, wl.q_dtype, d)
        self.block_tables = torch.from_numpy(wl.block_tables).to(d)
        self.context_lens = torch.from_numpy(wl.context_lens).to(d)
        self.slot_mapping = torch.from_numpy(wl.slot_mapping).to(d)
        if wl.kv_dtype == FP8:
            fill = 0xFF if wl.notes.get("fill_unused") == "nan" else 0
            self.k_cache = torch.full(wl.cache_shape(), fill, dtype=torch.uint8, device=d)
            self.v_cache = torch.full(wl.cache_shape(), fill, dtype=torch.uint8, device=d)
            if wl.prefill_slots is not None and len(wl.prefill_slots):
                pa.reshape_and_cache(to_device16(wl.prefill_key, wl.q_dtype, d),
                                     to_device16(wl.prefill_value, wl.q_dtype, d), self.k_cache, self.v_cache,
                                     torch.from_numpy(wl.prefill_slots).to(d), wl.kv_scale)
        else:
            self.k_cache = to_device16(wl.k_cache, wl.kv_dtype, d)
            self.v_cache = to_device16(wl.v_cache, wl.kv_dtype, d)
        self.out = torch.empty_like(self.q)
        self.workspace = None
        if self.partition_size:
            need = pa.decode_multi_split_workspace_size(wl.S, wl.qlen, wl.Hq, wl.D, wl.max_context_len,
                                                        self.partition_size)
            self.workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=d)

    INPUTS = ("q", "key", "value", "block_tables", "context_lens", "slot_mapping", "out")

    def io_set(self) -> dict:
        """The per-step input and output tensors the batch is bound to."""
        return {name: getattr(self, name) for name in self.INPUTS}

    def spare_io_set(self) -> dict:
        """A second set of per-step input and output tensors of the same shapes
        (the KV pool and workspace stay shared), for overlapping one step's
        copies with another step's kernels."""
        return {name: torch.empty_like(t) for name, t in self.io_set().items()}

    def bind(self, io: dict) -> None:
        for name in self.INPUTS:
            setattr(self, name, io[name])

    def scatter(self) -> None:
        pa.reshape_and_cache(self.key, self.value, self.k_cache, self.v_cache, self.slot_mapping,
                             self.wl.kv_scale)

    def decode(self) -> torch.Tensor:
        wl = self.wl
        if wl.qlen > 1 and self.partition_size:
            pa.decode_multi_split(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                  self.context_lens, wl.scale, wl.kv_scale, wl.max_context_len,
                                  self.partition_size, self.workspace)
        elif wl.qlen > 1:
            pa.decode_multi(self.out, self.q, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                            wl.scale, wl.kv_scale)
        elif self.partition_size:
            pa.decode_split(self.out, self.q, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                            wl.scale, wl.kv_scale, wl.max_context_len, self.partition_size, self.workspace)
        else:
            pa.decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                      wl.scale, wl.kv_scale)
        return self.out

    def step(self) -> torch.Tensor:
        if not self.fused:
            self.scatter()
            return self.decode()
        wl = self.wl
        pa.cache_and_decode(self.out, self.q, self.key, self.value, self.slot_mapping, self.k_cache, self.v_cache,
                            self.block_tables, self.context_lens, wl.scale, wl.kv_scale, wl.max_context_len,
                            self.partition_size, self.workspace)
        return self.out

    def tensor_core_path(self) -> bool:
        """Whether the decode goes to the tensor-core kernel (query group of
        more than 16 columns) instead of the warp-MMA decode kernel."""
        return self.wl.G * self.wl.qlen > 16

    def launches_per_step(self) -> int:
        merge = 1 if self.partition_size else 0
        if self.fused and not self.tensor_core_path():
            return 1 + merge  # the scatter runs inside the decode launch
        return 2 + merge
