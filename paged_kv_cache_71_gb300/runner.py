"""Stage a synthetic workload on the GPU and run one decode step through the C ABI.

A step is the whole hot path for one batch: the copy-on-write block copies
(when the batch has any), the cache write of this step's new tokens, and
paged decode attention over every sequence.  Only device memory, streams
and argument marshalling live here; the work runs in libpkv.so's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as B
from .workload import Workload

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8, "i8": torch.int8}


def to_device(a: np.ndarray, dtype: str | None = None, device="cuda") -> torch.Tensor:
    """Upload a host array; uint16 arrays are bf16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(device)


class DeviceStep:
    """Device copies of a workload's inputs plus output / workspace buffers."""

    def __init__(self, w: Workload, num_splits: int = 0, device="cuda", shared=None):
        self.w = w
        self.num_splits = num_splits
        # a batch whose tables share physical blocks takes the shared-block decode form (the host block manager
        # knows: the workload records its shared blocks)
        self.shared = bool(w.notes.get("shared_blocks")) if shared is None else bool(shared)
        self.k_cache = to_device(w.k_cache, device=device)
        self.v_cache = to_device(w.v_cache, device=device)
        self.q = to_device(w.q, device=device)
        self.block_tables = to_device(w.block_tables, device=device)
        self.context_lens = to_device(w.context_lens, device=device)
        self.k_new = to_device(w.k_new, device=device)
        self.v_new = to_device(w.v_new, device=device)
        self.slot_mapping = to_device(w.slot_mapping, device=device)
        self.copy_pairs = to_device(w.copy_pairs, device=device) if len(w.copy_pairs) else None
        self.cache = B.CacheDesc.for_cache(self.k_cache, w.k_scale, w.v_scale)
        self.out = torch.empty_like(self.q)
        ws = B.pkv_paged_attention_workspace_size(self.cache, w.num_seqs, w.num_q_heads, num_splits)
        self.workspace = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.max_context_len = int(w.context_lens.max()) if w.num_seqs else 0
        self.pf_q = self.pf_out = self.pf_table = None
        if w.prefill is not None:
            self.pf_q = to_device(w.prefill.q, device=device)
            self.pf_out = torch.empty_like(self.pf_q)
            self.pf_table = to_device(w.prefill.block_table, device=device)

    def write(self, stream=None) -> None:
        if self.copy_pairs is not None:
            B.pkv_copy_blocks(self.k_cache, self.v_cache, self.cache, self.copy_pairs, self.err, stream)
        B.pkv_reshape_and_cache(self.k_new, self.v_new, self.slot_mapping, self.k_cache, self.v_cache, self.cache,
                                self.err, stream)

    def attend(self, stream=None) -> None:
        fn = B.pkv_paged_attention_decode_shared if self.shared else B.pkv_paged_attention_decode
        fn(self.out, self.q, self.k_cache, self.v_cache, self.cache, self.block_tables, self.context_lens,
           self.w.scale, self.num_splits, self.max_context_len, self.workspace, self.err, stream)

    def prefill(self, stream=None) -> None:
        if self.pf_q is None:
            return
        pf = self.w.prefill
        B.pkv_paged_prefill_chunk(self.pf_out, self.pf_q, pf.q_start, self.k_cache, self.v_cache, self.cache,
                                  self.pf_table, pf.kv_len, self.w.scale, self.err, stream)

    def step(self, stream=None) -> None:
        self.write(stream)
        self.attend(stream)
        self.prefill(stream)

    def device_error(self) -> int:
        return int(self.err.item())
