"""Shared helpers for the parity tests: the oracle's version of one step and the tolerances.

Tolerances (stated for the decode output against the fp64 oracle):
  fp32 KV: max |gpu - ref| <= 1e-5
  bf16 KV: |gpu - ref| <= 2e-2 + 2e-2 |ref|   (fp32 accumulation, bf16 output)
  fp8  KV: |gpu - ref| <= 6e-2                 (oracle reads the same dequantised codes)
  int8 KV: |gpu - ref| <= 2e-2 + 2e-2 |ref|   (same dequantised codes, fp32 accumulation, bf16 output)
Cache writes, block copies and indexing are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"f32": (1e-5, 0.0), "bf16": (2e-2, 2e-2), "e4m3": (6e-2, 0.0), "i8": (2e-2, 2e-2)}


def oracle_step(w, seqs=None, threads=0):
    """Apply the step's copies and cache writes to host copies of the caches, then
    evaluate attention for `seqs` (all when None).  Returns (k_cache, v_cache, out)."""
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    if len(w.copy_pairs):
        oracle.copy_blocks(kc, vc, w.copy_pairs)
    cache_dt = {"f32": oracle.F32, "bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}[w.kv_dtype]
    oracle.reshape_and_cache(w.k_new, w.v_new, w.slot_mapping, kc, vc, cache_dtype=cache_dt,
                             k_scale=w.k_scale, v_scale=w.v_scale)
    out = oracle.paged_attention_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale,
                                        cache_dtype=cache_dt, k_scale=w.k_scale, v_scale=w.v_scale,
                                        seqs=seqs, threads=threads)
    return kc, vc, out


def to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw storage of a device tensor as a host array (bf16 -> uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def assert_close(kind: str, got: np.ndarray, ref: np.ndarray, what: str = "") -> float:
    atol, rtol = TOL[kind]
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance ({kind}); worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r}")
    return float(err.max()) if err.size else 0.0
