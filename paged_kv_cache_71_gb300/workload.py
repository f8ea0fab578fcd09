"""Seeded synthetic workloads for paged decode attention.

This module builds inputs only.  It holds none of the attention arithmetic:
it draws lengths and values from seeded generators, hands out physical
blocks the way a serving engine's block manager does, and records where
each new token must be written.  Both the CUDA path and the CPU oracle
consume what it produces; neither is imported here.

Physical blocks are handed out by ``block_manager.SequenceTables`` (free-id
stack, reference counts, copy-on-write of shared partial blocks), seeded
with a random permutation of the pool so that tables are scattered.

Value distributions (all seeded with ``numpy.random.default_rng``):
Q, K, V ~ N(0, 1) drawn in float32 and rounded once to the storage dtype;
FP8 E4M3 caches hold random codes (uniform sign and mantissa, exponent
field uniform in [4, 10]) with a per-tensor scale of 0.25, and INT8 caches
random codes uniform in [-127, 127] with a scale of 1/32, so that no
quantiser is involved in making them.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

from .block_manager import SequenceTables

# ---------------------------------------------------------------- value generation

DTYPES = ("f32", "bf16", "e4m3", "i8")
_ELEM = {"f32": 4, "bf16": 2, "e4m3": 1, "i8": 1}
FP8_SCALE = 0.25
INT8_SCALE = 1.0 / 32.0


def elem_size(dtype: str) -> int:
    return _ELEM[dtype]


def _normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _fill_chunk(base: int, c: int, a: int, b: int, dtype: str, out: np.ndarray) -> None:
    sub = np.random.default_rng([base, c])
    v = _normal_f32(sub, b - a)
    out[a:b] = v if dtype == "f32" else to_bf16_bits(v)


def random_values(rng: np.random.Generator, shape, dtype: str, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) values stored as float32 / bf16 bits (uint16); random E4M3 codes (uint8) or
    symmetric INT8 codes uniform in [-127, 127] (int8).

    Large arrays are drawn in fixed-size chunks, each from its own generator
    seeded by (a draw of ``rng``, chunk index), on a thread pool: the result
    depends only on ``rng``'s state, not on the number of threads."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    if dtype == "i8":
        return rng.integers(-127, 128, size=n, dtype=np.int8).reshape(shape)
    if dtype == "e4m3":
        sign = rng.integers(0, 2, size=n, dtype=np.uint8)
        expo = rng.integers(4, 11, size=n, dtype=np.uint8)
        mant = rng.integers(0, 8, size=n, dtype=np.uint8)
        return ((sign << 7) | (expo << 3) | mant).astype(np.uint8).reshape(shape)
    out = np.empty(n, dtype=np.float32 if dtype == "f32" else np.uint16)
    if n <= chunk:
        v = _normal_f32(rng, n)
        out[:] = v if dtype == "f32" else to_bf16_bits(v)
        return out.reshape(shape)
    base = int(rng.integers(0, 2**63 - 1))
    spans = [(c, a, min(n, a + chunk)) for c, a in enumerate(range(0, n, chunk))]
    workers = max(1, min(len(spans), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda t: _fill_chunk(base, t[0], t[1], t[2], dtype, out), spans))
    return out.reshape(shape)


# ---------------------------------------------------------------- configurations


@dataclass
class PrefillChunk:
    q: np.ndarray              # [NQ, Hq, D] in q dtype
    q_start: int               # position of the chunk's first query token
    kv_len: int                # keys visible to the last query (q_start + NQ)
    block_table: np.ndarray    # int32 [blocks] of the chunk's sequence


@dataclass
class Workload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str
    q_dtype: str
    k_scale: float
    v_scale: float
    q: np.ndarray                     # [B, Hq, D]
    k_cache: np.ndarray               # [NB, S, Hkv, D]
    v_cache: np.ndarray
    block_tables: np.ndarray          # int32 [B, MB], -1 padded
    context_lens: np.ndarray          # int32 [B], includes this step's token
    k_new: np.ndarray                 # [T, Hkv, D] in q dtype (the projection's output dtype)
    v_new: np.ndarray
    slot_mapping: np.ndarray          # int64 [T]
    copy_pairs: np.ndarray            # int64 [N, 2] (src, dst), may be empty
    prefill: PrefillChunk | None = None
    notes: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))


CONFIG_NAMES = ("tiny", "llama2_7b", "llama3_8b_gqa", "prefix_shared", "llama70b_mixed_bf16",
                "llama70b_mixed_fp8", "llama3_8b_gqa_int8")

CONFIG_SEEDS = {"tiny": 7100, "llama2_7b": 7101, "llama3_8b_gqa": 7102, "prefix_shared": 7103,
                "llama70b_mixed_bf16": 7104, "llama70b_mixed_fp8": 7104, "llama3_8b_gqa_int8": 7102}


def _pool_size(total_blocks: int, slack: float = 0.05) -> int:
    return int(total_blocks + max(1, int(np.ceil(total_blocks * slack))))


def _cache_and_q(rng, NB, S, Hkv, D, B, Hq, kv_dtype, q_dtype):
    k_cache = random_values(rng, (NB, S, Hkv, D), kv_dtype)
    v_cache = random_values(rng, (NB, S, Hkv, D), kv_dtype)
    q = random_values(rng, (B, Hq, D), q_dtype)
    return k_cache, v_cache, q


def _decode_batch(name, lens, Hq, Hkv, D, S, kv_dtype, q_dtype, seed, exact_pool=None):
    """B independent sequences: prefill L-1 tokens, then append this step's token."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    need = int(sum(-(-int(L) // S) for L in lens))
    NB = exact_pool or _pool_size(need)
    tabs = SequenceTables(NB, S, free_order=rng.permutation(NB))
    slots = []
    for s, L in enumerate(lens):
        tabs.prefill(s, int(L) - 1)
        slots.append(tabs.next_slot(s))
    sids = list(range(len(lens)))
    k_cache, v_cache, q = _cache_and_q(rng, NB, S, Hkv, D, len(lens), Hq, kv_dtype, q_dtype)
    k_new = random_values(rng, (len(lens), Hkv, D), q_dtype)
    v_new = random_values(rng, (len(lens), Hkv, D), q_dtype)
    scale = {"e4m3": FP8_SCALE, "i8": INT8_SCALE}.get(kv_dtype, 1.0)
    return Workload(name, seed, Hq, Hkv, D, S, kv_dtype, q_dtype, scale, scale, q, k_cache, v_cache,
                    tabs.block_tables(sids), lens.astype(np.int32), k_new, v_new,
                    np.array(slots, dtype=np.int64), np.zeros((0, 2), dtype=np.int64),
                    notes={"pool_blocks": NB, "used_blocks": need})


def tiny(seed: int = CONFIG_SEEDS["tiny"]) -> Workload:
    """4 sequences {10, 6, 33, 1}, S=4, 32 permuted physical blocks, 4 q / 2 kv heads, D=64, fp32.
    The 4 new tokens land at positions {9, 5, 32, 0}."""
    return _decode_batch("tiny", [10, 6, 33, 1], 4, 2, 64, 4, "f32", "f32", seed, exact_pool=32)


def llama2_7b(seed: int = CONFIG_SEEDS["llama2_7b"]) -> Workload:
    """Batch 64, 32 q = 32 kv heads, D=128, bf16, S=16, lengths uniform in [128, 4096]."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(128, 4097, size=64)
    return _decode_batch("llama2_7b", lens, 32, 32, 128, 16, "bf16", "bf16", seed + 1000)


def lognormal_lengths(rng, n, median=1024.0, sigma=1.0, lo=16, hi=8192) -> np.ndarray:
    return np.clip(np.round(np.exp(rng.normal(np.log(median), sigma, size=n))), lo, hi).astype(np.int64)


def llama3_8b_gqa(seed: int = CONFIG_SEEDS["llama3_8b_gqa"], batch: int = 256, kv_dtype: str = "bf16") -> Workload:
    """Batch 256, 32 q / 8 kv heads, D=128, bf16, S=16, lengths lognormal (median 1024,
    sigma 1) clipped to [16, 8192]; plus the cache write of the 256 new tokens.
    kv_dtype "i8" gives the same batch over a symmetric INT8 cache."""
    rng = np.random.default_rng(seed)
    lens = lognormal_lengths(rng, batch)
    name = "llama3_8b_gqa" + ("_int8" if kv_dtype == "i8" else "")
    return _decode_batch(name, lens, 32, 8, 128, 16, kv_dtype, "bf16", seed + 1000)


def prefix_shared(seed: int = CONFIG_SEEDS["prefix_shared"], batch: int = 128, prefix: int = 800,
                  private: int = 205, cow_parent_len: int = 805) -> Workload:
    """128 sequences share an 800-token prefix (the same 50 physical blocks, refcount 128) and
    then hold 205 private tokens each (L = 1005).  A fork of a parent whose last block is
    partial (805 tokens, 5 in block 50) into 128 children makes every child's first append
    copy that block: 128 (src, dst) pairs for copy_blocks, then each child writes its token
    at offset 5 of its copy; the parent keeps the original."""
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D = 16, 32, 8, 128
    need = (prefix // S) + batch * (-(-(prefix + private) // S) - prefix // S) \
        + (-(-cow_parent_len // S)) + batch
    NB = _pool_size(need)
    tabs = SequenceTables(NB, S, free_order=rng.permutation(NB))
    tabs.prefill("prefix", prefix)
    for s in range(batch):
        tabs.fork("prefix", s)
    tabs.drop("prefix")
    slots = []
    for s in range(batch):
        for _ in range(private - 1):
            tabs.next_slot(s)
        slots.append(tabs.next_slot(s))
    tabs.prefill("cow_parent", cow_parent_len)
    cow_children = [("cow", c) for c in range(batch)]
    for c in cow_children:
        tabs.fork("cow_parent", c)
    for c in cow_children:
        slots.append(tabs.next_slot(c))
    pairs = np.array(tabs.drain_copies(), dtype=np.int64).reshape(-1, 2)
    sids = list(range(batch))
    k_cache, v_cache, q = _cache_and_q(rng, NB, S, Hkv, D, batch, Hq, "bf16", "bf16")
    T = len(slots)
    k_new = random_values(rng, (T, Hkv, D), "bf16")
    v_new = random_values(rng, (T, Hkv, D), "bf16")
    lens = np.array([tabs.length(s) for s in sids], dtype=np.int32)
    shared = tabs.table(0)[: prefix // S]
    return Workload("prefix_shared", seed, Hq, Hkv, D, S, "bf16", "bf16", 1.0, 1.0, q, k_cache, v_cache,
                    tabs.block_tables(sids), lens, k_new, v_new, np.array(slots, dtype=np.int64), pairs,
                    notes={"pool_blocks": NB, "shared_blocks": list(map(int, shared)),
                           "shared_refcount": int(tabs.pool.refcount[shared[0]]),
                           "cow_parent_table": list(map(int, tabs.table("cow_parent"))),
                           "cow_child_tables": [list(map(int, tabs.table(c))) for c in cow_children],
                           "cow_child_len": tabs.length(cow_children[0]),
                           "num_decode_tokens": batch})


def llama70b_mixed(kv_dtype: str = "bf16", seed: int = CONFIG_SEEDS["llama70b_mixed_bf16"],
                   batch: int = 48, chunk: int = 512, prefix: int = 8192) -> Workload:
    """64 q / 8 kv heads, D=128, S=16: 48 decode sequences with lengths uniform in
    [4096, 32768] plus one chunked-prefill chunk of 512 query tokens at positions
    8192..8703 over an 8192-token paged prefix (the chunk's own K/V is written first,
    so 8704 keys are cached).  KV in bf16 or FP8 E4M3 with a per-tensor scale."""
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D = 16, 64, 8, 128
    lens = rng.integers(4096, 32769, size=batch)
    need = int(sum(-(-int(L) // S) for L in lens)) + (-(-(prefix + chunk) // S))
    NB = _pool_size(need)
    tabs = SequenceTables(NB, S, free_order=rng.permutation(NB))
    slots = []
    for s, L in enumerate(lens):
        tabs.prefill(s, int(L) - 1)
        slots.append(tabs.next_slot(s))
    tabs.prefill("chunked", prefix)
    for _ in range(chunk):
        slots.append(tabs.next_slot("chunked"))
    sids = list(range(batch))
    k_cache, v_cache, q = _cache_and_q(rng, NB, S, Hkv, D, batch, Hq, kv_dtype, "bf16")
    T = len(slots)
    k_new = random_values(rng, (T, Hkv, D), "bf16")
    v_new = random_values(rng, (T, Hkv, D), "bf16")
    q_chunk = random_values(rng, (chunk, Hq, D), "bf16")
    pf = PrefillChunk(q_chunk, prefix, prefix + chunk, np.array(tabs.table("chunked"), dtype=np.int32))
    scale = FP8_SCALE if kv_dtype == "e4m3" else 1.0
    name = "llama70b_mixed_" + ("fp8" if kv_dtype == "e4m3" else "bf16")
    return Workload(name, seed, Hq, Hkv, D, S, kv_dtype, "bf16", scale, scale, q, k_cache, v_cache,
                    tabs.block_tables(sids), lens.astype(np.int32), k_new, v_new,
                    np.array(slots, dtype=np.int64), np.zeros((0, 2), dtype=np.int64), prefill=pf,
                    notes={"pool_blocks": NB, "num_decode_tokens": batch})


def make(name: str, **kw) -> Workload:
    if name == "tiny":
        return tiny(**kw)
    if name == "llama2_7b":
        return llama2_7b(**kw)
    if name == "llama3_8b_gqa":
        return llama3_8b_gqa(**kw)
    if name == "prefix_shared":
        return prefix_shared(**kw)
    if name == "llama70b_mixed_bf16":
        return llama70b_mixed("bf16", **kw)
    if name == "llama70b_mixed_fp8":
        return llama70b_mixed("e4m3", seed=CONFIG_SEEDS["llama70b_mixed_fp8"], **kw)
    if name == "llama3_8b_gqa_int8":
        return llama3_8b_gqa(kv_dtype="i8", **kw)
    raise KeyError(name)
