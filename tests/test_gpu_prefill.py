"""GPU parity of the chunked-prefill tile (tcgen05) against the fp64 oracle.

Tolerance: bf16 inputs, fp32 accumulation, bf16 softmax weights and bf16
output -> |gpu - ref| <= 2e-2 + 2e-2 |ref| (the bf16 bound used for decode).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import _binding as B
from paged_kv_cache_71_gb300 import workload as wl
from paged_kv_cache_71_gb300.runner import to_device

from parity import assert_close, to_host

pytestmark = pytest.mark.gpu


def _chunk_case(NQ, q_start, Hq, Hkv, S, seed, extra_blocks=5, poison=False, kv="bf16"):
    """One sequence of kv_len = q_start + NQ tokens in a shuffled pool, plus a query chunk."""
    rng = np.random.default_rng(seed)
    D = 128
    kv_len = q_start + NQ
    nb = -(-kv_len // S)
    NB = nb + extra_blocks
    alloc = wl.BlockAllocator(NB, S, free_order=rng.permutation(NB))
    alloc.add_seq("s", kv_len)
    table = np.array(alloc.tables["s"], np.int32)
    kc = wl.random_values(rng, (NB, S, Hkv, D), kv)
    vc = wl.random_values(rng, (NB, S, Hkv, D), kv)
    if poison:  # NaN in every slot that is not one of the sequence's tokens
        owned = np.zeros((NB, S), bool)
        for p in range(kv_len):
            owned[table[p // S], p % S] = True
        kc[~owned] = 0x7FC0
        vc[~owned] = 0x7FC0
    q = wl.random_values(rng, (NQ, Hq, D), "bf16")
    return q, kc, vc, table, kv_len


def _run(q, kc, vc, table, q_start, kv_len, scale, k_scale=1.0, v_scale=1.0):
    dq, dk, dv = to_device(q), to_device(kc), to_device(vc)
    out = torch.full_like(dq, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_paged_prefill_chunk(out, dq, q_start, dk, dv, B.CacheDesc.for_cache(dk, k_scale, v_scale),
                                to_device(table), kv_len, scale, err)
    torch.cuda.synchronize()
    assert err.item() == 0, hex(err.item())
    return to_host(out)


@pytest.mark.parametrize("NQ,q_start,Hq,Hkv,S", [
    (16, 0, 8, 1, 16),        # one tile, pure prefill from position 0
    (40, 100, 8, 1, 16),      # ragged last query tile, keys straddle a 128-key tile
    (37, 250, 16, 4, 8),      # G = 4, block size 8
    (130, 3, 4, 4, 32),       # G = 1 (128 queries per CTA), block size 32
    (64, 128, 16, 2, 16),     # kv_len a multiple of 128
])
def test_prefill_chunk_matches_oracle(NQ, q_start, Hq, Hkv, S):
    q, kc, vc, table, kv_len = _chunk_case(NQ, q_start, Hq, Hkv, S, seed=NQ + q_start)
    scale = 1 / np.sqrt(128)
    ref = oracle.paged_prefill_chunk(q, q_start, kc, vc, table, kv_len, scale)
    got = _run(q, kc, vc, table, q_start, kv_len, scale)
    assert_close("bf16", got, ref, f"prefill NQ={NQ} q_start={q_start} G={Hq // Hkv} S={S}")


@pytest.mark.parametrize("NQ,q_start,Hq,Hkv,S", [(40, 100, 8, 1, 16), (130, 3, 4, 4, 32), (33, 500, 16, 2, 8)])
def test_prefill_chunk_fp8_cache(NQ, q_start, Hq, Hkv, S):
    q, kc, vc, table, kv_len = _chunk_case(NQ, q_start, Hq, Hkv, S, seed=7 + NQ, kv="e4m3")
    scale = 1 / np.sqrt(128)
    ref = oracle.paged_prefill_chunk(q, q_start, kc, vc, table, kv_len, scale, k_scale=0.25, v_scale=0.5)
    got = _run(q, kc, vc, table, q_start, kv_len, scale, 0.25, 0.5)
    assert_close("e4m3", got, ref, f"fp8 prefill NQ={NQ} q_start={q_start}")


def test_prefill_chunk_int8_cache():
    q, kc, vc, table, kv_len = _chunk_case(75, 300, 16, 2, 16, seed=9, kv="i8")
    scale = 1 / np.sqrt(128)
    ref = oracle.paged_prefill_chunk(q, 300, kc, vc, table, kv_len, scale, k_scale=1 / 32, v_scale=1 / 16)
    got = _run(q, kc, vc, table, 300, kv_len, scale, 1 / 32, 1 / 16)
    assert_close("i8", got, ref, "int8 prefill")


def test_prefill_poisoned_slots_do_not_leak():
    q, kc, vc, table, kv_len = _chunk_case(45, 70, 8, 1, 16, seed=3, poison=True)
    scale = 1 / np.sqrt(128)
    got = _run(q, kc, vc, table, 70, kv_len, scale)
    assert np.isfinite(got).all()
    ref = oracle.paged_prefill_chunk(q, 70, kc, vc, table, kv_len, scale)
    assert_close("bf16", got, ref, "poisoned prefill")


def test_prefill_rejects_missing_chunk_keys_and_bad_shapes():
    q, kc, vc, table, kv_len = _chunk_case(16, 10, 8, 1, 16, seed=5)
    dq, dk, dv = to_device(q), to_device(kc), to_device(vc)
    out = torch.empty_like(dq)
    with pytest.raises(pkv.PkvError) as ei:  # kv_len must cover the chunk's own keys
        pkv.pkv_paged_prefill_chunk(out, dq, 10, dk, dv, B.CacheDesc.for_cache(dk), to_device(table), 20, 0.1)
    assert ei.value.status == 1
    d = B.CacheDesc.for_cache(dk)
    d.block_size = 4
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_paged_prefill_chunk(out, dq, 10, dk, dv, d, to_device(table), kv_len, 0.1)
    assert ei.value.status == 2


@pytest.mark.parametrize("name", ["llama70b_mixed_bf16", "llama70b_mixed_fp8"])
def test_llama70b_chunk_sampled_rows(name):
    """The 512-token chunk at positions 8192..8703 over the Llama-70B-shaped pool (64 q / 8 kv heads)."""
    w = wl.make(name)
    pf = w.prefill
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    cdt = oracle.E4M3 if w.kv_dtype == "e4m3" else oracle.BF16
    oracle.reshape_and_cache(w.k_new, w.v_new, w.slot_mapping, kc, vc, cache_dtype=cdt, k_scale=w.k_scale,
                             v_scale=w.v_scale)
    rows = [0, 1, 15, 16, 127, 255, 256, 400, 510, 511]
    ref = oracle.paged_prefill_chunk(pf.q, pf.q_start, kc, vc, pf.block_table, pf.kv_len, w.scale, rows=rows,
                                     cache_dtype=cdt, k_scale=w.k_scale, v_scale=w.v_scale)
    dk, dv = to_device(w.k_cache), to_device(w.v_cache)
    desc = B.CacheDesc.for_cache(dk, w.k_scale, w.v_scale)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_reshape_and_cache(to_device(w.k_new), to_device(w.v_new), to_device(w.slot_mapping), dk, dv, desc, err)
    dq = to_device(pf.q)
    out = torch.full_like(dq, float("nan"))
    pkv.pkv_paged_prefill_chunk(out, dq, pf.q_start, dk, dv, desc, to_device(pf.block_table), pf.kv_len, w.scale,
                                err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = to_host(out)
    assert np.isfinite(got).all()
    assert_close(w.kv_dtype, got[rows], ref, name)
