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
from paged_kv_cache_71_gb300.block_manager import SequenceTables
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
    alloc = SequenceTables(NB, S, free_order=rng.permutation(NB))
    alloc.prefill("s", kv_len)
    table = np.array(alloc.table("s"), np.int32)
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


# ---------------------------------------------------------------- varlen: several chunks in one launch

def _varlen_case(chunks, Hq, Hkv, S, seed, tail_rows=3, kv="bf16"):
    """chunks: (q_start, n_q) per sequence; sequence s holds q_start + n_q cached tokens in one shared,
    shuffled pool.  Returns host arrays and the per-chunk metadata."""
    rng = np.random.default_rng(seed)
    D = 128
    kv_lens = np.array([qs + nq for qs, nq in chunks], np.int32)
    need = sum(-(-int(L) // S) for L in kv_lens)
    NB = need + 7
    alloc = SequenceTables(NB, S, free_order=rng.permutation(NB))
    for s, L in enumerate(kv_lens):
        alloc.prefill(s, int(L))
    tables = alloc.block_tables(list(range(len(chunks))))
    kc = wl.random_values(rng, (NB, S, Hkv, D), kv)
    vc = wl.random_values(rng, (NB, S, Hkv, D), kv)
    cu = np.zeros(len(chunks) + 1, np.int32)
    cu[1:] = np.cumsum([nq for _, nq in chunks])
    q = wl.random_values(rng, (int(cu[-1]) + tail_rows, Hq, D), "bf16")
    q_starts = np.array([qs for qs, _ in chunks], np.int32)
    return q, kc, vc, tables, cu, q_starts, kv_lens


def _run_varlen(q, kc, vc, tables, cu, q_starts, kv_lens, scale, k_scale=1.0, v_scale=1.0):
    dq, dk, dv = to_device(q), to_device(kc), to_device(vc)
    out = torch.full_like(dq, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_paged_prefill_varlen(out, dq, to_device(cu), to_device(q_starts), to_device(kv_lens), dk, dv,
                                 B.CacheDesc.for_cache(dk, k_scale, v_scale), to_device(tables), scale, err)
    torch.cuda.synchronize()
    return out, int(err.item())


# prefill chunks from position 0 and from the middle of a sequence, decode tokens (a chunk of one query),
# an empty chunk, ragged tiles, chunks that end exactly on a 128-key tile
MIXED = [(0, 200), (300, 1), (129, 0), (1000, 57), (5, 33), (2047, 1), (128, 128), (77, 1), (0, 1)]


@pytest.mark.parametrize("Hq,Hkv,S", [(16, 4, 16), (16, 2, 8), (4, 4, 32), (64, 8, 16)])
def test_prefill_varlen_mixed_batch_matches_oracle(Hq, Hkv, S):
    q, kc, vc, tables, cu, q_starts, kv_lens = _varlen_case(MIXED, Hq, Hkv, S, seed=Hq * 10 + S)
    scale = 1 / np.sqrt(128)
    out, err = _run_varlen(q, kc, vc, tables, cu, q_starts, kv_lens, scale)
    assert err == 0, hex(err)
    got = to_host(out)
    for s, (qs, nq) in enumerate(MIXED):
        if nq == 0:
            continue
        n_tab = -(-int(kv_lens[s]) // S)
        ref = oracle.paged_prefill_chunk(q[cu[s]:cu[s + 1]], qs, kc, vc, tables[s, :n_tab], int(kv_lens[s]), scale)
        assert_close("bf16", got[cu[s]:cu[s + 1]], ref, f"varlen chunk {s} (q_start={qs}, n_q={nq}) G={Hq // Hkv}")
    assert np.isnan(got[cu[-1]:]).all(), "rows outside every chunk were written"


@pytest.mark.parametrize("Hq,Hkv", [(16, 4), (64, 8)])
@pytest.mark.parametrize("kv,k_scale,v_scale", [("e4m3", 0.25, 0.5), ("i8", 1 / 32, 1 / 16)])
def test_prefill_varlen_one_byte_caches(kv, k_scale, v_scale, Hq, Hkv):
    """The mixed batch over an FP8 or INT8 cache: codes widened on chip, scales on scores and output.  Single-token
    chunks and chunk tails that leave query tile B empty run with split widening and a four-slot staging ring (up to
    32 key tiles here, so the ring wraps many times)."""
    q, kc, vc, tables, cu, q_starts, kv_lens = _varlen_case(MIXED, Hq, Hkv, 16, seed=29 + Hq, kv=kv)
    scale = 1 / np.sqrt(128)
    out, err = _run_varlen(q, kc, vc, tables, cu, q_starts, kv_lens, scale, k_scale, v_scale)
    assert err == 0, hex(err)
    got = to_host(out)
    cdt = oracle.E4M3 if kv == "e4m3" else oracle.I8
    for s, (qs, nq) in enumerate(MIXED):
        if nq == 0:
            continue
        n_tab = -(-int(kv_lens[s]) // 16)
        ref = oracle.paged_prefill_chunk(q[cu[s]:cu[s + 1]], qs, kc, vc, tables[s, :n_tab], int(kv_lens[s]), scale,
                                         cache_dtype=cdt, k_scale=k_scale, v_scale=v_scale)
        assert_close(kv, got[cu[s]:cu[s + 1]], ref, f"{kv} varlen chunk {s}")


def test_prefill_varlen_one_chunk_equals_chunk_call():
    """The same chunk through both entry points: identical bits (same tile arithmetic)."""
    q, kc, vc, tables, cu, q_starts, kv_lens = _varlen_case([(90, 75)], 16, 2, 16, seed=11, tail_rows=0)
    scale = 0.07
    out_v, err = _run_varlen(q, kc, vc, tables, cu, q_starts, kv_lens, scale)
    assert err == 0
    dq, dk, dv = to_device(q), to_device(kc), to_device(vc)
    out_c = torch.full_like(dq, float("nan"))
    pkv.pkv_paged_prefill_chunk(out_c, dq, 90, dk, dv, B.CacheDesc.for_cache(dk), to_device(tables[0]),
                                int(kv_lens[0]), scale)
    torch.cuda.synchronize()
    assert torch.equal(out_v.view(torch.int16), out_c.view(torch.int16))


def test_prefill_varlen_device_checks():
    """Chunk metadata is read on the device: a bad chunk raises BAD_LENGTH and is skipped, the rest run."""
    chunks = [(10, 20), (50, 30), (0, 40)]
    q, kc, vc, tables, cu, q_starts, kv_lens = _varlen_case(chunks, 8, 1, 16, seed=5, tail_rows=0)
    scale = 1 / np.sqrt(128)
    short = kv_lens.copy()
    short[1] = 60  # < q_start + n_q = 80: the chunk's own keys are not all cached
    out, err = _run_varlen(q, kc, vc, tables, cu, q_starts, short, scale)
    assert err & 0x4
    got = to_host(out)
    assert np.isnan(got[cu[1]:cu[2]]).all()
    for s in (0, 2):
        ref = oracle.paged_prefill_chunk(q[cu[s]:cu[s + 1]], chunks[s][0], kc, vc, tables[s, :-(-int(kv_lens[s]) // 16)],
                                         int(kv_lens[s]), scale)
        assert_close("bf16", got[cu[s]:cu[s + 1]], ref, f"chunk {s} beside a bad chunk")
    bad_cu = cu.copy()
    bad_cu[3] = cu[3] + 5  # past total_q_tokens
    out, err = _run_varlen(q, kc, vc, tables, bad_cu, q_starts, kv_lens, scale)
    assert err & 0x4
    assert np.isnan(to_host(out)[cu[2]:]).all()


def test_prefill_varlen_host_checks():
    q, kc, vc, tables, cu, q_starts, kv_lens = _varlen_case([(0, 4)], 8, 1, 16, seed=2, tail_rows=0)
    dq, dk, dv = to_device(q), to_device(kc), to_device(vc)
    out = torch.empty_like(dq)
    d = B.CacheDesc.for_cache(dk)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    pkv.pkv_paged_prefill_varlen(out, dq, to_device(cu[:1]), empty, empty, dk, dv, d, to_device(tables), 0.1)
    many = torch.zeros(2049, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_paged_prefill_varlen(out, dq, many, many, many, dk, dv, d, to_device(np.zeros((2049, 1), np.int32)),
                                     0.1)
    assert ei.value.status == 2
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_paged_prefill_varlen(out, dq, to_device(cu), to_device(q_starts), to_device(kv_lens), dk, dv, d,
                                     to_device(tables), -1.0)
    assert ei.value.status == 1


@pytest.mark.parametrize("NQ,q_start,Hq,Hkv,S", [
    (19, 60, 32, 2, 16),      # G = 16: 8 tokens per 128-row query tile
    (11, 200, 64, 2, 8),      # G = 32: 4 tokens per tile
    (1, 0, 8, 1, 16),         # one query at position 0 (a single key)
    (1, 5000, 16, 2, 32),     # one query deep into the sequence (a decode-like chunk)
])
def test_prefill_chunk_edge_shapes(NQ, q_start, Hq, Hkv, S):
    q, kc, vc, table, kv_len = _chunk_case(NQ, q_start, Hq, Hkv, S, seed=3 * NQ + q_start)
    scale = 1 / np.sqrt(128)
    ref = oracle.paged_prefill_chunk(q, q_start, kc, vc, table, kv_len, scale)
    got = _run(q, kc, vc, table, q_start, kv_len, scale)
    assert_close("bf16", got, ref, f"prefill NQ={NQ} q_start={q_start} G={Hq // Hkv} S={S}")


@pytest.mark.parametrize("kv,bits,flagged", [
    ("i8", 0x47C8, True),     # 102400: INT8 caches run the products on f16 operands, which cannot hold it
    ("e4m3", 0x47C8, False),  # FP8 caches scale each query row by a power of two first: any finite value is fine
    ("e4m3", 0x7F80, True),   # +inf is flagged on FP8 caches
])
def test_prefill_one_byte_cache_query_range(kv, bits, flagged):
    """A query value the tile's operands cannot carry raises PKV_DEVERR_Q_RANGE (0x10): beyond the f16 range for
    INT8 caches, non-finite for FP8 caches.  The rows without that value match the oracle either way."""
    q, kc, vc, table, kv_len = _chunk_case(40, 100, 8, 1, 16, seed=13, kv=kv)
    q = q.copy()
    q[5, 3, 7] = bits
    dq, dk, dv = to_device(q), to_device(kc), to_device(vc)
    out = torch.empty_like(dq)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_paged_prefill_chunk(out, dq, 100, dk, dv, B.CacheDesc.for_cache(dk, 0.25, 0.5), to_device(table),
                                kv_len, 1 / np.sqrt(128), err)
    torch.cuda.synchronize()
    assert bool(err.item() & 0x10) == flagged
    code = {"e4m3": oracle.E4M3, "i8": oracle.I8}[kv]
    rows = [0, 1, 20, 39]
    ref = oracle.paged_prefill_chunk(q, 100, kc, vc, table, kv_len, 1 / np.sqrt(128), rows=rows, cache_dtype=code,
                                     k_scale=0.25, v_scale=0.5)
    assert_close(kv, to_host(out)[rows], ref, "rows without the out-of-range query")


def test_fp8_prefill_query_rows_of_wide_range():
    """Query rows mixing values from 2^-12 to 2^6 (and exact zeros) over an FP8 cache: the tile scales each row by a
    power of two and splits it into two E4M3 parts, exact for values within 2^-10 of the row's largest and within
    2^-18 of it in absolute terms below that, so the chunk matches the oracle."""
    q, kc, vc, table, kv_len = _chunk_case(70, 250, 16, 2, 16, seed=17, kv="e4m3")
    rng = np.random.default_rng(5)
    mag = np.exp2(rng.integers(-12, 7, size=q.shape)).astype(np.float32)
    sign = np.where(rng.random(q.shape) < 0.5, -1.0, 1.0).astype(np.float32)
    vals = (mag * sign).astype(np.float32)
    vals[rng.random(q.shape) < 0.05] = 0.0
    q = (vals.view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16 (powers of two)
    dq, dk, dv = to_device(q), to_device(kc), to_device(vc)
    out = torch.empty_like(dq)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_paged_prefill_chunk(out, dq, 250, dk, dv, B.CacheDesc.for_cache(dk, 0.25, 0.5), to_device(table),
                                kv_len, 1 / np.sqrt(128), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle.paged_prefill_chunk(q, 250, kc, vc, table, kv_len, 1 / np.sqrt(128), cache_dtype=oracle.E4M3,
                                     k_scale=0.25, v_scale=0.5)
    assert_close("e4m3", to_host(out), ref, "wide-range query rows")
