"""GPU parity of the mixed-step launch (pkv_paged_attention_mixed) against the fp64 oracle.

Decode tokens (the first chunks, one query each at position kv_len - 1) and prefill chunks of different sequences in
one launch; every chunk is compared with the oracle, the decode tokens also with pkv_paged_attention_decode.
Tolerances are in parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import _binding as B
from paged_kv_cache_71_gb300 import workload as wl
from paged_kv_cache_71_gb300.block_manager import SequenceTables
from paged_kv_cache_71_gb300.runner import DeviceStep, to_device

from parity import assert_close, oracle_step, to_host

pytestmark = pytest.mark.gpu

SCALES = {"bf16": (1.0, 1.0), "e4m3": (0.25, 0.5), "i8": (1 / 32, 1 / 16)}
CODE = {"bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}


def _mixed_case(decode_lens, chunks, Hq, Hkv, seed, kv="bf16", tail_rows=2):
    """Decode tokens of sequences with decode_lens keys, then prefill chunks (q_start, n_q); one shuffled pool."""
    rng = np.random.default_rng(seed)
    S, D = 16, 128
    kv_lens = np.array(list(decode_lens) + [qs + nq for qs, nq in chunks], np.int32)
    n = len(kv_lens)
    NB = sum(-(-int(L) // S) for L in kv_lens) + 5
    t = SequenceTables(NB, S, free_order=rng.permutation(NB))
    for s, L in enumerate(kv_lens):
        t.prefill(s, int(L))
    tables = t.block_tables(list(range(n)))
    kc = wl.random_values(rng, (NB, S, Hkv, D), kv)
    vc = wl.random_values(rng, (NB, S, Hkv, D), kv)
    nq = [1] * len(decode_lens) + [c[1] for c in chunks]
    cu = np.zeros(n + 1, np.int32)
    cu[1:] = np.cumsum(nq)
    q = wl.random_values(rng, (int(cu[-1]) + tail_rows, Hq, D), "bf16")
    q_starts = np.array([L - 1 for L in decode_lens] + [qs for qs, _ in chunks], np.int32)
    return q, kc, vc, tables, cu, q_starts, kv_lens


def _run(case, num_decode, kv, head_scales=None):
    q, kc, vc, tables, cu, q_starts, kv_lens = case
    ks, vs = SCALES[kv]
    dq, dk, dv = to_device(q), to_device(kc), to_device(vc)
    if head_scales is None:
        desc = B.CacheDesc.for_cache(dk, ks, vs)
    else:
        dks, dvs = (torch.from_numpy(x).cuda() for x in head_scales)
        desc = B.CacheDesc.for_cache(dk, 1.0, 1.0, dks, dvs)
    out = torch.full_like(dq, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    need = pkv.pkv_paged_attention_mixed_workspace_size(desc, num_decode, q.shape[1])
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    pkv.pkv_paged_attention_mixed(out, dq, to_device(cu), to_device(q_starts), to_device(kv_lens), dk, dv, desc,
                                  to_device(tables), num_decode, 1 / np.sqrt(128), ws, err)
    torch.cuda.synchronize()
    return to_host(out), int(err.item())


def _check_all(case, num_decode, kv, what, head_scales=None):
    q, kc, vc, tables, cu, q_starts, kv_lens = case
    got, err = _run(case, num_decode, kv, head_scales)
    assert err == 0, hex(err)
    ks, vs = SCALES[kv]
    scales = dict(k_scale=ks, v_scale=vs) if head_scales is None else \
        dict(k_head_scales=head_scales[0], v_head_scales=head_scales[1])
    for s in range(len(kv_lens)):
        if cu[s + 1] == cu[s]:
            continue
        n_tab = -(-int(kv_lens[s]) // 16)
        ref = oracle.paged_prefill_chunk(q[cu[s]:cu[s + 1]], int(q_starts[s]), kc, vc, tables[s, :n_tab],
                                         int(kv_lens[s]), 1 / np.sqrt(128), cache_dtype=CODE[kv], **scales)
        assert_close(kv, got[cu[s]:cu[s + 1]], ref, f"{what}: chunk {s} (q_start {q_starts[s]}, kv_len {kv_lens[s]})")
    assert np.isnan(got[cu[-1]:]).all(), "rows outside every chunk were written"
    return got


DECODE = [1, 17, 300, 4100, 9000, 64]
CHUNKS = [(0, 200), (1000, 57), (129, 0), (5, 33), (128, 128)]


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "i8"])
@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (16, 4), (8, 8), (8, 4)])
def test_mixed_step_matches_oracle(kv, Hq, Hkv):
    case = _mixed_case(DECODE, CHUNKS, Hq, Hkv, seed=Hq + Hkv, kv=kv)
    _check_all(case, len(DECODE), kv, f"{kv} G={Hq // Hkv}")


@pytest.mark.parametrize("kv", ["e4m3", "i8"])
def test_mixed_step_per_head_scales(kv):
    """One-byte caches with one scale per KV head (replacing the per-tensor scale for both the decode tokens and the
    prefill chunks of the step)."""
    case = _mixed_case(DECODE, CHUNKS, 64, 8, seed=31, kv=kv)
    rng = np.random.default_rng(32)
    base = SCALES[kv]
    head = (np.float32(base[0]) * rng.uniform(0.5, 2.0, 8).astype(np.float32),
            np.float32(base[1]) * rng.uniform(0.5, 2.0, 8).astype(np.float32))
    _check_all(case, len(DECODE), kv, f"{kv} per-head scales", head_scales=head)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_mixed_step_odd_kv_head_count(kv):
    """Three KV heads in groups of two: the decode's work units and the tile slots run per KV head, at any count."""
    case = _mixed_case([5, 2000, 33], [(0, 70), (400, 9)], 6, 3, seed=33, kv=kv)
    _check_all(case, 3, kv, f"{kv} Hkv=3")


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_mixed_step_decode_only_and_prefill_only(kv):
    dec = _mixed_case([3000, 1, 77, 16, 15000], [], 64, 8, seed=3, kv=kv)
    _check_all(dec, 5, kv, "decode tokens only")
    pf = _mixed_case([], [(0, 300), (800, 40)], 64, 8, seed=4, kv=kv)
    _check_all(pf, 0, kv, "prefill chunks only")


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "i8"])
def test_more_prefill_tiles_than_sms(kv):
    """6000 prefill tokens at G = 8 need 188 tile slots per KV head: every CTA runs several prefill tiles (TMEM
    allocated and freed per tile) before it joins the decode."""
    case = _mixed_case([2000, 33, 700], [(0, 3000), (4000, 3000)], 64, 8, seed=21, kv=kv)
    q, kc, vc, tables, cu, q_starts, kv_lens = case
    got, err = _run(case, 3, kv)
    assert err == 0, hex(err)
    ks, vs = SCALES[kv]
    rows_by_chunk = {3: [0, 1, 31, 32, 1500, 2999], 4: [0, 777, 2998, 2999]}
    for s in range(3):
        ref = oracle.paged_prefill_chunk(q[s:s + 1], int(q_starts[s]), kc, vc, tables[s, :-(-int(kv_lens[s]) // 16)],
                                         int(kv_lens[s]), 1 / np.sqrt(128), cache_dtype=CODE[kv], k_scale=ks,
                                         v_scale=vs)
        assert_close(kv, got[s:s + 1], ref, f"{kv} decode token {s}")
    for s, rows in rows_by_chunk.items():
        n_tab = -(-int(kv_lens[s]) // 16)
        ref = oracle.paged_prefill_chunk(q[cu[s]:cu[s + 1]], int(q_starts[s]), kc, vc, tables[s, :n_tab],
                                         int(kv_lens[s]), 1 / np.sqrt(128), rows=rows, cache_dtype=CODE[kv],
                                         k_scale=ks, v_scale=vs)
        assert_close(kv, got[cu[s] + np.array(rows)], ref, f"{kv} chunk {s} sampled rows")


def test_decode_tokens_match_the_decode_call():
    """The decode tokens of a mixed step and the same sequences through pkv_paged_attention_decode agree within
    the tolerance (same tensor-core arithmetic, different work split)."""
    case = _mixed_case(DECODE, CHUNKS, 64, 8, seed=9, kv="e4m3")
    q, kc, vc, tables, cu, q_starts, kv_lens = case
    got, err = _run(case, len(DECODE), "e4m3")
    assert err == 0
    nd = len(DECODE)
    dk, dv = to_device(kc), to_device(vc)
    desc = B.CacheDesc.for_cache(dk, *SCALES["e4m3"])
    dq = to_device(q[:nd])
    out = torch.empty_like(dq)
    ws = torch.zeros(pkv.pkv_paged_attention_workspace_size(desc, nd, 64, 0), dtype=torch.uint8, device="cuda")
    pkv.pkv_paged_attention_decode(out, dq, dk, dv, desc, to_device(tables[:nd]), to_device(kv_lens[:nd]),
                                   1 / np.sqrt(128), 0, 0, ws)
    torch.cuda.synchronize()
    assert np.abs(to_host(out) - got[:nd]).max() < 6e-2


def test_decode_token_not_at_the_last_position_is_flagged():
    case = list(_mixed_case([40, 50], [(0, 20)], 16, 4, seed=12))
    case[5] = case[5].copy()
    case[5][1] = 30  # the second decode token's query is not at kv_len - 1
    _, err = _run(tuple(case), 2, "bf16")
    assert err & B.DEVERR_BAD_LENGTH


@pytest.mark.parametrize("name", ["llama70b_mixed_fp8", "llama70b_mixed_bf16"])
def test_llama70b_mixed_step(name):
    """The Llama-70B mixed step (48 decode tokens over 4096..32768 keys, the 512-token chunk at 8192..8703) in one
    launch: every decode token and 64 sampled chunk rows against the oracle."""
    w = wl.make(name)
    kind = "e4m3" if w.kv_dtype == "e4m3" else "bf16"
    st = DeviceStep(w)
    st.write()
    torch.cuda.synchronize()
    pf = w.prefill
    nd = w.num_seqs
    lens = w.context_lens.astype(np.int64)
    cu = np.concatenate([np.arange(nd + 1), [nd + pf.q.shape[0]]]).astype(np.int32)
    q_starts = np.concatenate([lens - 1, [pf.q_start]]).astype(np.int32)
    kv_lens = np.concatenate([lens, [pf.kv_len]]).astype(np.int32)
    MB = max(w.block_tables.shape[1], pf.block_table.shape[0])
    tables = np.full((nd + 1, MB), -1, np.int32)
    tables[:nd, : w.block_tables.shape[1]] = w.block_tables
    tables[nd, : pf.block_table.shape[0]] = pf.block_table
    q_all = torch.cat([st.q, st.pf_q], dim=0).contiguous()
    out = torch.full_like(q_all, float("nan"))
    need = pkv.pkv_paged_attention_mixed_workspace_size(st.cache, nd, w.num_q_heads)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    pkv.pkv_paged_attention_mixed(out, q_all, to_device(cu), to_device(q_starts), to_device(kv_lens), st.k_cache,
                                  st.v_cache, st.cache, to_device(tables), nd, w.scale, ws, st.err)
    torch.cuda.synchronize()
    assert st.device_error() == 0
    got = to_host(out)
    kc, vc, ref = oracle_step(w)
    assert_close(kind, got[:nd], ref, f"{name}: decode tokens")
    rows = np.random.default_rng(1).choice(pf.q.shape[0], 64, replace=False)
    pref = oracle.paged_prefill_chunk(pf.q, pf.q_start, kc, vc, pf.block_table, pf.kv_len, w.scale, rows=rows,
                                      cache_dtype=CODE[kind], k_scale=w.k_scale, v_scale=w.v_scale)
    assert_close(kind, got[nd + rows], pref, f"{name}: chunk rows")
