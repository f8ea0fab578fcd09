"""GPU parity of paged decode attention against the fp64 oracle.

Small cases are compared in full; the full-size batches in the launch
configuration the benchmark times are compared on sampled sequences that
include the longest and the shortest.  Tolerances are in parity.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import _binding as B
from paged_kv_cache_71_gb300 import workload as wl
from paged_kv_cache_71_gb300.block_manager import SequenceTables
from paged_kv_cache_71_gb300.runner import DeviceStep, to_device

from parity import assert_close, host_bits, oracle_step, to_host

pytestmark = pytest.mark.gpu


def _run(w, num_splits=0):
    st = DeviceStep(w, num_splits=num_splits)
    st.step()
    torch.cuda.synchronize()
    return st


def _random_workload(lens, Hq, Hkv, D, S, kv, q, seed, extra_blocks=7):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int64)
    need = int(sum(-(-int(L) // S) for L in lens))
    NB = need + extra_blocks
    alloc = SequenceTables(NB, S, free_order=rng.permutation(NB))
    slots = []
    for s, L in enumerate(lens):
        alloc.prefill(s, int(L) - 1)
        slots.append(alloc.next_slot(s))
    k_cache = wl.random_values(rng, (NB, S, Hkv, D), kv)
    v_cache = wl.random_values(rng, (NB, S, Hkv, D), kv)
    qa = wl.random_values(rng, (len(lens), Hq, D), q)
    kn = wl.random_values(rng, (len(lens), Hkv, D), q)
    vn = wl.random_values(rng, (len(lens), Hkv, D), q)
    sc = {"e4m3": wl.FP8_SCALE, "i8": wl.INT8_SCALE}.get(kv, 1.0)
    return wl.Workload("random", seed, Hq, Hkv, D, S, kv, q, sc, sc, qa, k_cache, v_cache,
                       alloc.block_tables(list(range(len(lens)))), lens.astype(np.int32), kn, vn,
                       np.array(slots, np.int64), np.zeros((0, 2), np.int64))


def test_tiny_config_all_split_modes():
    w = wl.tiny()
    kc, vc, ref = oracle_step(w)
    for ns in (0, 1, 2, 3, 9):
        st = _run(w, ns)
        assert st.device_error() == 0
        np.testing.assert_array_equal(host_bits(st.k_cache), kc)
        assert_close("f32", to_host(st.out), ref, f"tiny splits={ns}")


LENS = [1, 3, 4, 5, 15, 16, 17, 31, 33, 64, 100, 257]


@pytest.mark.parametrize("kv,q", [("f32", "f32"), ("bf16", "bf16"), ("e4m3", "bf16"), ("i8", "bf16")])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_shapes(kv, q, G, D):
    S = 16 if D == 128 else 8
    Hkv = 2
    w = _random_workload(LENS, G * Hkv, Hkv, D, S, kv, q, seed=G * 1000 + D)
    _, _, ref = oracle_step(w)
    for ns in (0, 1, 3):
        st = _run(w, ns)
        assert st.device_error() == 0
        assert_close(kv, to_host(st.out), ref, f"G={G} D={D} {kv} splits={ns}")


@pytest.mark.parametrize("kv,G", [("bf16", 4), ("bf16", 8), ("e4m3", 4), ("i8", 8)])
@pytest.mark.parametrize("S", [4, 8, 16, 32])
def test_decode_block_sizes(S, kv, G):
    """Every block size, ragged last blocks; the tensor-core form (one-byte caches, bf16 at G = 8) runs on 16-token
    MMA tiles (S = 32: two per block, S < 16: one partly filled)."""
    w = _random_workload([1, S - 1, S, S + 1, 3 * S + 2, 10 * S, 200], 2 * G, 2, 128, S, kv, "bf16", seed=S + G)
    _, _, ref = oracle_step(w)
    for ns in (0, 1, 4):
        st = _run(w, ns)
        assert st.device_error() == 0
        assert_close(kv, to_host(st.out), ref, f"S={S} {kv} splits={ns}")


@pytest.mark.parametrize("kv", ["e4m3", "i8", "bf16"])
def test_group_of_one_with_split_sequences(kv):
    """G = 1 over long sequences cut between workers: a worker's second segment writes its split-KV record to the odd
    slot, whose start is only 8-byte aligned when a record is G * (D + 2) floats with G = 1."""
    w = _random_workload([3000, 5000, 1000, 7000, 17], 4, 4, 128, 16, kv, "bf16", seed=101)
    _, _, ref = oracle_step(w)
    for ns in (0, 2, 5):
        st = _run(w, ns)
        assert st.device_error() == 0
        assert_close(kv, to_host(st.out), ref, f"G=1 {kv} splits={ns}")


@pytest.mark.parametrize("kv,G", [("e4m3", 1), ("i8", 4), ("e4m3", 8), ("bf16", 8)])
def test_odd_kv_head_count(kv, G):
    """Three KV heads: the tensor-core form takes KV heads in pairs only when their count is even, so this runs one
    head per work unit; ragged lengths, every split mode."""
    w = _random_workload([1, 15, 16, 17, 300, 2100], 3 * G, 3, 128, 16, kv, "bf16", seed=70 + G)
    _, _, ref = oracle_step(w)
    for ns in (0, 1, 3):
        st = _run(w, ns)
        assert st.device_error() == 0
        assert_close(kv, to_host(st.out), ref, f"Hkv=3 G={G} {kv} splits={ns}")


@pytest.mark.parametrize("kv", ["e4m3", "i8"])
def test_one_byte_decode_query_out_of_f16_range_is_flagged(kv):
    """Decode over a one-byte cache takes q to f16 for the tensor-core products: a query value of 2^17 (a bf16 value
    beyond f16) must set PKV_DEVERR_Q_RANGE in the device error word; in-range queries leave it clear."""
    w = _random_workload([40, 7, 300], 8, 2, 128, 16, kv, "bf16", seed=91)
    st = _run(w, 0)
    assert st.device_error() == 0
    q = w.q.copy()
    q[1, 3, 17] = np.uint16(0x4800)  # bf16 bits of 2^17 = 131072
    w.q = q
    st = _run(w, 0)
    assert st.device_error() & B.DEVERR_Q_RANGE


def test_split_modes_agree_closely():
    """Any split gives the same attention up to fp32 rounding order."""
    w = _random_workload([700, 1, 2048, 333, 5000], 16, 4, 64, 16, "f32", "f32", seed=77)
    outs = [to_host(_run(w, ns).out) for ns in (0, 1, 2, 7, 64)]
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=2e-6)


def test_empty_sequence_gives_zero_row():
    w = _random_workload([5, 9, 33], 8, 2, 128, 16, "bf16", "bf16", seed=3)
    w.context_lens = w.context_lens.copy()
    w.context_lens[1] = 0
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[1] = -1
    _, _, ref = oracle_step(w)
    for ns in (0, 1):
        st = _run(w, ns)
        out = to_host(st.out)
        assert (out[1] == 0).all()
        assert_close("bf16", out, ref, "empty row")


@pytest.mark.parametrize("kv,D,S,G", [("f32", 64, 8, 4), ("bf16", 64, 8, 4), ("bf16", 128, 16, 8), ("bf16", 128, 4, 8),
                                      ("e4m3", 128, 16, 4), ("e4m3", 128, 4, 4), ("i8", 128, 8, 4), ("i8", 128, 32, 8)])
def test_poisoned_unused_slots_do_not_leak(kv, D, S, G):
    """NaN (the largest code for INT8) in every slot that no sequence owns (tails of last blocks, free blocks)
    changes nothing: stale rows of a partly filled tile must not reach the scores or P.V."""
    q = "f32" if kv == "f32" else "bf16"
    w = _random_workload([13, 2, 40, 77], 2 * G, 2, D, S, kv, q, seed=21, extra_blocks=12)
    _, _, ref = oracle_step(w)
    clean = to_host(_run(w, 0).out)
    S = w.block_size
    owned = np.zeros((w.num_blocks, S), bool)
    for s in range(w.num_seqs):
        for p in range(int(w.context_lens[s])):
            owned[w.block_tables[s, p // S], p % S] = True
    nan = {"f32": np.float32(np.nan), "bf16": np.uint16(0x7FC0), "e4m3": np.uint8(0x7F), "i8": np.uint8(0x7F)}[kv]
    for cache in (w.k_cache, w.v_cache):
        cache[~owned] = nan
    for ns in (0, 1, 2):
        out = to_host(_run(w, ns).out)
        assert np.isfinite(out).all()
        assert_close(kv, out, ref, f"poisoned splits={ns}")
        if ns == 0:
            np.testing.assert_array_equal(out, clean)


def test_bad_block_id_and_bad_length_are_flagged():
    w = _random_workload([20, 20, 20, 20], 8, 2, 64, 4, "f32", "f32", seed=31)
    w.block_tables = w.block_tables.copy()
    w.block_tables[1, 2] = w.num_blocks + 5        # bad id inside sequence 1's context
    w.context_lens = w.context_lens.copy()
    w.context_lens[2] = w.block_tables.shape[1] * w.block_size + 1  # longer than its table
    st = _run(w, 1)
    e = st.device_error()
    assert e & B.DEVERR_BAD_BLOCK and e & B.DEVERR_BAD_LENGTH
    out = to_host(st.out)
    good = [0, 3]
    _, _, ref = oracle_step(w, seqs=good)
    assert_close("f32", out[good], ref, "sequences next to bad ones")
    assert (out[2] == 0).all()


def test_workspace_and_alignment_errors():
    w = _random_workload([10, 20], 8, 2, 64, 8, "bf16", "bf16", seed=4)
    st = DeviceStep(w, num_splits=0)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_paged_attention_decode(st.out, st.q, st.k_cache, st.v_cache, st.cache, st.block_tables,
                                       st.context_lens, w.scale, 0, 0, st.workspace[:16], st.err)
    assert ei.value.status == 4
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_paged_attention_decode(st.out, st.q, st.k_cache, st.v_cache, st.cache, st.block_tables,
                                       st.context_lens, w.scale, 0, 0, None, st.err)
    assert ei.value.status == 4
    assert pkv.pkv_paged_attention_workspace_size(st.cache, 2, 8, 1) == 0


# ---------------------------------------------------------------- the benchmark's batches

def _sample(w, k=24, seed=0):
    rng = np.random.default_rng(seed)
    L = w.context_lens
    pick = {int(np.argmax(L)), int(np.argmin(L))}
    pick |= set(rng.choice(w.num_seqs, size=min(k, w.num_seqs), replace=False).tolist())
    return sorted(pick)


@pytest.mark.parametrize("name", ["llama2_7b", "llama3_8b_gqa", "prefix_shared", "llama70b_mixed_bf16",
                                  "llama70b_mixed_fp8", "llama3_8b_gqa_int8"])
def test_full_size_batches_sampled(name):
    w = wl.make(name)
    seqs = _sample(w)
    kc, vc, ref = oracle_step(w, seqs=seqs)
    st = _run(w, 0)
    assert st.device_error() == 0
    out = to_host(st.out)
    assert_close(w.kv_dtype, out[seqs], ref, name)
    # the cache write is bit-exact for every new token
    gk = host_bits(st.k_cache)
    S = w.block_size
    for i, sl in enumerate(w.slot_mapping):
        np.testing.assert_array_equal(gk[sl // S, sl % S], kc[sl // S, sl % S])
    # the output is finite everywhere, and a split-free run agrees on every sequence
    assert np.isfinite(out).all()
    st1 = _run(w, 1)
    o1 = to_host(st1.out)
    assert np.abs(o1 - out).max() < (6e-2 if w.kv_dtype == "e4m3" else 3e-2)


def test_largest_batch_and_one_more_is_rejected():
    """num_seqs = 8192 (the largest batch one call takes) with short ragged contexts; 8193 is refused on the host."""
    rng = np.random.default_rng(8192)
    lens = rng.integers(1, 40, size=8192)
    w = _random_workload(lens, 8, 2, 64, 8, "bf16", "bf16", seed=81)
    st = _run(w)
    assert st.device_error() == 0
    seqs = [0, 1, 4095, 8190, 8191]
    kc, vc, ref = oracle_step(w, seqs=seqs)
    assert_close("bf16", to_host(st.out)[seqs], ref, "8192 sequences, sampled")
    q = torch.zeros((8193, 8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_paged_attention_decode(torch.empty_like(q), q, st.k_cache, st.v_cache, st.cache,
                                       torch.zeros((8193, 1), dtype=torch.int32, device="cuda"),
                                       torch.ones(8193, dtype=torch.int32, device="cuda"), 0.1, num_splits=1)
    assert ei.value.status == 2


def test_one_very_long_sequence_splits():
    """A single 131072-token sequence (8192 blocks): the split-KV plan spreads it over every SM and merges."""
    w = _random_workload([131072], 8, 2, 128, 16, "bf16", "bf16", seed=131)
    kc, vc, ref = oracle_step(w)
    for ns in (0, 1, 64):
        st = _run(w, ns)
        assert st.device_error() == 0
        assert_close("bf16", to_host(st.out), ref, f"131072-token sequence, splits={ns}")


@pytest.mark.parametrize("G", [4, 8])
def test_int8_long_sequence_of_small_codes(G):
    """One 32768-token INT8 sequence reduced by one worker and by the split plan: small codes in [-3, 3] with
    unit scales, then only the extreme codes -127 and 127, stay within the INT8 tolerance."""
    for lo, hi, seed in ((-3, 3, 90 + G), (-127, 127, 95 + G)):
        w = _random_workload([32768, 3, 40], 2 * G, 2, 128, 16, "i8", "bf16", seed=seed)
        rng = np.random.default_rng(seed)
        if hi == 3:
            w.k_cache = rng.integers(lo, hi + 1, w.k_cache.shape).astype(np.int8)
            w.v_cache = rng.integers(lo, hi + 1, w.v_cache.shape).astype(np.int8)
        else:
            w.k_cache = rng.choice(np.array([lo, hi], np.int8), w.k_cache.shape)
            w.v_cache = rng.choice(np.array([lo, hi], np.int8), w.v_cache.shape)
        w.k_scale = w.v_scale = 1.0 / 16 if hi == 127 else 1.0
        _, _, ref = oracle_step(w)
        for ns in (1, 0):
            st = _run(w, ns)
            assert st.device_error() == 0
            assert_close("i8", to_host(st.out), ref, f"INT8 codes in [{lo}, {hi}], G={G}, splits={ns}")


def test_unsupported_group_is_refused():
    w = _random_workload([20, 7], 32, 2, 128, 16, "bf16", "bf16", seed=16)  # G = 16
    with pytest.raises(pkv.PkvError) as ei:
        st = DeviceStep(w, num_splits=1)
        st.attend()
    assert ei.value.status == 2
