"""Pins of the CPU oracle against things other than itself.

Each test ties one oracle function to a value the pages print (golden
fixtures under tests/golden/, each with its citation), a closed form, an
invariant, or a library routine that computes the same definition
(torch's float64 scaled_dot_product_attention, torch's float8/bfloat16
casts).  Runs without a GPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_71_gb300.block_manager import SequenceTables
from paged_kv_cache_71_gb300.workload import random_values


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ indexing


def test_worked_example_lookup(golden_dir):
    """Token A.t9 -> block 5, offset 1; every position lands in the block the example lists."""
    g = _load(golden_dir, "worked_example_block_table.json")
    S = g["block_size"]
    q = g["query"]
    seq = g["sequences"][q["sequence"]]
    blk, off = oracle.lookup(np.array(seq["block_table"], np.int32), q["position"], S)
    assert (blk, off) == (q["physical_block"], q["offset"])
    for bid, content in g["pool"].items():
        if content is None:
            continue
        name, first, last = content
        table = np.array(g["sequences"][name]["block_table"], np.int32)
        for p in range(first, last + 1):
            assert oracle.lookup(table, p, S)[0] == int(bid)
    # wasted slots: S - used in each partial last block
    for name, seqd in g["sequences"].items():
        n = seqd["num_tokens"]
        last = seqd["block_table"][-1]
        used = n - (len(seqd["block_table"]) - 1) * S
        assert S - used == g["wasted_slots"].get(str(last), 0)


def test_worked_example_gather_via_cache_write(golden_dir):
    """Writing A's and B's tokens through slot = block*S + offset and gathering them back in
    logical order reproduces the sequences; free blocks stay untouched."""
    g = _load(golden_dir, "worked_example_block_table.json")
    S, Hkv, D, NB = g["block_size"], 1, 64, 8
    kc = np.full((NB, S, Hkv, D), -7.0, np.float32)
    vc = kc.copy()
    for name, seqd in g["sequences"].items():
        n = seqd["num_tokens"]
        table = np.array(seqd["block_table"], np.int32)
        slots = np.array([(lambda bo: bo[0] * S + bo[1])(oracle.lookup(table, p, S)) for p in range(n)], np.int64)
        tag = 100.0 if name == "A" else 200.0
        kn = (tag + np.arange(n, dtype=np.float32))[:, None, None] * np.ones((1, Hkv, D), np.float32)
        oracle.reshape_and_cache(kn, -kn, slots, kc, vc)
    for bid, content in g["pool"].items():
        b = int(bid)
        if content is None:
            assert (kc[b] == -7.0).all()
            continue
        name, first, last = content
        tag = 100.0 if name == "A" else 200.0
        for p in range(first, last + 1):
            assert (kc[b, p % S] == tag + p).all() and (vc[b, p % S] == -(tag + p)).all()


def test_allocator_simulation(golden_dir):
    g = _load(golden_dir, "allocator_simulation.json")
    a = SequenceTables(g["num_blocks"], g["block_size"])
    a.prefill("p", 6)
    a.fork("p", "s1")
    a.fork("p", "s2")
    for s in ("s1", "s2"):
        a.next_slot(s)
    assert {s: a.table(s) for s in ("p", "s1", "s2")} == g["after_appends"]["tables"]
    assert a.pool.num_free == g["after_appends"]["free"]
    assert [list(p) for p in a.drain_copies()] == g["cow_pairs"]
    a.drop("p")
    assert a.pool.refcount.tolist() == g["after_free_p"]["ref"]
    assert a.pool.num_free == g["after_free_p"]["free"]


def test_allocator_exhaustion_raises():
    a = SequenceTables(2, 4)
    a.prefill("x", 8)
    with pytest.raises(MemoryError):
        a.next_slot("x")


def test_block_count_self_test(golden_dir):
    g = _load(golden_dir, "block_count_self_test.json")
    a = SequenceTables(100, g["block_size"])
    a.prefill("r", g["num_tokens"])
    assert len(a.table("r")) == g["blocks"]
    assert len(a.table("r")) * g["block_size"] == g["slots"]
    assert g["slots"] - g["num_tokens"] == g["wasted"] < g["block_size"]
    # the last token sits in the last table entry, at offset (n-1) % S
    blk, off = oracle.lookup(np.array(a.table("r"), np.int32), g["num_tokens"] - 1, g["block_size"])
    assert blk == a.table("r")[-1] and off == (g["num_tokens"] - 1) % g["block_size"]


# ------------------------------------------------------------------ element formats


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert (ours[~nan] == ref[~nan]).all()
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encode_round_trip_and_grid():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes).astype(np.float32)
    back = oracle.f32_to_e4m3(vals)
    assert (back == codes).all()  # includes -0 -> 0x80
    # every midpoint between neighbouring codes and points either side of it:
    pos = np.sort(oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8)))
    mids = (pos[:-1] + pos[1:]) / 2
    grid = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                           np.nextafter(mids.astype(np.float32), np.float32(1e9)),
                           np.linspace(0, 447.9, 3001)]).astype(np.float32)
    grid = np.concatenate([grid, -grid])
    ours = oracle.f32_to_e4m3(grid)
    ref = torch.from_numpy(grid).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (ours == ref).all()


def test_e4m3_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf], np.float32)
    assert list(oracle.f32_to_e4m3(x)) == [0x7E] * 6 + [0xFE, 0xFE]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(4000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 4000),
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.3895314e38, np.inf, -np.inf,
                                  1e-40, -1e-45], np.float32)]).astype(np.float32)
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (ours == ref).all()
    back = oracle.bf16_to_f64(ours)
    assert (back == torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy()).all()


# ------------------------------------------------------------------ attention


def _scatter_problem(rng, lens, Hq, Hkv, D, S, extra_blocks=3, dtype=np.float64):
    """Random contiguous K/V per sequence, placed into a paged pool by a shuffled allocator."""
    need = sum(-(-L // S) for L in lens)
    NB = need + extra_blocks
    alloc = SequenceTables(NB, S, free_order=rng.permutation(NB))
    kc = rng.standard_normal((NB, S, Hkv, D)).astype(np.float32)
    vc = rng.standard_normal((NB, S, Hkv, D)).astype(np.float32)
    Ks, Vs = [], []
    for s, L in enumerate(lens):
        alloc.prefill(s, L)
        K = rng.standard_normal((L, Hkv, D)).astype(np.float32)
        V = rng.standard_normal((L, Hkv, D)).astype(np.float32)
        slots = np.array([alloc.slot(s, p) for p in range(L)], np.int64)
        oracle.reshape_and_cache(K, V, slots, kc, vc)
        Ks.append(K)
        Vs.append(V)
    bt = alloc.block_tables(list(range(len(lens))))
    q = rng.standard_normal((len(lens), Hq, D)).astype(np.float32)
    return q, kc, vc, bt, np.array(lens, np.int32), Ks, Vs, alloc


def _sdpa(qrow, K, V, scale, G, causal_limit=None):
    """torch float64 SDPA for one query position over contiguous K/V [L, Hkv, D]."""
    qt = torch.from_numpy(qrow.astype(np.float64))[:, None, :]            # [Hq, 1, D]
    kt = torch.from_numpy(K.astype(np.float64)).permute(1, 0, 2)          # [Hkv, L, D]
    vt = torch.from_numpy(V.astype(np.float64)).permute(1, 0, 2)
    kt = kt.repeat_interleave(G, dim=0)
    vt = vt.repeat_interleave(G, dim=0)
    if causal_limit is not None:
        kt, vt = kt[:, :causal_limit], vt[:, :causal_limit]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("Hq,Hkv,S", [(4, 2, 4), (8, 8, 16), (8, 1, 8)])
def test_decode_matches_sdpa_on_unpaged_arrays(Hq, Hkv, S):
    rng = np.random.default_rng(11 + Hq + S)
    lens = [10, 6, 33, 1, 17]
    D = 32
    q, kc, vc, bt, cl, Ks, Vs, _ = _scatter_problem(rng, lens, Hq, Hkv, D, S)
    scale = 1 / math.sqrt(D)
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, scale)
    for s in range(len(lens)):
        ref = _sdpa(q[s], Ks[s], Vs[s], scale, Hq // Hkv)
        np.testing.assert_allclose(out[s], ref, rtol=1e-12, atol=1e-12)


def test_decode_gqa_grouping_is_contiguous():
    """q head hq reads kv head hq // G: swapping the KV heads changes exactly the matching groups."""
    rng = np.random.default_rng(5)
    q, kc, vc, bt, cl, *_ = _scatter_problem(rng, [9, 14], 4, 2, 16, 4)
    a = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.25)
    kc2, vc2 = kc[:, :, ::-1].copy(), vc[:, :, ::-1].copy()
    b = oracle.paged_attention_decode(q, kc2, vc2, bt, cl, 0.25)
    q2 = q[:, [2, 3, 0, 1]].copy()
    c = oracle.paged_attention_decode(q2, kc2, vc2, bt, cl, 0.25)
    assert not np.allclose(a, b)
    np.testing.assert_array_equal(a, c[:, [2, 3, 0, 1]])


def test_decode_single_token_returns_v0():
    rng = np.random.default_rng(1)
    q, kc, vc, bt, cl, Ks, Vs, _ = _scatter_problem(rng, [1, 1], 4, 2, 64, 4)
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.125)
    for s in range(2):
        for hq in range(4):
            assert (out[s, hq] == Vs[s][0, hq // 2].astype(np.float64)).all()


def test_decode_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    q, kc, vc, bt, cl, Ks, Vs, alloc = _scatter_problem(rng, [23], 2, 1, 16, 4)
    kc[:] = 0.5  # every key identical (also the unused slots)
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 1.0)
    np.testing.assert_allclose(out[0, 0], Vs[0][:, 0].astype(np.float64).mean(0), rtol=0, atol=1e-13)


def test_decode_dominant_logit_selects_its_value():
    rng = np.random.default_rng(4)
    q, kc, vc, bt, cl, Ks, Vs, alloc = _scatter_problem(rng, [30], 1, 1, 8, 4)
    kc[:] = 0.0
    q[:] = 1.0
    slot = alloc.slot(0, 17)
    kc[slot // 4, slot % 4, 0, :] = 100.0
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl, 1.0)
    np.testing.assert_allclose(out[0, 0], Vs[0][17, 0], rtol=0, atol=1e-12)


def test_decode_block_permutation_invariance():
    rng = np.random.default_rng(6)
    q, kc, vc, bt, cl, *_ = _scatter_problem(rng, [13, 40, 3], 4, 2, 32, 4, extra_blocks=5)
    a = oracle.paged_attention_decode(q, kc, vc, bt, cl, 0.2)
    perm = rng.permutation(kc.shape[0])       # new id of old block b is perm[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    b = oracle.paged_attention_decode(q, kc2, vc2, bt2, cl, 0.2)
    np.testing.assert_array_equal(a, b)


def test_decode_shared_blocks_equal_private_copies():
    rng = np.random.default_rng(8)
    S, Hkv, D = 4, 2, 16
    a = SequenceTables(20, S, free_order=rng.permutation(20))
    a.prefill("p", 10)
    a.fork("p", "c")
    a.next_slot("c")  # CoW of the partial block
    a.next_slot("p")
    kc = rng.standard_normal((20, S, Hkv, D)).astype(np.float32)
    vc = rng.standard_normal((20, S, Hkv, D)).astype(np.float32)
    for src, dst in a.drain_copies():
        kc[dst], vc[dst] = kc[src], vc[src]
    # make the two new tokens equal so both sequences hold the same logical data
    for sid in ("p", "c"):
        sl = a.slot(sid, 10)
        kc[sl // S, sl % S] = 0.25
        vc[sl // S, sl % S] = -0.5
    bt = a.block_tables(["p", "c"])
    assert bt[0, 0] == bt[1, 0] and bt[0, 2] != bt[1, 2]
    q = np.repeat(rng.standard_normal((1, 4, D)).astype(np.float32), 2, axis=0)
    out = oracle.paged_attention_decode(q, kc, vc, bt, np.array([11, 11], np.int32), 0.3)
    np.testing.assert_array_equal(out[0], out[1])


def test_decode_empty_sequence_is_zero_and_subset_selection():
    rng = np.random.default_rng(9)
    q, kc, vc, bt, cl, *_ = _scatter_problem(rng, [5, 7, 9], 2, 1, 8, 4)
    cl2 = cl.copy()
    cl2[1] = 0
    out = oracle.paged_attention_decode(q, kc, vc, bt, cl2, 0.3)
    assert (out[1] == 0).all()
    sub = oracle.paged_attention_decode(q, kc, vc, bt, cl2, 0.3, seqs=[2, 0])
    np.testing.assert_array_equal(sub[0], out[2])
    np.testing.assert_array_equal(sub[1], out[0])


def test_decode_bf16_and_fp8_widen_exactly():
    """bf16 caches read as their exact values; e4m3 caches as code * scale."""
    rng = np.random.default_rng(10)
    q, kc, vc, bt, cl, *_ = _scatter_problem(rng, [6, 11], 4, 2, 16, 4)
    kb, vb = oracle.f32_to_bf16(kc), oracle.f32_to_bf16(vc)
    ref = oracle.paged_attention_decode(q, oracle.bf16_to_f64(kb).astype(np.float32),
                                        oracle.bf16_to_f64(vb).astype(np.float32), bt, cl, 0.25)
    out = oracle.paged_attention_decode(q, kb, vb, bt, cl, 0.25)
    np.testing.assert_array_equal(out, ref)
    k8 = random_values(rng, kc.shape, "e4m3")
    v8 = random_values(rng, vc.shape, "e4m3")
    out8 = oracle.paged_attention_decode(q, k8, v8, bt, cl, 0.25, k_scale=0.5, v_scale=0.125)
    kf = (oracle.e4m3_to_f64(k8) * 0.5).astype(np.float32)
    vf = (oracle.e4m3_to_f64(v8) * 0.125).astype(np.float32)
    ref8 = oracle.paged_attention_decode(q, kf, vf, bt, cl, 0.25)
    np.testing.assert_allclose(out8, ref8, rtol=1e-13, atol=1e-13)


def test_prefill_chunk_matches_causal_sdpa():
    rng = np.random.default_rng(12)
    S, Hq, Hkv, D = 4, 4, 2, 16
    q_start, NQ = 32, 8
    kv_len = q_start + NQ
    q, kc, vc, bt, cl, Ks, Vs, _ = _scatter_problem(rng, [kv_len], Hq, Hkv, D, S)
    qc = rng.standard_normal((NQ, Hq, D)).astype(np.float32)
    out = oracle.paged_prefill_chunk(qc, q_start, kc, vc, bt[0], kv_len, 0.25)
    for i in range(NQ):
        ref = _sdpa(qc[i], Ks[0], Vs[0], 0.25, Hq // Hkv, causal_limit=q_start + i + 1)
        np.testing.assert_allclose(out[i], ref, rtol=1e-12, atol=1e-12)
    # the last query sees everything: equals decode with context q_start + NQ
    dec = oracle.paged_attention_decode(qc[NQ - 1:NQ].copy(), kc, vc, bt, np.array([kv_len], np.int32), 0.25)
    np.testing.assert_allclose(out[NQ - 1], dec[0], rtol=1e-13, atol=1e-13)
    rows = oracle.paged_prefill_chunk(qc, q_start, kc, vc, bt[0], kv_len, 0.25, rows=[3, 0])
    np.testing.assert_array_equal(rows[0], out[3])


# ------------------------------------------------------------------ cache writes and copies


def test_reshape_and_cache_skips_padding_and_flags_bad_slots():
    rng = np.random.default_rng(13)
    NB, S, Hkv, D = 4, 4, 2, 8
    kc = np.zeros((NB, S, Hkv, D), np.float32)
    vc = np.zeros_like(kc)
    kn = rng.standard_normal((3, Hkv, D)).astype(np.float32)
    st = oracle.reshape_and_cache(kn, kn, np.array([5, -1, NB * S], np.int64), kc, vc)
    assert st == 2
    assert (kc[1, 1] == kn[0]).all() and np.count_nonzero(kc) == np.count_nonzero(kn[0])


def test_reshape_and_cache_bf16_and_fp8_conversions():
    rng = np.random.default_rng(14)
    NB, S, Hkv, D = 3, 4, 2, 16
    kn = (rng.standard_normal((5, Hkv, D)) * 3).astype(np.float32)
    slots = np.array([0, 3, 6, 9, 11], np.int64)
    kb = np.zeros((NB, S, Hkv, D), np.uint16)
    vb = np.zeros_like(kb)
    oracle.reshape_and_cache(kn, kn, slots, kb, vb)
    ref = torch.from_numpy(kn).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for i, sl in enumerate(slots):
        assert (kb[sl // S, sl % S] == ref[i]).all()
    k8 = np.zeros((NB, S, Hkv, D), np.uint8)
    v8 = np.zeros_like(k8)
    oracle.reshape_and_cache(kn, kn, slots, k8, v8, k_scale=0.5, v_scale=0.25)
    for i, sl in enumerate(slots):
        y = (kn[i] / np.float32(0.5)).astype(np.float32)
        assert (k8[sl // S, sl % S] == torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()).all()
        y = (kn[i] / np.float32(0.25)).astype(np.float32)
        assert (v8[sl // S, sl % S] == torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()).all()


def test_copy_blocks_page_example(golden_dir):
    """The data copies that the allocator simulation's copy-on-write implies."""
    g = _load(golden_dir, "allocator_simulation.json")
    rng = np.random.default_rng(15)
    kc = rng.standard_normal((8, 4, 2, 8)).astype(np.float32)
    vc = rng.standard_normal((8, 4, 2, 8)).astype(np.float32)
    k0, v0 = kc.copy(), vc.copy()
    oracle.copy_blocks(kc, vc, np.array(g["cow_pairs"], np.int64))
    for src, dst in g["cow_pairs"]:
        assert (kc[dst] == k0[src]).all() and (vc[dst] == v0[src]).all()
    untouched = [b for b in range(8) if b not in {d for _, d in g["cow_pairs"]}]
    assert (kc[untouched] == k0[untouched]).all() and (vc[untouched] == v0[untouched]).all()
    assert oracle.copy_blocks(kc, vc, np.array([[0, 8]], np.int64)) == 3


def test_swap_blocks_round_trip_and_agrees_with_copy_blocks():
    rng = np.random.default_rng(16)
    dev_k = rng.standard_normal((10, 4, 2, 8)).astype(np.float32)
    dev_v = rng.standard_normal((10, 4, 2, 8)).astype(np.float32)
    host_k = np.zeros((6, 4, 2, 8), np.float32)
    host_v = np.zeros_like(host_k)
    out_pairs = np.array([[7, 0], [2, 5], [9, 3]], np.int64)
    oracle.swap_blocks(dev_k, dev_v, host_k, host_v, out_pairs)
    k2, v2 = np.zeros_like(dev_k), np.zeros_like(dev_v)
    oracle.swap_blocks(host_k, host_v, k2, v2, out_pairs[:, ::-1].copy())
    for src, _ in out_pairs:
        assert (k2[src] == dev_k[src]).all() and (v2[src] == dev_v[src]).all()
    # within one pool, a swap from a snapshot equals copy_blocks
    pairs = np.array([[1, 4], [3, 8]], np.int64)
    a_k, a_v = dev_k.copy(), dev_v.copy()
    oracle.copy_blocks(a_k, a_v, pairs)
    b_k, b_v = dev_k.copy(), dev_v.copy()
    oracle.swap_blocks(dev_k.copy(), dev_v.copy(), b_k, b_v, pairs)
    assert (a_k == b_k).all() and (a_v == b_v).all()
    assert oracle.swap_blocks(dev_k, dev_v, host_k, host_v, np.array([[0, 6]], np.int64)) == 3


def test_fnv1a64_published_vectors():
    """FNV-1a 64-bit test vectors from the algorithm's reference description."""
    assert oracle.fnv1a64(b"") == 0xCBF29CE484222325
    assert oracle.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert oracle.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hashes_chain_and_prefix_property():
    """Equal prefixes give equal block hashes; a change in block j changes hashes j.. only;
    partial last blocks get no hash; the chain is the stated two-level FNV-1a."""
    rng = np.random.default_rng(30)
    S = 4
    a = rng.integers(0, 32000, 23).astype(np.int32)
    b = a.copy()
    b[13] += 1                       # block 3 differs
    c = a[:9].copy()                 # 2 full blocks + 1 partial
    toks = np.concatenate([a, b, c])
    cu = np.array([0, 23, 46, 55], np.int64)
    h = oracle.block_hashes(toks, cu, S)
    ha, hb, hc = h[:5], h[5:10], h[10:]
    assert len(h) == 5 + 5 + 2
    assert (ha[:3] == hb[:3]).all() and (ha[3:] != hb[3:]).all()
    assert (hc == ha[:2]).all()
    # by hand, from the definition
    d0 = oracle.fnv1a64(a[:4].astype("<i4").tobytes())
    h0 = oracle.fnv1a64((0).to_bytes(8, "little") + d0.to_bytes(8, "little"))
    d1 = oracle.fnv1a64(a[4:8].astype("<i4").tobytes())
    h1 = oracle.fnv1a64(h0.to_bytes(8, "little") + d1.to_bytes(8, "little"))
    assert int(ha[0]) == h0 and int(ha[1]) == h1


def test_int8_encoder_matches_numpy_rint_and_clamp():
    grid = np.concatenate([np.arange(-130, 130, 0.25), np.arange(-3, 3, 0.5) + 1e-7,
                           np.array([127.5, -127.5, 1e9, -1e9, 0.0, -0.0])]).astype(np.float32)
    ours = oracle.f32_to_i8(grid)
    ref = np.clip(np.rint(grid.astype(np.float64)), -127, 127).astype(np.int8)
    np.testing.assert_array_equal(ours, ref)


def test_int8_cache_reads_code_times_scale():
    rng = np.random.default_rng(17)
    q, kc, vc, bt, cl, *_ = _scatter_problem(rng, [6, 11], 4, 2, 16, 4)
    k8 = random_values(rng, kc.shape, "i8")
    v8 = random_values(rng, vc.shape, "i8")
    out = oracle.paged_attention_decode(q, k8, v8, bt, cl, 0.25, k_scale=1 / 32, v_scale=1 / 16)
    ref = oracle.paged_attention_decode(q, (k8.astype(np.float32) / 32), (v8.astype(np.float32) / 16), bt, cl, 0.25)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    # the cache write quantises x / scale with ties to even
    kn = (rng.standard_normal((3, 2, 16)) * 2).astype(np.float32)
    kq = np.zeros((2, 4, 2, 16), np.int8)
    oracle.reshape_and_cache(kn, kn, np.array([0, 3, 6], np.int64), kq, kq.copy(), k_scale=1 / 32, v_scale=1.0)
    y = (kn / np.float32(1 / 32)).astype(np.float32)
    np.testing.assert_array_equal(kq[0, 0], np.clip(np.rint(y[0]), -127, 127))


def test_per_head_scales_write_codes_by_kv_head():
    """Head h of every token is quantised with its own scale: inputs built as (d + 1) * s_h give codes d + 1 in
    every head, which a wrong head index (or the per-tensor scale) would not."""
    Hkv, D, S = 3, 8, 4
    s_h = np.array([0.5, 0.125, 2.0], np.float32)
    kn = ((np.arange(D, dtype=np.float32) + 1)[None, None, :] * s_h[None, :, None]).repeat(2, axis=0)
    vn = -kn
    kc = np.zeros((2, S, Hkv, D), np.int8)
    vc = np.zeros_like(kc)
    oracle.reshape_and_cache(kn, vn, np.array([1, 6], np.int64), kc, vc, k_scale=1.0, v_scale=1.0,
                             k_head_scales=s_h, v_head_scales=s_h)
    want = np.arange(1, D + 1, dtype=np.int8)
    for slot in (1, 6):
        for h in range(Hkv):
            np.testing.assert_array_equal(kc[slot // S, slot % S, h], want)
            np.testing.assert_array_equal(vc[slot // S, slot % S, h], -want)
    # the E4M3 encoder takes the same per-head division
    k8 = np.zeros((2, S, Hkv, D), np.uint8)
    oracle.reshape_and_cache(kn, vn, np.array([1, 6], np.int64), k8, k8.copy(), cache_dtype=oracle.E4M3,
                             k_scale=1.0, v_scale=1.0, k_head_scales=s_h, v_head_scales=s_h)
    np.testing.assert_array_equal(oracle.e4m3_to_f64(k8[0, 1, 2]), np.arange(1, D + 1))


def test_per_head_scales_decode_closed_form():
    """Two cached tokens per head: key codes 0 and c, value codes a and b.  With per-head scales ks_h, vs_h the
    output of head h is vs_h * (a + b * e^z) / (1 + e^z), z = scale * (q . c) * ks_h."""
    Hkv, G, D, S = 2, 2, 4, 4
    ks = np.array([0.25, 1.0]); vs = np.array([0.5, 3.0])
    kc = np.zeros((1, S, Hkv, D), np.int8)
    vc = np.zeros((1, S, Hkv, D), np.int8)
    kc[0, 1, :, :] = np.array([1, 2, 0, -1], np.int8)
    vc[0, 0, :, :] = np.array([4, 0, -2, 1], np.int8)
    vc[0, 1, :, :] = np.array([-3, 5, 1, 0], np.int8)
    q = np.tile(np.array([1.0, 0.5, 2.0, -1.0], np.float32), (1, Hkv * G, 1))
    scale = 0.7
    out = oracle.paged_attention_decode(q, kc, vc, np.zeros((1, 1), np.int32), np.array([2], np.int32), scale,
                                        cache_dtype=oracle.I8, k_head_scales=ks, v_head_scales=vs)
    qc = float(np.dot(q[0, 0].astype(np.float64), kc[0, 1, 0].astype(np.float64)))
    for h in range(Hkv):
        z = scale * qc * ks[h]
        w1 = math.exp(z) / (1 + math.exp(z))
        want = vs[h] * ((1 - w1) * vc[0, 0, h].astype(np.float64) + w1 * vc[0, 1, h].astype(np.float64))
        for g in range(G):
            np.testing.assert_allclose(out[0, h * G + g], want, rtol=1e-13, atol=1e-13)
    # equal per-head scales reproduce the per-tensor path exactly (decode and prefill)
    same = oracle.paged_attention_decode(q, kc, vc, np.zeros((1, 1), np.int32), np.array([2], np.int32), scale,
                                         cache_dtype=oracle.I8, k_scale=0.25, v_scale=0.5,
                                         k_head_scales=np.full(Hkv, 0.25), v_head_scales=np.full(Hkv, 0.5))
    tensor = oracle.paged_attention_decode(q, kc, vc, np.zeros((1, 1), np.int32), np.array([2], np.int32), scale,
                                           cache_dtype=oracle.I8, k_scale=0.25, v_scale=0.5)
    np.testing.assert_array_equal(same, tensor)
    pf = oracle.paged_prefill_chunk(q, 1, kc, vc, np.zeros(1, np.int32), 2, scale, cache_dtype=oracle.I8,
                                    k_head_scales=ks, v_head_scales=vs)
    np.testing.assert_allclose(pf, out, rtol=1e-13, atol=1e-13)  # the last position sees both tokens
