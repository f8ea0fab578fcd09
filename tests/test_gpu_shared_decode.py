"""GPU parity of the shared-block decode form (pkv_paged_attention_decode_shared) against the fp64 oracle.

The form is for batches whose block tables name the same physical blocks (forks of one sequence, a common prompt
prefix).  It computes what pkv_paged_attention_decode computes; for bf16 caches of 128-dim heads it runs the
tensor-core kernel at every GQA group.  Tolerances are in parity.py.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import workload as wl
from paged_kv_cache_71_gb300.block_manager import SequenceTables
from paged_kv_cache_71_gb300.runner import DeviceStep

from parity import assert_close, oracle_step, to_host

pytestmark = pytest.mark.gpu


def _forked_workload(n_prefix, suffixes, Hq, Hkv, S, kv, seed):
    """Sequences forked from one parent of n_prefix tokens, each then extended by its own suffix (the last token
    being this step's): the parent's full blocks stay shared, a partial last block is copied on the first write."""
    rng = np.random.default_rng(seed)
    D = 128
    need = -(-n_prefix // S) + sum(-(-(n_prefix + x) // S) for x in suffixes) + 2
    NB = need + 5
    t = SequenceTables(NB, S, free_order=rng.permutation(NB))
    t.prefill("parent", n_prefix)
    for s in range(len(suffixes)):
        t.fork("parent", s)
    t.drop("parent")
    slots = []
    for s, x in enumerate(suffixes):
        for _ in range(x - 1):
            t.next_slot(s)
        slots.append(t.next_slot(s))
    pairs = np.array(t.drain_copies(), np.int64).reshape(-1, 2)
    B = len(suffixes)
    sc = {"e4m3": wl.FP8_SCALE, "i8": wl.INT8_SCALE}.get(kv, 1.0)
    shared = t.table(0)[: n_prefix // S]
    return wl.Workload("forked", seed, Hq, Hkv, D, S, kv, "bf16", sc, sc,
                       wl.random_values(rng, (B, Hq, D), "bf16"),
                       wl.random_values(rng, (NB, S, Hkv, D), kv), wl.random_values(rng, (NB, S, Hkv, D), kv),
                       t.block_tables(list(range(B))), np.array([t.length(s) for s in range(B)], np.int32),
                       wl.random_values(rng, (B, Hkv, D), "bf16"), wl.random_values(rng, (B, Hkv, D), "bf16"),
                       np.array(slots, np.int64), pairs, notes={"shared_blocks": list(map(int, shared))})


def _run(w, num_splits, shared):
    st = DeviceStep(w, num_splits=num_splits, shared=shared)
    st.step()
    torch.cuda.synchronize()
    assert st.device_error() == 0
    return st


def test_prefix_sharing_batch_every_sequence():
    """The prefix-sharing batch (128 sequences over the same 50 blocks, then 205 private tokens each): every
    sequence against the oracle, after the step's copy-on-write copies and cache writes."""
    w = wl.prefix_shared()
    kc, vc, ref = oracle_step(w)
    st = _run(w, 0, True)
    assert_close("bf16", to_host(st.out), ref, "prefix-sharing batch, shared-block form")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_bf16_forks_every_group(G, num_splits):
    """bf16 forks at GQA groups 1..8, 16-token blocks, a shared prefix ending mid-block (copy-on-write), ragged
    suffixes including single tokens and long ones that the work split cuts."""
    w = _forked_workload(333, [1, 2, 17, 64, 700, 1500, 5, 2100], 2 * G, 2, 16, "bf16", seed=40 + G)
    kc, vc, ref = oracle_step(w)
    st = _run(w, num_splits, True)
    assert_close("bf16", to_host(st.out), ref, f"bf16 forks G={G} splits={num_splits}")


@pytest.mark.parametrize("S", [8, 32])
def test_bf16_forks_block_sizes(S):
    w = _forked_workload(200, [3, 90, 800, 1], 8, 2, S, "bf16", seed=S)
    kc, vc, ref = oracle_step(w)
    st = _run(w, 0, True)
    assert_close("bf16", to_host(st.out), ref, f"bf16 forks S={S}")


@pytest.mark.parametrize("kv", ["e4m3", "i8"])
def test_one_byte_caches_match_the_regular_form(kv):
    """One-byte caches take the same kernel in both forms: identical bits, and the oracle agrees."""
    w = _forked_workload(500, [10, 300, 1200, 4], 8, 2, 16, kv, seed=77)
    a = _run(w, 0, True)
    b = _run(w, 0, False)
    assert torch.equal(a.out, b.out)
    kc, vc, ref = oracle_step(w)
    assert_close(kv, to_host(a.out), ref, f"{kv} forks")


def test_workspace_of_the_regular_size_is_enough():
    """pkv_paged_attention_workspace_size covers the shared-block form (its split records are never larger)."""
    w = _forked_workload(100, [50, 2000, 7], 16, 4, 16, "bf16", seed=5)
    st = DeviceStep(w, num_splits=0, shared=True)
    need = pkv.pkv_paged_attention_workspace_size(st.cache, w.num_seqs, w.num_q_heads, 0)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    st.write()
    pkv.pkv_paged_attention_decode_shared(st.out, st.q, st.k_cache, st.v_cache, st.cache, st.block_tables,
                                          st.context_lens, w.scale, 0, st.max_context_len, ws, st.err)
    torch.cuda.synchronize()
    assert st.device_error() == 0
    kc, vc, ref = oracle_step(w)
    assert_close("bf16", to_host(st.out), ref, "regular-size workspace")
