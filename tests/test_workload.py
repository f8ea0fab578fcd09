"""Host-side workload construction: shapes, seeds, slot mapping and sharing structure."""
import numpy as np

import oracle
from paged_kv_cache_71_gb300 import workload as wl


def _check_slots(w):
    """Every new token's slot is the (block, offset) of position L-1 of its sequence."""
    S = w.block_size
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        blk, off = oracle.lookup(w.block_tables[s], L - 1, S)
        assert w.slot_mapping[s] == blk * S + off


def test_tiny_shape_and_positions():
    w = wl.tiny()
    assert list(w.context_lens) == [10, 6, 33, 1]
    assert w.k_cache.shape == (32, 4, 2, 64) and w.k_cache.dtype == np.float32
    assert w.q.shape == (4, 4, 64)
    _check_slots(w)
    used = w.block_tables[w.block_tables >= 0]
    assert len(used) == 3 + 2 + 9 + 1 and len(set(used.tolist())) == len(used)
    # new tokens at positions {9, 5, 32, 0}: offsets 1, 1, 0, 0 in S=4 blocks
    assert list(w.slot_mapping % 4) == [1, 1, 0, 0]


def test_seeded_reproducible():
    a, b = wl.tiny(), wl.tiny()
    assert (a.k_cache == b.k_cache).all() and (a.block_tables == b.block_tables).all()
    c = wl.tiny(seed=1)
    assert not (a.k_cache == c.k_cache).all()


def test_llama3_lengths_distribution():
    rng = np.random.default_rng(wl.CONFIG_SEEDS["llama3_8b_gqa"])
    L = wl.lognormal_lengths(rng, 256)
    assert L.min() >= 16 and L.max() <= 8192
    assert 700 < np.median(L) < 1500


def test_prefix_shared_structure():
    w = wl.prefix_shared()
    assert w.num_seqs == 128 and (w.context_lens == 1005).all()
    shared = w.notes["shared_blocks"]
    assert len(shared) == 50 and w.notes["shared_refcount"] == 128
    assert (w.block_tables[:, :50] == np.array(shared)[None, :]).all()
    private = w.block_tables[:, 50:63]
    assert len(set(private.ravel().tolist())) == 128 * 13
    _check_slots(w)
    # copy-on-write: 128 copies of the parent's partial block 50 into fresh blocks
    parent = w.notes["cow_parent_table"]
    assert w.copy_pairs.shape == (128, 2) and (w.copy_pairs[:, 0] == parent[50]).all()
    assert len(set(w.copy_pairs[:, 1].tolist())) == 128
    for c, tbl in enumerate(w.notes["cow_child_tables"]):
        assert tbl[:50] == parent[:50] and tbl[50] == w.copy_pairs[c, 1]
        assert w.slot_mapping[128 + c] == tbl[50] * 16 + 5   # the child's token at offset 5


def test_fp8_codes_have_no_nan():
    rng = np.random.default_rng(0)
    v = wl.random_values(rng, (1000,), "e4m3")
    assert not np.isnan(oracle.e4m3_to_f64(v)).any()


def test_block_manager_cow_on_empty_pool_changes_nothing():
    """A copy-on-write that finds no free block raises before touching the tables or the counts."""
    from paged_kv_cache_71_gb300.block_manager import SequenceTables
    import pytest
    t = SequenceTables(2, 4)
    t.prefill("p", 6)                 # blocks 1, 0: the pool is now empty
    t.fork("p", "c")
    before = (list(t.table("c")), t.pool.refcount.tolist(), t.length("c"))
    with pytest.raises(MemoryError):
        t.next_slot("c")              # block 0 is shared and partly filled: needs a copy
    assert (list(t.table("c")), t.pool.refcount.tolist(), t.length("c")) == before
    assert t.drain_copies() == []


def test_block_manager_released_blocks_come_back_first():
    from paged_kv_cache_71_gb300.block_manager import SequenceTables
    t = SequenceTables(6, 4)
    t.prefill("a", 8)                 # blocks 5, 4
    t.prefill("b", 4)                 # block 3
    t.drop("a")                       # 5 then 4 go back on the stack: 4 is on top
    t.prefill("c", 12)
    assert t.table("c") == [4, 5, 2]
    assert t.pool.num_free == 6 - 4
