"""GPU parity of the cache write and block copy kernels: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import _binding as B
from paged_kv_cache_71_gb300 import workload as wl
from paged_kv_cache_71_gb300.runner import to_device

from parity import host_bits

pytestmark = pytest.mark.gpu

_CODE = {"f32": oracle.F32, "bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}


def _cache_pair(rng, NB, S, Hkv, D, dt):
    return wl.random_values(rng, (NB, S, Hkv, D), dt), wl.random_values(rng, (NB, S, Hkv, D), dt)


@pytest.mark.parametrize("src", ["f32", "bf16"])
@pytest.mark.parametrize("dst", ["f32", "bf16", "e4m3", "i8"])
@pytest.mark.parametrize("S,Hkv,D", [(4, 2, 64), (16, 8, 128), (32, 1, 64)])
def test_reshape_and_cache_bit_exact(src, dst, S, Hkv, D):
    rng = np.random.default_rng(100 + S + D)
    NB, T = 40, 37
    kc, vc = _cache_pair(rng, NB, S, Hkv, D, dst)
    kn = wl.random_values(rng, (T, Hkv, D), src)
    vn = wl.random_values(rng, (T, Hkv, D), src)
    if src == "f32":  # include large values to exercise FP8 saturation and bf16 rounding ties
        kn *= np.float32(60.0)
    slots = rng.choice(NB * S, size=T, replace=False).astype(np.int64)
    slots[3] = -1          # padding token
    slots[7] = -5
    ks, vs = {"e4m3": (0.37, 1.9), "i8": (0.05, 0.013)}.get(dst, (1.0, 1.0))
    ref_k, ref_v = kc.copy(), vc.copy()
    oracle.reshape_and_cache(kn, vn, slots, ref_k, ref_v, cache_dtype=_CODE[dst], k_scale=ks, v_scale=vs)
    dk, dv = to_device(kc), to_device(vc)
    desc = B.CacheDesc.for_cache(dk, ks, vs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_reshape_and_cache(to_device(kn), to_device(vn), to_device(slots), dk, dv, desc, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    np.testing.assert_array_equal(host_bits(dk), ref_k)
    np.testing.assert_array_equal(host_bits(dv), ref_v)


def test_reshape_and_cache_flags_slot_beyond_pool():
    rng = np.random.default_rng(5)
    NB, S, Hkv, D = 8, 4, 2, 64
    kc, vc = _cache_pair(rng, NB, S, Hkv, D, "f32")
    kn = wl.random_values(rng, (3, Hkv, D), "f32")
    slots = np.array([2, NB * S, 5], np.int64)
    ref_k, ref_v = kc.copy(), vc.copy()
    assert oracle.reshape_and_cache(kn, kn, slots, ref_k, ref_v) == 2
    dk, dv = to_device(kc), to_device(vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_reshape_and_cache(to_device(kn), to_device(kn), to_device(slots), dk, dv, B.CacheDesc.for_cache(dk), err)
    torch.cuda.synchronize()
    assert err.item() & B.DEVERR_BAD_SLOT
    np.testing.assert_array_equal(host_bits(dk), ref_k)


@pytest.mark.parametrize("dt", ["f32", "bf16", "e4m3", "i8"])
def test_copy_blocks_bit_exact(dt):
    rng = np.random.default_rng(9)
    NB, S, Hkv, D = 64, 16, 8, 128
    kc, vc = _cache_pair(rng, NB, S, Hkv, D, dt)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:20], perm[20:40]], axis=1).astype(np.int64)  # disjoint src / dst sets
    ref_k, ref_v = kc.copy(), vc.copy()
    oracle.copy_blocks(ref_k, ref_v, pairs)
    dk, dv = to_device(kc), to_device(vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_copy_blocks(dk, dv, B.CacheDesc.for_cache(dk, 0.5, 0.5), to_device(pairs), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    np.testing.assert_array_equal(host_bits(dk), ref_k)
    np.testing.assert_array_equal(host_bits(dv), ref_v)


def test_copy_blocks_flags_bad_ids_and_copies_the_rest():
    rng = np.random.default_rng(10)
    NB, S, Hkv, D = 16, 8, 2, 64
    kc, vc = _cache_pair(rng, NB, S, Hkv, D, "bf16")
    pairs = np.array([[1, 2], [3, NB], [-1, 4], [5, 6]], np.int64)
    ref_k, ref_v = kc.copy(), vc.copy()
    assert oracle.copy_blocks(ref_k, ref_v, pairs) == 3
    dk, dv = to_device(kc), to_device(vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_copy_blocks(dk, dv, B.CacheDesc.for_cache(dk), to_device(pairs), err)
    torch.cuda.synchronize()
    assert err.item() & B.DEVERR_BAD_BLOCK
    np.testing.assert_array_equal(host_bits(dk), ref_k)
    np.testing.assert_array_equal(host_bits(dv), ref_v)


def test_prefix_shared_cow_step():
    """The prefix-sharing batch's copy-on-write: 128 copies of the parent's partial block, then each
    child's token lands at offset 5 of its own copy; the parent's block is untouched."""
    w = wl.prefix_shared()
    ref_k, ref_v = w.k_cache.copy(), w.v_cache.copy()
    oracle.copy_blocks(ref_k, ref_v, w.copy_pairs)
    oracle.reshape_and_cache(w.k_new, w.v_new, w.slot_mapping, ref_k, ref_v)
    dk, dv = to_device(w.k_cache), to_device(w.v_cache)
    desc = B.CacheDesc.for_cache(dk)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_copy_blocks(dk, dv, desc, to_device(w.copy_pairs), err)
    pkv.pkv_reshape_and_cache(to_device(w.k_new), to_device(w.v_new), to_device(w.slot_mapping), dk, dv, desc, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    gk, gv = host_bits(dk), host_bits(dv)
    np.testing.assert_array_equal(gk, ref_k)
    np.testing.assert_array_equal(gv, ref_v)
    src = int(w.copy_pairs[0, 0])
    np.testing.assert_array_equal(gk[src], w.k_cache[src])           # source untouched
    for c, dst in enumerate(w.copy_pairs[:, 1]):
        np.testing.assert_array_equal(gk[dst, :5], w.k_cache[src, :5])  # inherited tokens
        np.testing.assert_array_equal(gk[dst, 5], w.k_new[128 + c])     # the child's own token
