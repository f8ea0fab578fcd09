"""GPU parity of swap_blocks (device pool <-> pinned host pool): bit-exact against the oracle."""
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


def _pinned(a: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.pin_memory()


@pytest.mark.parametrize("dt", ["bf16", "e4m3", "f32"])
def test_swap_out_and_in(dt):
    rng = np.random.default_rng(40)
    NB, NH, S, Hkv, D = 64, 24, 16, 8, 128
    dev_k, dev_v = wl.random_values(rng, (NB, S, Hkv, D), dt), wl.random_values(rng, (NB, S, Hkv, D), dt)
    host_k, host_v = wl.random_values(rng, (NH, S, Hkv, D), dt), wl.random_values(rng, (NH, S, Hkv, D), dt)
    out_pairs = np.stack([rng.choice(NB, 20, replace=False), rng.choice(NH, 20, replace=False)], 1).astype(np.int64)
    in_pairs = np.stack([out_pairs[:12, 1], rng.choice(NB, 12, replace=False)], 1).astype(np.int64)
    ref_hk, ref_hv = host_k.copy(), host_v.copy()
    oracle.swap_blocks(dev_k, dev_v, ref_hk, ref_hv, out_pairs)
    ref_dk, ref_dv = dev_k.copy(), dev_v.copy()
    oracle.swap_blocks(ref_hk, ref_hv, ref_dk, ref_dv, in_pairs)

    dk, dv = to_device(dev_k), to_device(dev_v)
    hk, hv = _pinned(host_k), _pinned(host_v)
    desc = B.CacheDesc.for_cache(dk, 0.5, 0.5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_swap_blocks(dk, dv, hk, hv, desc, to_device(out_pairs), err)        # swap out
    pkv.pkv_swap_blocks(hk, hv, dk, dv, desc, to_device(in_pairs), err)         # swap in
    torch.cuda.synchronize()
    assert err.item() == 0
    got_hk = hk.view(torch.int16).numpy().view(np.uint16) if dt == "bf16" else hk.numpy()
    np.testing.assert_array_equal(got_hk, ref_hk)
    np.testing.assert_array_equal(host_bits(dk), ref_dk)
    np.testing.assert_array_equal(host_bits(dv), ref_dv)


def test_swap_flags_bad_ids_and_rejects_unreachable_memory():
    rng = np.random.default_rng(41)
    dev = wl.random_values(rng, (8, 16, 2, 64), "bf16")
    dk, dv = to_device(dev), to_device(dev)
    hk, hv = _pinned(np.zeros((4, 16, 2, 64), np.uint16)), _pinned(np.zeros((4, 16, 2, 64), np.uint16))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = B.CacheDesc.for_cache(dk)
    pkv.pkv_swap_blocks(dk, dv, hk, hv, desc, to_device(np.array([[1, 4], [2, 0]], np.int64)), err)
    torch.cuda.synchronize()
    assert err.item() & B.DEVERR_BAD_BLOCK
    assert (hk[0].view(torch.int16).numpy().view(np.uint16) == dev[2]).all()
