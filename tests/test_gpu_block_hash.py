"""GPU block content hashes: bit-exact against the oracle's FNV-1a chain."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import _binding as B
from paged_kv_cache_71_gb300.runner import to_device

pytestmark = pytest.mark.gpu


def _case(lens, S, seed):
    rng = np.random.default_rng(seed)
    toks = rng.integers(-2**31, 2**31 - 1, int(sum(lens)), dtype=np.int64).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    nfull = np.array(lens) // S
    offs = np.concatenate([[0], np.cumsum(nfull)[:-1]]).astype(np.int64)
    return toks, cu, offs, int(nfull.sum())


@pytest.mark.parametrize("S", [4, 16, 32])
def test_block_hashes_match_oracle(S):
    lens = [0, 1, S - 1, S, S + 1, 33 * S, 100 * S + 7, 5000, 17]
    toks, cu, offs, n = _case(lens, S, seed=S)
    ref = oracle.block_hashes(toks, cu, S)
    out = torch.zeros(n, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_block_hashes(to_device(toks), to_device(cu), S, to_device(offs), out, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint64), ref)


def test_block_hashes_shared_prefix_and_capacity_check():
    S = 16
    rng = np.random.default_rng(1)
    prefix = rng.integers(0, 50000, 800).astype(np.int32)
    a = np.concatenate([prefix, rng.integers(0, 50000, 205).astype(np.int32)])
    b = np.concatenate([prefix, rng.integers(0, 50000, 205).astype(np.int32)])
    toks = np.concatenate([a, b])
    cu = np.array([0, 1005, 2010], np.int64)
    offs = np.array([0, 62], np.int64)
    out = torch.zeros(124, dtype=torch.int64, device="cuda")
    pkv.pkv_block_hashes(to_device(toks), to_device(cu), S, to_device(offs), out)
    h = out.cpu().numpy().view(np.uint64)
    assert (h[:50] == h[62:112]).all() and (h[50:62] != h[112:124]).all()  # 800 = 50 shared full blocks
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    small = torch.zeros(100, dtype=torch.int64, device="cuda")
    pkv.pkv_block_hashes(to_device(toks), to_device(cu), S, to_device(offs), small, err)
    torch.cuda.synchronize()
    assert err.item() & B.DEVERR_BAD_SLOT
