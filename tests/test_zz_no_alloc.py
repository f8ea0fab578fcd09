"""The decode entry point that allocates nothing.

pkv_paged_attention_decode_static_scratch serves callers that cannot
allocate device memory when they run attention (a fixed memory plan, a
host that owns every allocation, a plain-C runtime without an allocator):
it keeps the split-KV scratch in a static device array owned by the
library.  These tests call it through the C ABI and check it on two calls
in a row against the workspace-taking entry point and against the fp64
oracle, within the same tolerances as the other parity tests.  This file is
collected last.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import _binding as B
from paged_kv_cache_71_gb300 import workload as wl
from paged_kv_cache_71_gb300.block_manager import SequenceTables
from paged_kv_cache_71_gb300.runner import DeviceStep

from parity import TOL, assert_close, oracle_step, to_host

pytestmark = pytest.mark.gpu


def _random(lens, Hq, Hkv, D, S, kv, q, seed):
    rng = np.random.default_rng(seed)
    need = int(sum(-(-L // S) for L in lens))
    NB = need + 3
    alloc = SequenceTables(NB, S, free_order=rng.permutation(NB))
    slots = []
    for s, L in enumerate(lens):
        alloc.prefill(s, L - 1)
        slots.append(alloc.next_slot(s))
    sc = {"e4m3": wl.FP8_SCALE, "i8": wl.INT8_SCALE}.get(kv, 1.0)
    return wl.Workload("random", seed, Hq, Hkv, D, S, kv, q, sc, sc,
                       wl.random_values(rng, (len(lens), Hq, D), q),
                       wl.random_values(rng, (NB, S, Hkv, D), kv), wl.random_values(rng, (NB, S, Hkv, D), kv),
                       alloc.block_tables(list(range(len(lens)))), np.array(lens, np.int32),
                       wl.random_values(rng, (len(lens), Hkv, D), q), wl.random_values(rng, (len(lens), Hkv, D), q),
                       np.array(slots, np.int64), np.zeros((0, 2), np.int64))


CASES = [
    ("tiny", lambda: wl.tiny()),
    ("bf16_gqa4", lambda: _random([1, 17, 300, 2048, 999, 64], 32, 8, 128, 16, "bf16", "bf16", 5)),
    ("fp8_gqa8", lambda: _random([4096, 12, 777], 64, 8, 128, 16, "e4m3", "bf16", 6)),
    # tensor-core form with two KV heads per work unit: split-KV records over 8 query heads
    ("int8_gqa4_pairs", lambda: _random([3000, 5, 640, 17, 1500], 32, 8, 128, 16, "i8", "bf16", 7)),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("num_splits", [0, 3])
def test_static_scratch_matches_workspace_entry_point(name, make, num_splits):
    w = make()
    st = DeviceStep(w, num_splits=num_splits)
    st.write()
    st.attend()
    torch.cuda.synchronize()
    assert st.device_error() == 0
    ref = st.out.double().cpu().numpy()
    atol, rtol = TOL[w.kv_dtype]
    _, _, oref = oracle_step(w)
    for call in range(2):
        out = torch.full_like(st.out, float("nan"))
        pkv.pkv_paged_attention_decode_static_scratch(out, st.q, st.k_cache, st.v_cache, st.cache, st.block_tables,
                                                      st.context_lens, w.scale, num_splits, st.max_context_len,
                                                      st.err)
        torch.cuda.synchronize()
        assert st.device_error() == 0
        got = out.double().cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}"
        assert (np.abs(got - ref) <= atol + rtol * np.abs(ref)).all(), f"call {call}: max diff {np.abs(got - ref).max()}"
        # and independently of the other CUDA entry point: against the oracle
        assert_close(w.kv_dtype, to_host(out), oref, f"{name} splits={num_splits} call {call} vs oracle")


def test_static_scratch_rejects_batches_beyond_its_size():
    # 8192 sequences x 128 KV heads of completion counters alone exceed the array
    desc = B.CacheDesc(num_blocks=64, block_size=16, num_kv_heads=128, head_dim=128, dtype=B.PKV_BF16,
                       k_scale=1.0, v_scale=1.0)
    need = pkv.pkv_paged_attention_workspace_size(desc, 8192, 1024, 0)
    assert need > B.STATIC_SCRATCH_BYTES
    out = torch.zeros(16, dtype=torch.uint8, device="cuda")
    L = pkv.lib()
    p = out.data_ptr()
    st = L.pkv_paged_attention_decode_static_scratch(p, p, B.PKV_BF16, p, p, __import__("ctypes").byref(desc), p, 4,
                                                     p, 8192, 1024, 0.1, 0, 0, None, None)
    assert st == 4 and "PKV_STATIC_SCRATCH_BYTES" in pkv.pkv_last_error()
    torch.cuda.synchronize()
    assert (out == 0).all()
    # without splits no scratch is needed, so the same sizes pass the size check
    assert pkv.pkv_paged_attention_workspace_size(desc, 8192, 1024, 1) == 0
