"""GPU parity of per-KV-head scales for one-byte caches (INT8 and FP8 E4M3): the cache write is bit-exact against
the oracle, decode and the prefill tile agree within the tolerance of their dtype, and per-head scales that all
equal the per-tensor scale give the per-tensor results bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import _binding as B
from paged_kv_cache_71_gb300 import workload as wl
from paged_kv_cache_71_gb300.block_manager import SequenceTables
from paged_kv_cache_71_gb300.runner import to_device

from parity import assert_close, host_bits, to_host

pytestmark = pytest.mark.gpu

_CODE = {"e4m3": oracle.E4M3, "i8": oracle.I8}
_HEAD_SCALES = {
    "i8": (np.array([0.02, 0.05, 0.011, 0.08, 0.03, 0.016, 0.04, 0.06], np.float32),
           np.array([0.015, 0.07, 0.02, 0.01, 0.05, 0.03, 0.025, 0.09], np.float32)),
    "e4m3": (np.array([0.1, 0.4, 0.025, 1.5, 0.7, 0.05, 0.2, 0.9], np.float32),
             np.array([0.3, 0.06, 1.1, 0.15, 0.45, 0.08, 0.6, 0.02], np.float32)),
}


def _problem(rng, kv, lens, Hq=32, Hkv=8, D=128, S=16):
    """A paged pool written through the cache write with per-head scales (oracle image and device copy)."""
    need = sum(-(-L // S) for L in lens)
    NB = need + 5
    alloc = SequenceTables(NB, S, free_order=rng.permutation(NB))
    slots = []
    for s, L in enumerate(lens):
        alloc.prefill(s, L)
        slots += [alloc.slot(s, p) for p in range(L)]
    slots = np.array(slots, np.int64)
    T = slots.shape[0]
    ks, vs = _HEAD_SCALES[kv]
    # per-head magnitudes roughly matched to the scales, so that codes use their range
    kn = (wl.random_values(rng, (T, Hkv, D), "f32") * (ks * (40 if kv == "i8" else 8))[None, :, None]).astype(np.float32)
    vn = (wl.random_values(rng, (T, Hkv, D), "f32") * (vs * (40 if kv == "i8" else 8))[None, :, None]).astype(np.float32)
    kc = np.zeros((NB, S, Hkv, D), np.int8 if kv == "i8" else np.uint8)
    vc = np.zeros_like(kc)
    oracle.reshape_and_cache(kn, vn, slots, kc, vc, cache_dtype=_CODE[kv], k_scale=1.0, v_scale=1.0,
                             k_head_scales=ks, v_head_scales=vs)
    q = wl.random_values(rng, (len(lens), Hq, D), "bf16")
    return q, kn, vn, slots, kc, vc, alloc.block_tables(list(range(len(lens)))), np.array(lens, np.int32)


@pytest.mark.parametrize("kv", ["i8", "e4m3"])
def test_head_scales_cache_write_bit_exact(kv):
    rng = np.random.default_rng(41)
    q, kn, vn, slots, ref_k, ref_v, bt, cl = _problem(rng, kv, [37, 5, 80])
    ks, vs = _HEAD_SCALES[kv]
    dk, dv = to_device(np.zeros_like(ref_k)), to_device(np.zeros_like(ref_v))
    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    desc = B.CacheDesc.for_cache(dk, 1.0, 1.0, dks, dvs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_reshape_and_cache(to_device(kn), to_device(vn), to_device(slots), dk, dv, desc, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    np.testing.assert_array_equal(host_bits(dk), ref_k)
    np.testing.assert_array_equal(host_bits(dv), ref_v)


@pytest.mark.parametrize("kv", ["i8", "e4m3"])
@pytest.mark.parametrize("splits", [1, 0])
def test_head_scales_decode(kv, splits):
    rng = np.random.default_rng(43 + splits)
    q, kn, vn, slots, kc, vc, bt, cl = _problem(rng, kv, [300, 17, 1000, 64])
    ks, vs = _HEAD_SCALES[kv]
    ref = oracle.paged_attention_decode(q, kc, vc, bt, cl, 1 / np.sqrt(128), cache_dtype=_CODE[kv],
                                        k_head_scales=ks, v_head_scales=vs)
    dk, dv = to_device(kc), to_device(vc)
    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    desc = B.CacheDesc.for_cache(dk, 1.0, 1.0, dks, dvs)
    dq = to_device(q)
    out = torch.full_like(dq, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_bytes = pkv.pkv_paged_attention_workspace_size(desc, q.shape[0], q.shape[1], splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
    pkv.pkv_paged_attention_decode(out, dq, dk, dv, desc, to_device(bt), to_device(cl), 1 / np.sqrt(128),
                                   num_splits=splits, workspace=ws, device_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert_close(kv, to_host(out), ref, f"decode with per-head {kv} scales, splits={splits}")


@pytest.mark.parametrize("kv", ["i8", "e4m3"])
def test_head_scales_prefill_chunk_and_varlen(kv):
    rng = np.random.default_rng(47)
    q, kn, vn, slots, kc, vc, bt, cl = _problem(rng, kv, [300])
    ks, vs = _HEAD_SCALES[kv]
    q_start, NQ = 200, 100
    qc = wl.random_values(rng, (NQ, 32, 128), "bf16")
    scale = 1 / np.sqrt(128)
    ref = oracle.paged_prefill_chunk(qc, q_start, kc, vc, bt[0], 300, scale, cache_dtype=_CODE[kv],
                                     k_head_scales=ks, v_head_scales=vs)
    dk, dv = to_device(kc), to_device(vc)
    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    desc = B.CacheDesc.for_cache(dk, 1.0, 1.0, dks, dvs)
    dq = to_device(qc)
    out = torch.full_like(dq, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.pkv_paged_prefill_chunk(out, dq, q_start, dk, dv, desc, to_device(bt[0]), 300, scale, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert_close(kv, to_host(out), ref, f"prefill chunk with per-head {kv} scales")
    # the same chunk through the varlen entry point
    out2 = torch.full_like(dq, float("nan"))
    pkv.pkv_paged_prefill_varlen(out2, dq, to_device(np.array([0, NQ], np.int32)),
                                 to_device(np.array([q_start], np.int32)), to_device(np.array([300], np.int32)),
                                 dk, dv, desc, to_device(bt[:1]), scale, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_equal_head_scales_reproduce_per_tensor_bits():
    rng = np.random.default_rng(53)
    q, kn, vn, slots, kc, vc, bt, cl = _problem(rng, "i8", [120, 33])
    dk, dv = to_device(kc), to_device(vc)
    dq = to_device(q)
    per_tensor = B.CacheDesc.for_cache(dk, 0.03, 0.02)
    hs_k = torch.full((8,), 0.03, dtype=torch.float32, device="cuda")
    hs_v = torch.full((8,), 0.02, dtype=torch.float32, device="cuda")
    per_head = B.CacheDesc.for_cache(dk, 0.5, 0.5, hs_k, hs_v)  # the per-tensor fields are ignored
    outs = []
    for desc in (per_tensor, per_head):
        out = torch.empty_like(dq)
        pkv.pkv_paged_attention_decode(out, dq, dk, dv, desc, to_device(bt), to_device(cl), 0.088, num_splits=1)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
