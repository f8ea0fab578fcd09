"""The C ABI without a GPU: the library loads, exports what include/pkv.h declares,
and its host-side argument checks reject bad calls before touching a device."""
import ctypes

import pytest

import paged_kv_cache_71_gb300 as pkv
from paged_kv_cache_71_gb300 import _binding as B


def test_library_exports_every_declared_entry_point():
    names = pkv.declared_entry_points()
    assert {"pkv_reshape_and_cache", "pkv_paged_attention_decode", "pkv_copy_blocks",
            "pkv_paged_attention_workspace_size", "pkv_status_string"} <= set(names)
    L = pkv.lib()
    for n in names:
        assert hasattr(L, n), n


def test_binding_constants_match_the_header():
    """The device error bits and dtype codes the binding uses are the ones include/pkv.h defines."""
    import os
    import re
    text = open(os.path.join(os.path.dirname(__file__), "..", "include", "pkv.h")).read()
    defs = {m.group(1): int(m.group(2), 0) for m in re.finditer(r"#define (PKV_DEVERR_\w+) (0x[0-9a-fA-F]+|\d+)", text)}
    assert defs == {"PKV_DEVERR_BAD_SLOT": B.DEVERR_BAD_SLOT, "PKV_DEVERR_BAD_BLOCK": B.DEVERR_BAD_BLOCK,
                    "PKV_DEVERR_BAD_LENGTH": B.DEVERR_BAD_LENGTH, "PKV_DEVERR_TIMEOUT": B.DEVERR_TIMEOUT,
                    "PKV_DEVERR_Q_RANGE": B.DEVERR_Q_RANGE}
    enums = {m.group(1): int(m.group(2)) for m in re.finditer(r"(PKV_(?:F32|BF16|FP8_E4M3|INT8))\s*=\s*(\d+)", text)}
    assert enums == {"PKV_F32": B.PKV_F32, "PKV_BF16": B.PKV_BF16, "PKV_FP8_E4M3": B.PKV_FP8_E4M3,
                     "PKV_INT8": B.PKV_INT8}


def test_status_strings_and_version():
    assert pkv.pkv_abi_version() == 2  # the cache descriptor carries optional per-head scales
    for code, name in B.STATUS_NAMES.items():
        assert pkv.pkv_status_string(code) == name
    assert pkv.pkv_status_string(99) == "PKV_ERR_UNKNOWN"


def _desc(**kw):
    d = dict(num_blocks=16, block_size=16, num_kv_heads=8, head_dim=128, dtype=B.PKV_BF16, k_scale=1.0, v_scale=1.0)
    d.update(kw)
    return B.CacheDesc(**d)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 2), (dict(block_size=12), 2), (dict(block_size=64), 2), (dict(num_blocks=0), 1),
    (dict(dtype=7), 1), (dict(dtype=B.PKV_FP8_E4M3, k_scale=0.0), 1), (dict(num_kv_heads=-1), 1),
    (dict(k_head_scales=4096), 1),                           # per-head scales on a bf16 cache
    (dict(dtype=B.PKV_INT8, v_head_scales=4098), 1),         # misaligned per-head scale array
])
def test_cache_descriptor_checks(kw, status):
    L = pkv.lib()
    out = ctypes.c_size_t(0)
    st = L.pkv_paged_attention_workspace_size(ctypes.byref(_desc(**kw)), 4, 32, 0, ctypes.byref(out))
    assert st == status, pkv.pkv_last_error()
    assert pkv.pkv_last_error()


def test_decode_host_checks_before_any_device_work():
    L = pkv.lib()
    d = _desc()
    args = lambda **o: dict(dict(out=16, q=16, q_dtype=B.PKV_BF16, k=16, v=16, bt=16, mb=4, cl=16, B=2, Hq=32,
                                 scale=0.1, splits=1, maxlen=0, ws=None, wsb=0), **o)

    def call(a):
        return L.pkv_paged_attention_decode(a["out"], a["q"], a["q_dtype"], a["k"], a["v"], ctypes.byref(d), a["bt"],
                                            a["mb"], a["cl"], a["B"], a["Hq"], a["scale"], a["splits"], a["maxlen"],
                                            a["ws"], a["wsb"], None, None)
    assert call(args(Hq=30)) == 1            # not a multiple of Hkv
    assert call(args(Hq=8 * 3)) == 2         # G = 3
    assert call(args(Hq=8 * 16)) == 2        # G = 16
    assert call(args(q_dtype=B.PKV_F32)) == 2  # f32 q with bf16 cache
    assert call(args(B=-1)) == 1
    assert call(args(mb=0)) == 1
    assert call(args(out=None)) == 1
    assert call(args(q=24)) == 1             # misaligned
    assert call(args(scale=float("nan"))) == 1
    assert call(args(B=9000)) == 2
    assert call(args(B=0)) == 0              # empty batch is a no-op
    # the shared-block form takes the same arguments and the same checks
    shared = lambda a: L.pkv_paged_attention_decode_shared(a["out"], a["q"], a["q_dtype"], a["k"], a["v"],
                                                           ctypes.byref(d), a["bt"], a["mb"], a["cl"], a["B"],
                                                           a["Hq"], a["scale"], a["splits"], a["maxlen"], a["ws"],
                                                           a["wsb"], None, None)
    assert shared(args(Hq=30)) == 1
    assert shared(args(Hq=8 * 3)) == 2
    assert shared(args(q=24)) == 1
    assert shared(args(B=0)) == 0


def test_reshape_and_copy_host_checks():
    L = pkv.lib()
    d = _desc()
    assert L.pkv_reshape_and_cache(16, 16, B.PKV_BF16, 16, -1, 16, 16, ctypes.byref(d), None, None) == 1
    assert L.pkv_reshape_and_cache(16, 16, B.PKV_BF16, 16, 0, 16, 16, ctypes.byref(d), None, None) == 0
    assert L.pkv_reshape_and_cache(16, 16, B.PKV_FP8_E4M3, 16, 4, 16, 16, ctypes.byref(d), None, None) == 2
    assert L.pkv_reshape_and_cache(16, 17, B.PKV_BF16, 16, 4, 16, 16, ctypes.byref(d), None, None) == 1
    assert L.pkv_reshape_and_cache(16, 16, B.PKV_BF16, 12, 4, 16, 16, ctypes.byref(d), None, None) == 1
    assert L.pkv_copy_blocks(16, 16, ctypes.byref(d), 16, -2, None, None) == 1
    assert L.pkv_copy_blocks(16, 16, ctypes.byref(d), 16, 0, None, None) == 0
    assert L.pkv_copy_blocks(16, 16, ctypes.byref(d), 12, 3, None, None) == 1
    assert L.pkv_copy_blocks(None, 16, ctypes.byref(d), 16, 3, None, None) == 1
    # one CTA per (pair, tensor): 2^30 pairs would overflow the grid
    assert L.pkv_copy_blocks(16, 16, ctypes.byref(d), 16, 1 << 30, None, None) == 3
    assert L.pkv_swap_blocks(16, 16, 4, 16, 16, 4, ctypes.byref(d), 16, 1 << 30, None, None) == 3


def test_product_path_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No CPU fallback: with libpkv.so absent every call raises instead of computing anything."""
    import torch
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libpkv.so"))
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()
    desc = B.CacheDesc(num_blocks=4, block_size=16, num_kv_heads=2, head_dim=128, dtype=B.PKV_BF16,
                       k_scale=1.0, v_scale=1.0)
    with pytest.raises(RuntimeError, match="not built"):
        pkv.pkv_paged_attention_workspace_size(desc, 2, 4, 0)
    q = torch.zeros(2, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(RuntimeError, match="not built"):
        pkv.pkv_paged_attention_decode(q.clone(), q, torch.zeros(4, 16, 2, 128, dtype=torch.bfloat16),
                                       torch.zeros(4, 16, 2, 128, dtype=torch.bfloat16), desc,
                                       torch.zeros(2, 1, dtype=torch.int32), torch.ones(2, dtype=torch.int32), 0.1)


def test_mixed_step_host_checks_before_any_device_work():
    """pkv_paged_attention_mixed rejects bad steps on the host, before it asks for the device."""
    L = pkv.lib()

    def call(desc=None, **o):
        a = dict(out=16, q=16, q_dtype=B.PKV_BF16, total=40, cu=16, qs=16, kl=16, k=16, v=16, bt=16, mb=4, n=3,
                 nd=2, Hq=64, scale=0.1, ws=16, wsb=1 << 20)
        a.update(o)
        d = desc or _desc()
        return L.pkv_paged_attention_mixed(a["out"], a["q"], a["q_dtype"], a["total"], a["cu"], a["qs"], a["kl"],
                                           a["k"], a["v"], ctypes.byref(d), a["bt"], a["mb"], a["n"], a["nd"],
                                           a["Hq"], a["scale"], a["ws"], a["wsb"], None, None)
    assert call(nd=4) == 1                           # more decode tokens than chunks
    assert call(nd=-1) == 1
    assert call(total=1) == 1                        # fewer query tokens than decode tokens
    assert call(Hq=60) == 1                          # not a multiple of the KV heads
    assert call(Hq=8 * 16) == 2                      # G = 16
    assert call(Hq=8 * 3) == 2                       # G = 3
    assert call(q_dtype=B.PKV_F32) == 2
    assert call(desc=_desc(block_size=8)) == 2       # block_size 16 only
    assert call(desc=_desc(head_dim=64)) == 2        # head_dim 128 only
    assert call(desc=_desc(dtype=B.PKV_F32)) == 2    # bf16, FP8 or INT8 caches
    assert call(n=4096, nd=2) == 2                   # more chunks than one launch takes
    assert call(n=0, nd=0) == 0                      # an empty step is a no-op
    assert call(total=0, nd=0) == 0
    out = ctypes.c_size_t(1)
    assert L.pkv_paged_attention_mixed_workspace_size(ctypes.byref(_desc()), -1, 64, ctypes.byref(out)) == 1
    assert L.pkv_paged_attention_mixed_workspace_size(ctypes.byref(_desc()), 4, 60, ctypes.byref(out)) == 1
