"""The benchmark's byte and flop accounting, pinned to the pages' capacity arithmetic."""
import json
import math
import os

import numpy as np

import bench
from paged_kv_cache_71_gb300 import workload as wl


def test_kv_bytes_per_token_matches_capacity_example(golden_dir):
    with open(os.path.join(golden_dir, "capacity_worked_example.json")) as f:
        g = json.load(f)
    per_tok = bench.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["dtype_bytes"])
    assert per_tok == g["kv_bytes_per_token"] == 128 * 1024
    assert per_tok * g["block_size"] == g["block_bytes"]
    assert g["kv_pool_bytes"] // g["block_bytes"] == g["pool_blocks"]
    assert g["pool_blocks"] * g["block_size"] == g["pool_tokens"]
    req = g["request_blocks_at_end"]
    assert math.ceil(req["tokens"] / g["block_size"]) == req["blocks"] and req["blocks"] * 16 == req["slots"]
    assert round(g["pool_tokens"] / g["contiguous_reservation_tokens"]) == g["concurrency"]["contiguous"]
    assert round(g["pool_tokens"] / req["slots"]) == g["concurrency"]["paged"]


def test_decode_algorithmic_bytes_by_hand():
    w = wl.tiny()
    L = np.array([10, 6, 33, 1])
    kv = int(L.sum()) * 2 * 2 * 64 * 4            # K and V, 2 kv heads, d = 64, fp32
    qo = 2 * 4 * 4 * 64 * 4                       # q and out, 4 seqs x 4 heads x 64 x fp32
    table = int(np.ceil(L / 4).sum()) * 4         # block-table entries read
    assert bench.decode_algorithmic_bytes(w) == kv + qo + table + 4 * 4


def test_prefill_flops_closed_form():
    class PF:
        q = np.zeros((512, 64, 128))
        q_start = 8192

    class W:
        prefill = PF()
        head_dim = 128
        num_q_heads = 64
    # sum_{i<512} (8193 + i) = 512 * 8193 + 511 * 512 / 2
    keys = 512 * 8193 + 511 * 256
    assert bench.prefill_flops(W()) == 4 * 128 * 64 * keys == 141742309376


def test_decode_ceiling_switches_to_fma_where_arithmetic_binds():
    """2 * G flops per cached element: the Llama-3-8B batch (G = 4, bf16) needs far less fp32 FMA work than the CUDA
    cores give when its K/V streams at the HBM peak; the FP8 Llama-70B step (G = 8, one-byte codes) needs more."""
    import bench
    from paged_kv_cache_71_gb300 import workload as wl
    hbm = 6663.6e9
    for name, alu in (("llama3_8b_gqa", False), ("llama70b_mixed_fp8", True)):
        w = wl.make(name, batch=8)
        G = w.num_q_heads // w.num_kv_heads
        elems = int(w.context_lens.sum()) * w.num_kv_heads * w.head_dim * 2
        assert bench.decode_fma_flops(w) == 2 * G * elems
        need = bench.decode_fma_flops(w) / bench.decode_algorithmic_bytes(w) * hbm / 1e12
        assert (need > bench.FP32_FMA_TFLOPS) == alu
    assert abs(bench.FP32_FMA_TFLOPS - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9


def test_decode_kernel_attribution_follows_the_library_policy():
    """The benchmark names the decode kernel a workload runs on as the library dispatches it: the tensor-core form
    for FP8 / INT8 caches with 128-dim heads and for bf16 caches of 128-dim heads in GQA groups of 8, the CUDA-core
    form otherwise; only the CUDA-core form is ever reported against the fp32 FMA ceiling."""
    import bench
    from paged_kv_cache_71_gb300 import workload as wl
    expect = {"tiny": "paged_decode_kernel", "llama2_7b": "paged_decode_kernel",
              "llama3_8b_gqa": "paged_decode_kernel", "prefix_shared": "paged_decode_kernel",
              "llama3_8b_gqa_int8": "paged_decode_mma_kernel", "llama70b_mixed_bf16": "paged_decode_mma_kernel",
              "llama70b_mixed_fp8": "paged_decode_mma_kernel"}
    for name, kernel in expect.items():
        w = wl.make(name, batch=8) if name in ("llama3_8b_gqa", "llama70b_mixed_bf16", "llama70b_mixed_fp8") \
            else wl.make(name)
        got, sources = bench.decode_kernel(w)
        assert got == kernel, name
        for f in sources:  # every source the profile digest covers exists
            assert os.path.exists(os.path.join(bench.ROOT, "paged_kv_cache_71_gb300", "csrc", f)), (name, f)
    # the policy constants the attribution mirrors
    api = open(os.path.join(bench.ROOT, "paged_kv_cache_71_gb300", "csrc", "api.cu")).read()
    assert "#define PKV_BF16_MMA_MIN_G 8" in api
