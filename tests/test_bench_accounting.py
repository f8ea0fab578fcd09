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
    for FP8 / INT8 caches with 128-dim heads, for bf16 caches of 128-dim heads in GQA groups of 8, and for the
    prefix-sharing batch (shared-block form), the CUDA-core form otherwise; only the CUDA-core form is ever reported
    against the fp32 FMA ceiling."""
    import bench
    from paged_kv_cache_71_gb300 import workload as wl
    expect = {"tiny": "paged_decode_kernel", "llama2_7b": "paged_decode_kernel",
              "llama3_8b_gqa": "paged_decode_kernel", "prefix_shared": "paged_decode_mma_kernel",
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


def test_unique_bytes_count_shared_blocks_once():
    """Prefix-sharing batch: 128 sequences of 1005 tokens whose first 800 (50 blocks) are one shared copy."""
    w = wl.prefix_shared()
    per_tok = 2 * 8 * 128 * 2                       # K and V, 8 kv heads, d = 128, bf16
    qo = 2 * 128 * 32 * 128 * 2
    table = 128 * 63 * 4 + 4 * 128
    assert bench.decode_algorithmic_bytes(w) == 128 * 1005 * per_tok + qo + table
    assert bench.decode_unique_bytes(w) == (800 + 128 * 205) * per_tok + qo + table
    # no sharing: the two counts agree
    t = wl.tiny()
    assert bench.decode_unique_bytes(t) == bench.decode_algorithmic_bytes(t)


def test_contiguous_layout_holds_the_same_tokens_in_order():
    """Identity tables over a permuted copy of the pool read every sequence's tokens exactly as the scattered
    tables do; each sequence's blocks are consecutive."""
    import oracle
    w = wl.tiny()
    perm, tables = bench.contiguous_layout(w)
    kc = w.k_cache[perm]
    S = w.block_size
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        nb = -(-L // S)
        row = tables[s, :nb]
        assert (np.diff(row) == 1).all() and (tables[s, nb:] == -1).all()
        for p in range(L):
            b0, o0 = oracle.lookup(w.block_tables[s], p, S)
            b1, o1 = oracle.lookup(tables[s], p, S)
            assert o0 == o1 and (kc[b1, o1] == w.k_cache[b0, o0]).all()


def test_l2_plan_and_reference_config():
    """Batches whose unique K/V fits twice in L2 are timed with an L2 flush between steps; the reference arm prints
    the same `config` as the GPU arm for the same workload, whichever of GB300's quoted L2 sizes the device gives."""
    for name, plan in (("tiny", "flush"), ("prefix_shared", "flush"), ("llama3_8b_gqa", "large")):
        w = wl.make(name)
        for l2 in (bench.REFERENCE_L2_BYTES, 129 * 10**6, 132 * 2**20):
            assert bench.l2_plan(w, l2) == plan, (name, l2)
    w = wl.tiny()
    cfg = bench.line_config(w, 0, 1, bench.l2_note(w, bench.l2_plan(w, bench.REFERENCE_L2_BYTES)))
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference", "--config",
                        "tiny", "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"] == cfg
