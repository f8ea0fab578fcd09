"""Benchmark of the paged decode step on GB300.

One step = the whole hot path for one batch: the cache write of the step's
new tokens (reshape_and_cache), copy-on-write block copies when the batch
has any, and paged decode attention over every sequence.  Default workload:
the Llama-3-8B GQA batch (256 sequences, 32 q / 8 kv heads, head_dim 128,
bf16 KV, 16-token blocks, lognormal lengths) -- one layer.

Prints ONE JSON line (rank 0).  `value` is sequence-steps per second per
layer over all ranks, with inputs resident in HBM; `e2e` repeats the
measurement through the C ABI with host buffers (the step's inputs copied
in and the output copied out inside the timed region); `roofline` rates the
decode kernel's algorithmic bytes per launch against the measured HBM copy
bandwidth; `cpu_baseline` times the fp64 oracle on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attn KV GB/s & % of GB300 HBM peak; seq-steps/sec per layer"
UNIT = "seq-steps/s"
FALLBACK_HBM_GBS = 6800.0
# GB300's L2 size, for the reference arm's `config` (it runs on the host and queries no device); the GPU arm reads
# the size from the device
REFERENCE_L2_BYTES = 126 * 2**20


# ---------------------------------------------------------------- byte accounting

def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """K and V bytes one token occupies: 2 x layers x kv heads x head_dim x element size."""
    return 2 * n_layers * n_kv_heads * head_dim * dtype_bytes


def decode_algorithmic_bytes(w) -> int:
    """Bytes one decode launch must touch at least: every sequence's K and V once per KV head,
    the queries, the outputs, the block-table entries it reads and the context lengths."""
    from paged_kv_cache_71_gb300.workload import elem_size
    L = w.context_lens.astype(np.int64)
    kv = int(L.sum()) * kv_bytes_per_token(1, w.num_kv_heads, w.head_dim, elem_size(w.kv_dtype))
    qo = 2 * w.num_seqs * w.num_q_heads * w.head_dim * elem_size(w.q_dtype)
    table = int(((L + w.block_size - 1) // w.block_size).sum()) * 4
    return kv + qo + table + 4 * w.num_seqs


def decode_unique_bytes(w) -> int:
    """decode_algorithmic_bytes with every physical block's K and V counted once, however many sequences' tables
    name it (a shared prefix is read by every sequence that holds it; these are the bytes that must come from
    DRAM at least once)."""
    from paged_kv_cache_71_gb300.workload import elem_size
    S = w.block_size
    L = w.context_lens.astype(np.int64)
    nb = (L + S - 1) // S
    seq = np.repeat(np.arange(w.num_seqs), nb)
    j = np.arange(int(nb.sum())) - np.repeat(np.cumsum(nb) - nb, nb)
    blocks = w.block_tables[seq, j].astype(np.int64)
    valid = np.minimum(S, L[seq] - j * S)
    most = np.zeros(max(int(blocks.max()) + 1 if blocks.size else 1, 1), dtype=np.int64)
    np.maximum.at(most, blocks, valid)
    kv = int(most.sum()) * kv_bytes_per_token(1, w.num_kv_heads, w.head_dim, elem_size(w.kv_dtype))
    qo = 2 * w.num_seqs * w.num_q_heads * w.head_dim * elem_size(w.q_dtype)
    return kv + qo + int(nb.sum()) * 4 + 4 * w.num_seqs


def contiguous_layout(w):
    """The same batch with every sequence's K/V in consecutive physical blocks in logical order (the contiguous
    KV cache that paging replaces): (permutation new block -> old block, int32 tables [B, MB])."""
    S = w.block_size
    L = w.context_lens.astype(np.int64)
    nb = (L + S - 1) // S
    first = np.cumsum(nb) - nb
    perm = np.concatenate([w.block_tables[s, : nb[s]] for s in range(w.num_seqs)]).astype(np.int64)
    tables = np.full((w.num_seqs, max(int(nb.max()), 1)), -1, dtype=np.int32)
    for s in range(w.num_seqs):
        tables[s, : nb[s]] = first[s] + np.arange(nb[s])
    return perm, tables


def l2_plan(w, l2_bytes: int) -> str:
    """How the timed steps keep L2 from serving K/V left by the previous step: a batch whose unique K/V bytes are
    at least twice the L2 size evicts itself; a smaller one gets the L2 flushed (a 2x-L2 buffer written) before
    every timed step, outside the events that time it."""
    return "large" if decode_unique_bytes(w) >= 2 * l2_bytes else "flush"


def line_config(w, num_splits: int, ws: int, l2: str) -> dict:
    """The `config` of a bench line, identical for both arms on the same workload."""
    return {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
            "kv_dtype": w.kv_dtype, "mean_context": float(w.context_lens.mean()), "num_splits": num_splits,
            "parallelism": f"replicas{ws}", "l2": l2}


def l2_note(w, plan: str) -> str:
    if plan == "large":
        return f"inputs larger than L2: {decode_algorithmic_bytes(w) / 1e9:.2f} GB of K/V read per step"
    return (f"L2 flushed before every timed step (2x L2 written outside the timed events): the step's "
            f"{decode_unique_bytes(w) / 1e6:.1f} MB of unique K/V would fit in L2")


def prefill_flops(w) -> int:
    """Multiply-add work of the causal chunk: query i sees q_start + i + 1 keys; QK^T and P.V each
    cost 2 * head_dim flops per (query head, key)."""
    pf = w.prefill
    nq = pf.q.shape[0]
    keys = sum(pf.q_start + i + 1 for i in range(nq))
    return 4 * w.head_dim * w.num_q_heads * keys


def write_bytes(w) -> int:
    from paged_kv_cache_71_gb300.workload import elem_size
    T = len(w.slot_mapping)
    row = w.num_kv_heads * w.head_dim
    return 2 * T * row * (elem_size(w.q_dtype) + elem_size(w.kv_dtype)) + 8 * T


# ---------------------------------------------------------------- environment helpers

def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback"


# fp32 FMA ceiling of the CUDA-core decode: 152 SMs x 128 fp32 lanes x 2 flops x the 2070 MHz maximum SM clock
# (GB300's unit counts and clock).  Decode does 2 * G FMAs per cached K/V element (G for q.k, G for p.v).
GB300_SMS, FP32_LANES_PER_SM, SM_MAX_HZ = 152, 128, 2.07e9
FP32_FMA_TFLOPS = GB300_SMS * FP32_LANES_PER_SM * 2 * SM_MAX_HZ / 1e12


def decode_fma_flops(w) -> int:
    """fp32 flops of the decode arithmetic: every cached K and V element of every (sequence, KV head) meets the
    G query heads of its group once (q.k for K, p.v for V): 2 * G flops per element."""
    G = w.num_q_heads // w.num_kv_heads
    elems = int(sum(int(L) for L in w.context_lens)) * w.num_kv_heads * w.head_dim * 2
    return 2 * G * elems


DECODE_SOURCES = ("decode.cuh", "pkv_device.cuh", "decode_bf16_s16.cu")


def decode_kernel(w) -> tuple[str, tuple]:
    """The decode kernel a workload runs on, and the sources its profile digest covers: FP8 / INT8 caches with
    128-dim heads, and bf16 caches of 128-dim heads in GQA groups of 8 (or any group when the batch shares blocks
    and takes the shared-block form), take the tensor-core form, everything else the CUDA-core form."""
    G = w.num_q_heads // w.num_kv_heads
    shared = bool(w.notes.get("shared_blocks"))
    if w.head_dim == 128 and (w.kv_dtype in ("e4m3", "i8") or (w.kv_dtype == "bf16" and (G >= 8 or shared))):
        tag = {"e4m3": "fp8", "i8": "i8", "bf16": "bf16"}[w.kv_dtype]
        return "paged_decode_mma_kernel", ("decode_mma.cuh", "decode.cuh", "pkv_device.cuh",
                                           f"decode_mma_{tag}_s{w.block_size}.cu")
    tag = {"f32": "f32", "bf16": "bf16", "e4m3": "fp8", "i8": "i8"}[w.kv_dtype]
    return "paged_decode_kernel", ("decode.cuh", "pkv_device.cuh", f"decode_{tag}_s{w.block_size}.cu")


def kernel_digest(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_71_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, sources=DECODE_SOURCES):
    """DRAM bytes per decode launch from the committed ncu summary of this workload, if that summary was
    taken on the kernel sources as they are now (same digest); otherwise None."""
    import re
    path = os.path.join(ROOT, "profiles", f"decode_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    dig = re.search(r"kernel_digest:\s*([0-9a-f]+)", text)
    tr = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    if not dig or not tr or dig.group(1) != kernel_digest(sources):
        return None
    return int(tr.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle timing

def time_oracle_one_core(w, max_seconds: float = 8.0, chunk: int = 8) -> dict:
    """fp64 oracle on ONE host core: the step's cache write, then the decode of successive groups of `chunk`
    sequences until the batch is done or `max_seconds` pass; seq-steps/s over the sequences done (the write's
    time counted in proportion)."""
    import oracle
    oracle.build()
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    cache_dt = {"f32": oracle.F32, "bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}[w.kv_dtype]
    t0 = time.perf_counter()
    oracle.reshape_and_cache(w.k_new, w.v_new, w.slot_mapping, kc, vc, cache_dtype=cache_dt,
                             k_scale=w.k_scale, v_scale=w.v_scale)
    t_write = time.perf_counter() - t0
    done, t1 = 0, time.perf_counter()
    while done < w.num_seqs and time.perf_counter() - t1 < max_seconds:
        sel = np.arange(done, min(done + chunk, w.num_seqs))
        oracle.paged_attention_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, cache_dtype=cache_dt,
                                      k_scale=w.k_scale, v_scale=w.v_scale, seqs=sel, threads=1)
        done += len(sel)
    t_dec = time.perf_counter() - t1
    dt = t_dec + t_write * done / w.num_seqs
    return {"value": round(done / dt, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"cache write of the whole {w.name} batch, then fp64 decode of its first {done} of "
                      f"{w.num_seqs} sequences on one core, {dt:.1f} s"}


def time_oracle(w, steps: int = 1, max_seconds: float = 20.0) -> dict:
    """fp64 oracle on the host cores: the step's cache write and decode over the whole batch,
    repeated up to `steps` times or until `max_seconds` pass."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    cache_dt = {"f32": oracle.F32, "bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}[w.kv_dtype]
    done, t0 = 0, time.perf_counter()
    while done < steps:
        oracle.reshape_and_cache(w.k_new, w.v_new, w.slot_mapping, kc, vc, cache_dtype=cache_dt,
                                 k_scale=w.k_scale, v_scale=w.v_scale)
        oracle.paged_attention_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, cache_dtype=cache_dt,
                                      k_scale=w.k_scale, v_scale=w.v_scale, threads=threads)
        done += 1
        if time.perf_counter() - t0 > max_seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": w.num_seqs * done / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} full step(s) of the {w.name} batch ({w.num_seqs} sequences), fp64, "
                      f"{dt:.1f} s", "seconds": dt, "steps": done}


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_workload_kwargs(config: str, rank: int, batch: int = 0) -> dict:
    """Arguments of the workload a rank serves: every rank holds its own batch (its own sequences, pool and
    seed), so sequences shard across GPUs with no exchange in the data path."""
    from paged_kv_cache_71_gb300 import workload as wl
    kw = {"seed": wl.CONFIG_SEEDS[config] + 1000 * rank} if config != "llama70b_mixed_fp8" else {}
    if config == "llama70b_mixed_fp8" and rank:
        kw["seed"] = wl.CONFIG_SEEDS[config] + 1000 * rank
    if batch and config in ("llama3_8b_gqa", "llama3_8b_gqa_int8", "llama70b_mixed_bf16", "llama70b_mixed_fp8"):
        kw["batch"] = batch
    return kw


def max_over_ranks(value: float, dist, device) -> float:
    """The job's time is its slowest rank's: all-reduce MAX (no-op without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ws: int, seqs_per_rank: int, ms_per_step: float) -> float:
    """Whole-job seq-steps/s: the sequences all ranks served per step over the slowest rank's step time."""
    return ws * seqs_per_rank / (ms_per_step / 1e3)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama3_8b_gqa")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="smaller decode batch of the Llama-3-8B or Llama-70B mixed workload (profiling)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the chunked-prefill kernel on a pool holding just the chunk's sequence")
    ap.add_argument("--swap-only", action="store_true",
                    help="time swap_blocks between the device pool and pinned host memory (Llama-3-8B block geometry)")
    ap.add_argument("--varlen", action="store_true",
                    help="the Llama-70B mixed step (48 decode tokens + one 512-token chunk) as one launch "
                         "(pkv_paged_attention_mixed), timed beside the decode + chunk kernels and beside the "
                         "all-tile varlen launch")
    ap.add_argument("--hash-only", action="store_true",
                    help="time the chained block content hashes of the Llama-3-8B batch's token ids")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-contiguous", action="store_true", help="skip the paged-vs-contiguous decode comparison")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    ws, rank, local = dist_env()
    import torch
    from paged_kv_cache_71_gb300 import workload as wl

    if args.impl == "reference":
        return run_reference(args, ws, rank)
    if args.prefill_only:
        return run_prefill_only(args, local)
    if args.varlen:
        return run_varlen(args, local)
    if args.swap_only:
        return run_swap_only(args, local)
    if args.hash_only:
        return run_hash_only(args, local)

    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from paged_kv_cache_71_gb300.runner import DeviceStep

    # every rank serves its own batch (sequences shard across GPUs; no exchange)
    w = wl.make(args.config, **rank_workload_kwargs(args.config, rank, args.batch))
    st = DeviceStep(w, num_splits=args.num_splits)
    stream = torch.cuda.current_stream()
    launches_per_step = 2 + (1 if st.copy_pairs is not None else 0)
    has_prefill = st.pf_q is not None
    launches_per_step += 1 if has_prefill else 0
    l2_bytes = int(getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 0) or 126 * 2**20)
    plan = l2_plan(w, l2_bytes)
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device="cuda") if plan == "flush" else None

    def flush():
        if flush_buf is not None:
            flush_buf.fill_(1)

    def step():
        st.write(stream)
        st.attend(stream)
        st.prefill(stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if st.device_error():
        raise RuntimeError(f"device error {st.device_error():#x}")

    # ---- device-resident timing: events around each step and around each decode launch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        st.write(stream)
        ev[i][1].record(stream)
        st.attend(stream)
        ev[i][2].record(stream)
        st.prefill(stream)
        ev[i][3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    decode_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    write_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    prefill_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(args.steps)] if has_prefill else None
    if plan == "flush":  # the steps alone, without the flushes between them
        total_ms = sum(ev[i][0].elapsed_time(ev[i][3]) for i in range(args.steps))
    else:
        total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, dist, "cuda")
    ms_per_step = total_ms / args.steps
    value = job_throughput(ws, w.num_seqs, ms_per_step)

    e2e = None if args.no_e2e else time_e2e(args, w, st, plan, flush, dist, ws)

    peak, peak_src = measured_peaks()
    alg = decode_algorithmic_bytes(w)
    dec_avg = float(np.mean(decode_ms))
    achieved = alg / (dec_avg / 1e3) / 1e9
    kname, ksrc = decode_kernel(w)
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": profiled_traffic(w.name, ksrc), "peak_source": peak_src,
            "kernel": kname, "algorithmic_bytes": alg, "avg_launch_us": round(dec_avg * 1e3, 2)}
    uniq = decode_unique_bytes(w)
    if uniq != alg:  # shared blocks: the logical bytes stay the headline, the unique bytes beside them
        roof["unique_bytes"] = uniq
        roof["unique_gbps"] = round(uniq / (dec_avg / 1e3) / 1e9, 1)
    # the binding ceiling of the CUDA-core form: reading the K/V at the HBM peak needs (flops per byte) x peak of
    # fp32 FMA work; where that exceeds the CUDA cores' FMA peak the kernel is bound by arithmetic instead (the
    # tensor-core form does its contractions on the tensor pipe, far below its peak, and stays HBM-bound)
    flops = decode_fma_flops(w)
    fma_needed = flops / alg * peak * 1e9 / 1e12  # TFLOP/s at the HBM peak
    if kname == "paged_decode_kernel" and fma_needed > FP32_FMA_TFLOPS:
        achieved_tf = flops / (dec_avg / 1e3) / 1e12
        roof.update({"bound": "alu", "achieved": round(achieved_tf, 2), "peak": round(FP32_FMA_TFLOPS, 2),
                     "unit": "TFLOP/s", "frac": round(achieved_tf / FP32_FMA_TFLOPS, 4),
                     "peak_source": "fp32 FMA peak from unit counts and clock", "algorithmic_flops": flops,
                     "hbm_gbs": round(achieved, 1), "hbm_frac": round(achieved / peak, 4)})

    contig = None
    if not args.no_contiguous and ws == 1:
        contig = paged_vs_contiguous(args, w, st, flush, stream)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, steps=1000, max_seconds=12.0)
        cpu.pop("seconds", None)
        cpu.pop("steps", None)
        cpu["one_core"] = time_oracle_one_core(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
            "config": line_config(w, args.num_splits, ws, l2_note(w, plan)),
            "kv_gbps": round(achieved, 1), "pct_of_hbm_peak": round(100 * achieved / peak, 2),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "kernels": {"paged_decode_us": round(dec_avg * 1e3, 2),
                        "reshape_and_cache_us": round(float(np.mean(write_ms)) * 1e3, 2),
                        "write_bytes": write_bytes(w)},
        }
        if contig is not None:
            line["paged_vs_contiguous"] = contig
        if has_prefill:
            pf_us = float(np.mean(prefill_ms)) * 1e3
            fl = prefill_flops(w)
            line["kernels"]["paged_prefill_us"] = round(pf_us, 2)
            line["kernels"]["prefill_tflops"] = round(fl / (pf_us * 1e-6) / 1e12, 1)
            line["kernels"]["prefill_flops"] = fl
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def time_e2e(args, w, st, plan, flush, dist, ws) -> dict:
    """The step through the C ABI from host buffers: each step's inputs (q, new K/V, slots, block tables,
    lengths) are copied from pinned host memory and its output copied back, inside the timed region.  Two
    device-side input/output sets alternate, so that a copy stream moves step i+1's inputs in and step i-1's
    output out while the compute stream runs step i; the KV cache itself is device-resident state."""
    import torch
    from paged_kv_cache_71_gb300.runner import DeviceStep
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    outs = ("out",)
    if st.copy_pairs is not None:  # the copy-on-write pairs of the step
        names += ("copy_pairs",)
    if st.pf_q is not None:  # the prefill chunk's queries in, its output out
        names += ("pf_q",)
        outs += ("pf_out",)
    host = {k: getattr(st, k).cpu().pin_memory() for k in names}
    out_host = [{k: torch.empty_like(getattr(st, k), device="cpu").pin_memory() for k in outs} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host[0].values())
    # slot 1: its own input and output buffers, the same caches, workspace and error word
    other = DeviceStep.__new__(DeviceStep)
    other.__dict__.update(st.__dict__)
    for k in names + outs:
        setattr(other, k, torch.empty_like(getattr(st, k)))
    slots = (st, other)
    comp = torch.cuda.current_stream()
    cs = torch.cuda.Stream()
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def h2d_into(i):
        d = slots[i % 2]
        if i >= 2:
            cs.wait_event(comp_done[i % 2])  # step i-2 has finished with these buffers
        with torch.cuda.stream(cs):
            for k in names:
                getattr(d, k).copy_(host[k], non_blocking=True)
        h2d_done[i % 2].record(cs)

    def compute(i):
        d = slots[i % 2]
        comp.wait_event(h2d_done[i % 2])
        d.write(comp)
        d.attend(comp)
        d.prefill(comp)
        comp_done[i % 2].record(comp)

    def d2h_from(i):
        cs.wait_event(comp_done[i % 2])
        with torch.cuda.stream(cs):
            for k in outs:
                out_host[i % 2][k].copy_(getattr(slots[i % 2], k), non_blocking=True)

    def run(n, per_step_flush):
        """n steps; returns the copy stream's (start, end) events around them."""
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if per_step_flush:  # flush, then time one whole step (copies in, compute, copy out) at a time
            ms = 0.0
            for i in range(n):
                with torch.cuda.stream(cs):
                    flush()
                a.record(cs)
                h2d_into(i)
                compute(i)
                d2h_from(i)
                b.record(cs)
                b.synchronize()
                ms += a.elapsed_time(b)
            return ms
        a.record(cs)
        h2d_into(0)
        for i in range(n):
            if i + 1 < n:
                h2d_into(i + 1)
            compute(i)
            d2h_from(i)
        b.record(cs)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    run(args.warmup, plan == "flush")
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = run(args.steps, plan == "flush")
    e2e_ms = max_over_ranks(ms / args.steps, dist, "cuda")
    return {"value": job_throughput(ws, w.num_seqs, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
            "overlap": "copies of step i+1 in and step i out on a copy stream beside step i"
            if plan != "flush" else "one step at a time (L2 flushed between steps)"}


def paged_vs_contiguous(args, w, st, flush, stream) -> dict:
    """The decode kernel over the batch's scattered blocks beside the same kernel over a copy of the pool in which
    every sequence's blocks are consecutive and in logical order (identity block tables: a contiguous KV cache).
    Same values, same work split, so the outputs agree bit for bit; the time difference is what paging costs."""
    import torch
    from paged_kv_cache_71_gb300 import _binding as B
    from paged_kv_cache_71_gb300.runner import to_device
    perm, tables = contiguous_layout(w)
    idx = torch.from_numpy(perm).to("cuda")
    kc = st.k_cache.index_select(0, idx)
    vc = st.v_cache.index_select(0, idx)
    desc = B.CacheDesc.for_cache(kc, w.k_scale, w.v_scale)
    dt = to_device(tables)
    out_c = torch.empty_like(st.out)
    ws_c = torch.zeros(max(B.pkv_paged_attention_workspace_size(desc, w.num_seqs, w.num_q_heads, st.num_splits), 16),
                       dtype=torch.uint8, device="cuda")

    def paged():
        st.attend(stream)

    fn = B.pkv_paged_attention_decode_shared if st.shared else B.pkv_paged_attention_decode

    def contiguous():  # the same decode form as the paged launch
        fn(out_c, st.q, kc, vc, desc, dt, st.context_lens, w.scale, st.num_splits, st.max_context_len, ws_c, st.err,
           stream)

    def timed(fn, n):
        ts = []
        for _ in range(n):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        return [x.elapsed_time(y) * 1e3 for x, y in ts]

    timed(paged, 3)
    timed(contiguous, 3)
    tp, tc = [], []
    for _ in range(3):  # interleaved rounds: both layouts see the same clocks
        tp += timed(paged, args.steps)
        tc += timed(contiguous, args.steps)
    same = bool(torch.equal(out_c, st.out))
    p_us, c_us = float(np.median(tp)), float(np.median(tc))
    return {"paged_us": round(p_us, 2), "contiguous_us": round(c_us, 2),
            "overhead_pct": round(100.0 * (p_us - c_us) / c_us, 2), "outputs_identical": same,
            "contiguous": "each sequence's blocks consecutive and in logical order (shared blocks duplicated)",
            "launches_each": 3 * args.steps}


def run_prefill_only(args, local):
    """The Llama-70B-shaped prefill chunk alone (512 queries at positions 8192..8703, 64 q / 8 kv
    heads, head_dim 128, 16-token blocks) over a pool that holds only that sequence."""
    import torch
    from paged_kv_cache_71_gb300 import _binding as B
    from paged_kv_cache_71_gb300 import workload as wl
    from paged_kv_cache_71_gb300.block_manager import SequenceTables
    from paged_kv_cache_71_gb300.runner import to_device
    torch.cuda.set_device(local)
    kv = "e4m3" if args.config.endswith("fp8") else "bf16"
    NQ, q_start, Hq, Hkv, S, D = 512, 8192, 64, 8, 16, 128
    rng = np.random.default_rng(wl.CONFIG_SEEDS["llama70b_mixed_bf16"])
    kv_len = q_start + NQ
    NB = -(-kv_len // S) + 16
    alloc = SequenceTables(NB, S, free_order=rng.permutation(NB))
    alloc.prefill("chunk", kv_len)
    table = to_device(np.array(alloc.table("chunk"), np.int32))
    dk = to_device(wl.random_values(rng, (NB, S, Hkv, D), kv))
    dv = to_device(wl.random_values(rng, (NB, S, Hkv, D), kv))
    dq = to_device(wl.random_values(rng, (NQ, Hq, D), "bf16"))
    out = torch.empty_like(dq)
    sc = wl.FP8_SCALE if kv == "e4m3" else 1.0
    desc = B.CacheDesc.for_cache(dk, sc, sc)
    scale = 1.0 / np.sqrt(D)

    def run():
        B.pkv_paged_prefill_chunk(out, dq, q_start, dk, dv, desc, table, kv_len, scale)

    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        run()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / args.steps * 1e3
    flops = 4 * D * Hq * sum(q_start + i + 1 for i in range(NQ))
    tflops = flops / (us * 1e-6) / 1e12
    peak = 1941.1
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        pass
    print(json.dumps({"metric": "chunked-prefill tile TFLOP/s", "value": round(tflops, 1), "unit": "TFLOP/s",
                      "us": round(us, 1), "flops": flops, "kv_dtype": kv, "steps": args.steps,
                      "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                                   "unit": "TFLOP/s", "frac": round(tflops / peak, 4)}}), flush=True)


def run_varlen(args, local):
    """The mixed step of the Llama-70B workload (48 decode sequences, one token each, plus the 512-token chunk at
    positions 8192..8703; 64 q / 8 kv heads, bf16 or FP8 KV) as ONE pkv_paged_prefill_varlen launch, in which a
    decode token is a chunk of one query.  Timed beside the two-kernel form of the same step (split-KV decode +
    chunk tile), and the two outputs compared."""
    import torch
    from paged_kv_cache_71_gb300 import _binding as B
    from paged_kv_cache_71_gb300 import workload as wl
    from paged_kv_cache_71_gb300.runner import DeviceStep, to_device
    torch.cuda.set_device(local)
    name = args.config if args.config.startswith("llama70b_mixed") else "llama70b_mixed_bf16"
    kw = {"batch": args.batch} if args.batch else {}
    w = wl.make(name, **kw)
    st = DeviceStep(w, num_splits=args.num_splits)
    st.write()
    torch.cuda.synchronize()
    pf = w.prefill
    B_ = w.num_seqs
    lens = w.context_lens.astype(np.int64)
    # chunks: the 48 decode tokens (query at position L-1, L keys) then the prefill chunk
    cu = np.concatenate([np.arange(B_ + 1), [B_ + pf.q.shape[0]]]).astype(np.int32)
    q_starts = np.concatenate([lens - 1, [pf.q_start]]).astype(np.int32)
    kv_lens = np.concatenate([lens, [pf.kv_len]]).astype(np.int32)
    MB = max(w.block_tables.shape[1], pf.block_table.shape[0])
    tables = np.full((B_ + 1, MB), -1, np.int32)
    tables[:B_, : w.block_tables.shape[1]] = w.block_tables
    tables[B_, : pf.block_table.shape[0]] = pf.block_table
    q_all = torch.cat([st.q, st.pf_q], dim=0).contiguous()
    out_all = torch.empty_like(q_all)
    out_tile = torch.empty_like(q_all)
    d_cu, d_qs, d_kv, d_tab = to_device(cu), to_device(q_starts), to_device(kv_lens), to_device(tables)
    ws_mixed = torch.zeros(max(B.pkv_paged_attention_mixed_workspace_size(st.cache, B_, w.num_q_heads), 16),
                           dtype=torch.uint8, device="cuda")

    def one_launch():  # the mixed-step launch: decode tokens through the decode's work split, chunk on the tile
        B.pkv_paged_attention_mixed(out_all, q_all, d_cu, d_qs, d_kv, st.k_cache, st.v_cache, st.cache, d_tab, B_,
                                    w.scale, ws_mixed, st.err)

    def tile_launch():  # every chunk, decode tokens included, on the prefill tile
        B.pkv_paged_prefill_varlen(out_tile, q_all, d_cu, d_qs, d_kv, st.k_cache, st.v_cache, st.cache, d_tab,
                                   w.scale, st.err)

    def two_kernels():
        st.attend()
        st.prefill()

    def time_it(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps * 1e3

    us_one, us_two, us_tile = [], [], []
    for _ in range(3):  # interleaved rounds: the three forms see the same clocks
        us_one.append(time_it(one_launch))
        us_two.append(time_it(two_kernels))
        us_tile.append(time_it(tile_launch))
    us_one, us_two, us_tile = (float(np.median(x)) for x in (us_one, us_two, us_tile))
    if st.device_error():
        raise RuntimeError(f"device error word {st.device_error():#x}")
    ref = torch.cat([st.out, st.pf_out], dim=0).float()
    diff = float((out_all.float() - ref).abs().max())
    diff_tile = float((out_tile.float() - ref).abs().max())
    print(json.dumps({"metric": "mixed step (48 decode tokens + 512-token chunk) in one launch",
                      "value": round(B_ / (us_one * 1e-6), 1), "unit": "seq-steps/s", "us": round(us_one, 1),
                      "two_kernel_us": round(us_two, 1), "varlen_tile_us": round(us_tile, 1),
                      "kv_dtype": w.kv_dtype, "steps": args.steps,
                      "max_abs_diff_vs_two_kernel_path": round(diff, 5),
                      "varlen_tile_max_abs_diff": round(diff_tile, 5), "config": {"workload": name}}), flush=True)


def run_swap_only(args, local, nblocks: int = 2048):
    """Swap 2048 scattered blocks (16 tokens x 8 kv heads x 128 x bf16, K and V: 64 KB each) out to pinned
    host memory and back in; a contiguous pinned copy of the same bytes is timed beside it."""
    import torch
    from paged_kv_cache_71_gb300 import _binding as B
    from paged_kv_cache_71_gb300 import workload as wl
    from paged_kv_cache_71_gb300.runner import to_device
    torch.cuda.set_device(local)
    rng = np.random.default_rng(7110)
    NB, S, Hkv, D = 8192, 16, 8, 128
    dk = torch.empty((NB, S, Hkv, D), dtype=torch.bfloat16, device="cuda").normal_()
    dv = torch.empty_like(dk).normal_()
    hk = torch.empty((nblocks, S, Hkv, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    out_pairs = to_device(np.stack([rng.choice(NB, nblocks, replace=False), rng.permutation(nblocks)], 1).astype(np.int64))
    in_pairs = to_device(np.stack([rng.permutation(nblocks), rng.choice(NB, nblocks, replace=False)], 1).astype(np.int64))
    desc = B.CacheDesc.for_cache(dk)
    moved = 2 * nblocks * S * Hkv * D * 2
    ref_dev = torch.empty(moved // 2, dtype=torch.bfloat16, device="cuda")
    ref_host = torch.empty(moved // 2, dtype=torch.bfloat16).pin_memory()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps * 1e3

    out_us = timed(lambda: B.pkv_swap_blocks(dk, dv, hk, hv, desc, out_pairs))
    in_us = timed(lambda: B.pkv_swap_blocks(hk, hv, dk, dv, desc, in_pairs))
    d2h_us = timed(lambda: ref_host.copy_(ref_dev, non_blocking=True))
    h2d_us = timed(lambda: ref_dev.copy_(ref_host, non_blocking=True))
    gbs = lambda us: round(moved / (us * 1e-6) / 1e9, 1)
    print(json.dumps({"metric": "swap_blocks GB/s (device <-> pinned host)", "blocks": nblocks, "bytes": moved,
                      "swap_out_us": round(out_us, 1), "swap_out_GBps": gbs(out_us),
                      "swap_in_us": round(in_us, 1), "swap_in_GBps": gbs(in_us),
                      "contiguous_d2h_GBps": gbs(d2h_us), "contiguous_h2d_GBps": gbs(h2d_us),
                      "swap_out_frac_of_contiguous": round(d2h_us / out_us, 3),
                      "swap_in_frac_of_contiguous": round(h2d_us / in_us, 3)}), flush=True)


def run_hash_only(args, local):
    """Content hashes of every full 16-token block of 256 sequences with the Llama-3-8B lengths."""
    import torch
    from paged_kv_cache_71_gb300 import _binding as B
    from paged_kv_cache_71_gb300 import workload as wl
    from paged_kv_cache_71_gb300.runner import to_device
    torch.cuda.set_device(local)
    rng = np.random.default_rng(wl.CONFIG_SEEDS["llama3_8b_gqa"])
    lens = wl.lognormal_lengths(rng, 256)
    S = 16
    toks = to_device(rng.integers(0, 128000, int(lens.sum())).astype(np.int32))
    cu = to_device(np.concatenate([[0], np.cumsum(lens)]).astype(np.int64))
    nfull = lens // S
    offs = to_device(np.concatenate([[0], np.cumsum(nfull)[:-1]]).astype(np.int64))
    out = torch.zeros(int(nfull.sum()), dtype=torch.int64, device="cuda")
    run = lambda: B.pkv_block_hashes(toks, cu, S, offs, out)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        run()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / args.steps * 1e3
    print(json.dumps({"metric": "block content hashes per second", "blocks": int(nfull.sum()),
                      "tokens": int(lens.sum()), "us": round(us, 1),
                      "blocks_per_s": round(int(nfull.sum()) / (us * 1e-6)),
                      "token_GBps": round(4 * int(lens.sum()) / (us * 1e-6) / 1e9, 2)}), flush=True)


def run_reference(args, ws, rank):
    """The oracle, as it stands, timed on the host cores on the same workload (rank 0 only)."""
    if rank != 0:
        return
    from paged_kv_cache_71_gb300 import workload as wl
    w = wl.make(args.config)
    time_oracle(w, steps=1, max_seconds=5.0)  # warm the library and caches
    per = []
    for _ in range(args.warmup):
        time_oracle(w, steps=1, max_seconds=60.0)
    for _ in range(args.steps):
        r = time_oracle(w, steps=1, max_seconds=60.0)
        per.append(r["seconds"])
    ms = 1e3 * float(np.mean(per))
    value = w.num_seqs / (ms / 1e3)
    cores = r["cores"]
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(w, args.num_splits, ws, l2_note(w, l2_plan(w, REFERENCE_L2_BYTES))),
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step = the full {w.name} batch ({w.num_seqs} sequences): cache "
                                       f"write + fp64 decode"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
