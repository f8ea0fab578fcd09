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
    128-dim heads, and bf16 caches of 128-dim heads in GQA groups of 8, take the tensor-core form, everything else
    the CUDA-core form."""
    G = w.num_q_heads // w.num_kv_heads
    if w.head_dim == 128 and (w.kv_dtype in ("e4m3", "i8") or (w.kv_dtype == "bf16" and G >= 8)):
        tag = {"e4m3": "fp8", "i8": "i8", "bf16": "bf16"}[w.kv_dtype]
        return "paged_decode_mma_kernel", ("decode_mma.cuh", "decode.cuh", "pkv_device.cuh",
                                           f"decode_mma_{tag}_s{w.block_size}.cu")
    return "paged_decode_kernel", DECODE_SOURCES


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
    if batch and config in ("llama3_8b_gqa", "llama70b_mixed_bf16", "llama70b_mixed_fp8"):
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
                    help="the Llama-70B mixed step (48 decode tokens + one 512-token chunk) as one varlen prefill "
                         "launch, timed beside the decode + chunk kernels")
    ap.add_argument("--hash-only", action="store_true",
                    help="time the chained block content hashes of the Llama-3-8B batch's token ids")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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

    from paged_kv_cache_71_gb300 import _binding as B
    from paged_kv_cache_71_gb300.runner import DeviceStep, to_device

    # every rank serves its own batch (sequences shard across GPUs; no exchange)
    w = wl.make(args.config, **rank_workload_kwargs(args.config, rank, args.batch))
    st = DeviceStep(w, num_splits=args.num_splits)
    stream = torch.cuda.current_stream()
    launches_per_step = 2 + (1 if st.copy_pairs is not None else 0)

    has_prefill = st.pf_q is not None
    launches_per_step += 1 if has_prefill else 0

    def step():
        st.write(stream)
        st.attend(stream)
        st.prefill(stream)

    for _ in range(args.warmup):
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
    total_ms = t_start.elapsed_time(t_end)
    decode_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    write_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    prefill_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(args.steps)] if has_prefill else None
    total_ms = max_over_ranks(total_ms, dist, "cuda")
    ms_per_step = total_ms / args.steps
    value = job_throughput(ws, w.num_seqs, ms_per_step)

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        host = {k: getattr(st, k).cpu().pin_memory() for k in
                ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")}
        out_host = torch.empty_like(st.out, device="cpu").pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size()

        def e2e_step():
            for k, t in host.items():
                getattr(st, k).copy_(t, non_blocking=True)
            step()
            out_host.copy_(st.out, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / args.steps, dist, "cuda")
        e2e = {"value": job_throughput(ws, w.num_seqs, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms}

    peak, peak_src = measured_peaks()
    alg = decode_algorithmic_bytes(w)
    dec_avg = float(np.mean(decode_ms))
    achieved = alg / (dec_avg / 1e3) / 1e9
    kname, ksrc = decode_kernel(w)
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": profiled_traffic(w.name, ksrc), "peak_source": peak_src,
            "kernel": kname, "algorithmic_bytes": alg, "avg_launch_us": round(dec_avg * 1e3, 2)}
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

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, steps=1000, max_seconds=12.0)
        cpu.pop("seconds", None)
        cpu.pop("steps", None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
            "config": {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                       "kv_dtype": w.kv_dtype, "mean_context": float(w.context_lens.mean()),
                       "num_splits": args.num_splits, "parallelism": f"replicas{ws}",
                       "l2": f"inputs larger than L2: {alg / 1e9:.2f} GB of K/V read per step"},
            "kv_gbps": round(achieved, 1), "pct_of_hbm_peak": round(100 * achieved / peak, 2),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "kernels": {"paged_decode_us": round(dec_avg * 1e3, 2),
                        "reshape_and_cache_us": round(float(np.mean(write_ms)) * 1e3, 2),
                        "write_bytes": write_bytes(w)},
        }
        if has_prefill:
            pf_us = float(np.mean(prefill_ms)) * 1e3
            fl = prefill_flops(w)
            line["kernels"]["paged_prefill_us"] = round(pf_us, 2)
            line["kernels"]["prefill_tflops"] = round(fl / (pf_us * 1e-6) / 1e12, 1)
            line["kernels"]["prefill_flops"] = fl
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


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
    d_cu, d_qs, d_kv, d_tab = to_device(cu), to_device(q_starts), to_device(kv_lens), to_device(tables)

    def one_launch():
        B.pkv_paged_prefill_varlen(out_all, q_all, d_cu, d_qs, d_kv, st.k_cache, st.v_cache, st.cache, d_tab,
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

    us_one = time_it(one_launch)
    us_two = time_it(two_kernels)
    if st.device_error():
        raise RuntimeError(f"device error word {st.device_error():#x}")
    ref = torch.cat([st.out, st.pf_out], dim=0).float()
    diff = float((out_all.float() - ref).abs().max())
    print(json.dumps({"metric": "mixed step (48 decode tokens + 512-token chunk) in one varlen launch",
                      "value": round(B_ / (us_one * 1e-6), 1), "unit": "seq-steps/s", "us": round(us_one, 1),
                      "two_kernel_us": round(us_two, 1), "kv_dtype": w.kv_dtype, "steps": args.steps,
                      "max_abs_diff_vs_two_kernel_path": round(diff, 5), "config": {"workload": name}}), flush=True)


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
            "config": {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
                       "kv_dtype": w.kv_dtype},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step = the full {w.name} batch ({w.num_seqs} sequences): cache "
                                       f"write + fp64 decode"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
