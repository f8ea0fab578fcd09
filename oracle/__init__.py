"""CPU oracle for paged KV-cache decode (fp64, plain C, OpenMP).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The
product path (the CUDA library and its binding) never imports, links or
runs it, and shares no code with it.

Every function here is a thin numpy marshalling layer over ``pkv_oracle.c``;
the arithmetic lives in that file, with the page citations for each step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

F32, BF16, E4M3, I8 = 0, 1, 2, 3
_STATUS = {0: "ok", 1: "bad argument", 2: "slot out of range", 3: "block id out of range", 4: "out of memory"}

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        lib.orc_bf16_to_double.restype = f64
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        lib.orc_f32_to_bf16.argtypes = [f32]
        lib.orc_e4m3_to_double.restype = f64
        lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
        lib.orc_f32_to_e4m3.argtypes = [f32]
        lib.orc_f32_to_i8.restype = ctypes.c_int8
        lib.orc_f32_to_i8.argtypes = [f32]
        lib.orc_lookup.restype = i32
        lib.orc_lookup.argtypes = [P, i64, i32, ctypes.POINTER(ctypes.c_int)]
        lib.orc_reshape_and_cache.restype = i32
        lib.orc_reshape_and_cache.argtypes = [P, P, i32, P, i32, P, P, i32, i32, i32, i32, i32, f32, f32, P, P]
        lib.orc_copy_blocks.restype = i32
        lib.orc_copy_blocks.argtypes = [P, P, ctypes.c_size_t, i32, P, i32]
        lib.orc_swap_blocks.restype = i32
        lib.orc_swap_blocks.argtypes = [P, P, i32, P, P, i32, ctypes.c_size_t, P, i32]
        lib.orc_fnv1a64.restype = ctypes.c_uint64
        lib.orc_fnv1a64.argtypes = [P, ctypes.c_size_t, ctypes.c_uint64]
        lib.orc_block_hashes.restype = None
        lib.orc_block_hashes.argtypes = [P, P, i32, i32, P, P]
        lib.orc_paged_attention_decode.restype = i32
        lib.orc_paged_attention_decode.argtypes = [P, P, i32, P, P, i32, f64, f64, P, P, i32, i32, i32, i32,
                                                   P, i32, P, i32, i32, f64, P, i32, i32]
        lib.orc_paged_prefill_chunk.restype = i32
        lib.orc_paged_prefill_chunk.argtypes = [P, P, i32, i32, i32, P, P, i32, f64, f64, P, P, i32, i32, i32,
                                                i32, P, i32, i32, f64, P, i32, i32]
        lib.orc_max_threads.restype = i32
        lib.orc_max_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _dtype_code(a: np.ndarray, declared: int | None = None) -> int:
    if declared is not None:
        return declared
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.uint8:
        return E4M3
    if a.dtype == np.int8:
        return I8
    raise TypeError(f"oracle: unsupported array dtype {a.dtype} (f32, bf16 as uint16, e4m3 as uint8, int8)")


def _check(status: int, what: str, allow=()):
    if status != 0 and status not in allow:
        raise OracleError(f"{what}: {_STATUS.get(status, status)}")
    return status


# ---------------------------------------------------------------- formats

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.orc_bf16_to_double(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_f32_to_bf16(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(x))


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_e4m3_to_double(int(c)) for c in flat], dtype=np.float64).reshape(np.shape(codes))


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_f32_to_e4m3(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(x))


def f32_to_i8(y: np.ndarray) -> np.ndarray:
    """Symmetric INT8 code of already-divided values y (RNE, clamped to +-127)."""
    lib = _load()
    flat = np.ascontiguousarray(y, dtype=np.float32).ravel()
    return np.array([lib.orc_f32_to_i8(float(v)) for v in flat], dtype=np.int8).reshape(np.shape(y))


def lookup(table: np.ndarray, p: int, block_size: int) -> tuple[int, int]:
    """(physical block, offset) of logical position p through one block table."""
    lib = _load()
    t = np.ascontiguousarray(table, dtype=np.int32)
    off = ctypes.c_int(0)
    blk = lib.orc_lookup(_ptr(t), int(p), int(block_size), ctypes.byref(off))
    return int(blk), int(off.value)


# ---------------------------------------------------------------- kernels' definitions

def _head_scales(x, dtype):
    return None if x is None else np.ascontiguousarray(x, dtype=dtype)


def reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, *, src_dtype=None,
                      cache_dtype=None, k_scale=1.0, v_scale=1.0, k_head_scales=None, v_head_scales=None):
    """Write new tokens into host byte images of the caches, in place.

    k_new/v_new: [T, Hkv, D] (float32, or uint16 holding bf16 bits);
    caches: [NB, S, Hkv, D] (float32 / uint16 bf16 / uint8 e4m3 / int8).
    k_head_scales / v_head_scales: optional fp32 [Hkv], replacing the per-tensor scales per KV head.
    Returns 0, or 2 if some slot was beyond the pool (those tokens skipped)."""
    lib = _load()
    T, Hkv, D = k_new.shape
    NB, S = k_cache.shape[:2]
    assert k_cache.shape == (NB, S, Hkv, D) and v_cache.shape == k_cache.shape
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    khs, vhs = _head_scales(k_head_scales, np.float32), _head_scales(v_head_scales, np.float32)
    st = lib.orc_reshape_and_cache(_ptr(k_new), _ptr(v_new), _dtype_code(k_new, src_dtype), _ptr(sm), T,
                                   _ptr(k_cache), _ptr(v_cache), _dtype_code(k_cache, cache_dtype),
                                   NB, S, Hkv, D, float(k_scale), float(v_scale), _ptr(khs), _ptr(vhs))
    return _check(st, "reshape_and_cache", allow=(2,))


def copy_blocks(k_cache, v_cache, block_mapping):
    """Copy whole physical blocks (src -> dst pairs, in order), in place."""
    lib = _load()
    NB = k_cache.shape[0]
    bm = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    block_bytes = k_cache[0].nbytes
    st = lib.orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), block_bytes, NB, _ptr(bm), bm.shape[0])
    return _check(st, "copy_blocks", allow=(3,))


def swap_blocks(src_k, src_v, dst_k, dst_v, block_mapping):
    """Copy whole blocks from one pool to another (src -> dst pairs, in order), in place."""
    lib = _load()
    bm = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    assert src_k[0].nbytes == dst_k[0].nbytes
    st = lib.orc_swap_blocks(_ptr(src_k), _ptr(src_v), src_k.shape[0], _ptr(dst_k), _ptr(dst_v), dst_k.shape[0],
                             src_k[0].nbytes, _ptr(bm), bm.shape[0])
    return _check(st, "swap_blocks", allow=(3,))


FNV_OFFSET_BASIS = 14695981039346656037


def fnv1a64(data: bytes, h: int = FNV_OFFSET_BASIS) -> int:
    lib = _load()
    buf = np.frombuffer(bytes(data), dtype=np.uint8).copy() if len(data) else np.zeros(1, np.uint8)
    return int(lib.orc_fnv1a64(_ptr(buf), len(data), h))


def block_hashes(tokens, cu_tokens, block_size):
    """Chained content hashes of every full block of every sequence (uint64, concatenated)."""
    lib = _load()
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    cu = np.ascontiguousarray(cu_tokens, dtype=np.int64)
    B = cu.shape[0] - 1
    nfull = (cu[1:] - cu[:-1]) // block_size
    offs = np.zeros(B, np.int64)
    if B > 1:
        offs[1:] = np.cumsum(nfull)[:-1]
    out = np.zeros(max(1, int(nfull.sum())), np.uint64)
    lib.orc_block_hashes(_ptr(tok if tok.size else np.zeros(1, np.int32)), _ptr(cu), B, int(block_size),
                         _ptr(offs), _ptr(out))
    return out[: int(nfull.sum())]


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, *,
                           q_dtype=None, cache_dtype=None, k_scale=1.0, v_scale=1.0,
                           k_head_scales=None, v_head_scales=None, seqs=None, threads=0) -> np.ndarray:
    """Textbook fp64 attention of each sequence's query over its paged K/V.

    q: [B, Hq, D]; caches [NB, S, Hkv, D]; block_tables [B, MB] int32;
    context_lens [B] int32.  Returns float64 [len(seqs) or B, Hq, D]."""
    lib = _load()
    B, Hq, D = q.shape
    NB, S, Hkv, D2 = k_cache.shape
    assert D2 == D
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    sel = None if seqs is None else np.ascontiguousarray(seqs, dtype=np.int32)
    n = B if sel is None else sel.shape[0]
    out = np.empty((n, Hq, D), dtype=np.float64)
    khs, vhs = _head_scales(k_head_scales, np.float64), _head_scales(v_head_scales, np.float64)
    st = lib.orc_paged_attention_decode(_ptr(out), _ptr(q), _dtype_code(q, q_dtype), _ptr(k_cache),
                                        _ptr(v_cache), _dtype_code(k_cache, cache_dtype), float(k_scale),
                                        float(v_scale), _ptr(khs), _ptr(vhs), NB, S, Hkv, D, _ptr(bt),
                                        bt.shape[1], _ptr(cl), B, Hq,
                                        float(scale), _ptr(sel), n, int(threads))
    _check(st, "paged_attention_decode")
    return out


def paged_prefill_chunk(q, q_start, k_cache, v_cache, block_table, kv_len, scale, *,
                        q_dtype=None, cache_dtype=None, k_scale=1.0, v_scale=1.0,
                        k_head_scales=None, v_head_scales=None, rows=None, threads=0) -> np.ndarray:
    """Causal fp64 attention of a chunk of NQ query tokens (positions
    q_start..q_start+NQ-1) over one sequence's paged K/V.  Returns
    float64 [len(rows) or NQ, Hq, D]."""
    lib = _load()
    NQ, Hq, D = q.shape
    NB, S, Hkv, D2 = k_cache.shape
    assert D2 == D
    tb = np.ascontiguousarray(block_table, dtype=np.int32)
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = NQ if sel is None else sel.shape[0]
    out = np.empty((n, Hq, D), dtype=np.float64)
    khs, vhs = _head_scales(k_head_scales, np.float64), _head_scales(v_head_scales, np.float64)
    st = lib.orc_paged_prefill_chunk(_ptr(out), _ptr(q), _dtype_code(q, q_dtype), NQ, int(q_start),
                                     _ptr(k_cache), _ptr(v_cache), _dtype_code(k_cache, cache_dtype),
                                     float(k_scale), float(v_scale), _ptr(khs), _ptr(vhs), NB, S, Hkv, D,
                                     _ptr(tb), int(kv_len),
                                     Hq, float(scale), _ptr(sel), n, int(threads))
    _check(st, "paged_prefill_chunk")
    return out


def max_threads() -> int:
    return int(_load().orc_max_threads())
