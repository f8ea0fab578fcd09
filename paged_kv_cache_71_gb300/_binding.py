"""ctypes binding of libpkv.so: argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but turn tensors into pointers and sizes, pick the current CUDA
stream, call the library and raise on a non-OK status.  All computation
happens in the library's CUDA kernels.  There is no fallback: without a
built libpkv.so these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpkv.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "pkv.h")

PKV_F32, PKV_BF16, PKV_FP8_E4M3, PKV_INT8 = 0, 1, 2, 3
PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_OUT_OF_RANGE",
                4: "PKV_ERR_WORKSPACE", 5: "PKV_ERR_CUDA"}
DEVERR_BAD_SLOT, DEVERR_BAD_BLOCK, DEVERR_BAD_LENGTH, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
DEVERR_Q_RANGE = 0x10

_DTYPE_CODE = {torch.float32: PKV_F32, torch.bfloat16: PKV_BF16, torch.uint8: PKV_FP8_E4M3,
               torch.float8_e4m3fn: PKV_FP8_E4M3, torch.int8: PKV_INT8}


class PkvError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)}: {detail}")


class CacheDesc(ctypes.Structure):
    """Mirror of pkv_cache_desc."""
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("k_head_scales", ctypes.c_void_p), ("v_head_scales", ctypes.c_void_p)]

    @classmethod
    def for_cache(cls, k_cache: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0, k_head_scales=None,
                  v_head_scales=None) -> "CacheDesc":
        """Descriptor of a [NB][S][Hkv][D] cache; the optional per-head scales are fp32 device tensors [Hkv]
        (kept alive by the caller)."""
        NB, S, Hkv, D = k_cache.shape
        return cls(NB, S, Hkv, D, _DTYPE_CODE[k_cache.dtype], float(k_scale), float(v_scale),
                   _ptr(k_head_scales), _ptr(v_head_scales))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libpkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libpkv.so is not built ({LIB_PATH}); run __graft_entry__.build() or "
                           "python -m paged_kv_cache_71_gb300.build")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    D = ctypes.POINTER(CacheDesc)
    L.pkv_reshape_and_cache.argtypes = [P, P, i32, P, i32, P, P, D, P, P]
    L.pkv_paged_attention_workspace_size.argtypes = [D, i32, i32, i32, ctypes.POINTER(sz)]
    L.pkv_paged_attention_decode.argtypes = [P, P, i32, P, P, D, P, i32, P, i32, i32, f32, i32, i32, P, sz, P, P]
    L.pkv_paged_attention_decode_shared.argtypes = L.pkv_paged_attention_decode.argtypes
    L.pkv_copy_blocks.argtypes = [P, P, D, P, i32, P, P]
    L.pkv_paged_attention_decode_static_scratch.argtypes = [P, P, i32, P, P, D, P, i32, P, i32, i32, f32, i32, i32,
                                                            P, P]
    L.pkv_paged_prefill_chunk.argtypes = [P, P, i32, i32, i32, P, P, D, P, i32, i32, f32, P, P]
    L.pkv_paged_prefill_varlen.argtypes = [P, P, i32, i32, P, P, P, P, P, D, P, i32, i32, i32, f32, P, P]
    L.pkv_paged_attention_mixed.argtypes = [P, P, i32, i32, P, P, P, P, P, D, P, i32, i32, i32, i32, f32, P, sz,
                                            P, P]
    L.pkv_paged_attention_mixed_workspace_size.argtypes = [D, i32, i32, ctypes.POINTER(sz)]
    L.pkv_swap_blocks.argtypes = [P, P, i32, P, P, i32, D, P, i32, P, P]
    L.pkv_block_hashes.argtypes = [P, P, i32, i32, P, P, ctypes.c_int64, P, P]
    for name in ("pkv_reshape_and_cache", "pkv_paged_attention_workspace_size", "pkv_paged_attention_decode",
                 "pkv_copy_blocks", "pkv_paged_attention_decode_static_scratch", "pkv_paged_prefill_chunk",
                 "pkv_paged_prefill_varlen", "pkv_swap_blocks", "pkv_block_hashes"):
        getattr(L, name).restype = ctypes.c_int
    L.pkv_status_string.argtypes = [ctypes.c_int]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_last_error.argtypes = []
    L.pkv_last_error.restype = ctypes.c_char_p
    L.pkv_abi_version.argtypes = []
    L.pkv_abi_version.restype = ctypes.c_int32
    _lib = L
    return L


def declared_entry_points() -> list[str]:
    """Names of the functions declared in include/pkv.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:pkv_status|const char\*|int32_t)\s+(pkv_\w+)\s*\(", text, re.M)))


def _check(status: int, func: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, func, (lib().pkv_last_error() or b"").decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype(t: torch.Tensor) -> int:
    return _DTYPE_CODE[t.dtype]


# ---------------------------------------------------------------- entry points

def pkv_reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, cache: CacheDesc, device_error=None,
                          stream=None) -> None:
    _check(lib().pkv_reshape_and_cache(_ptr(k_new), _ptr(v_new), _dtype(k_new), _ptr(slot_mapping),
                                       int(slot_mapping.shape[0]), _ptr(k_cache), _ptr(v_cache),
                                       ctypes.byref(cache), _ptr(device_error), _stream(stream)),
           "pkv_reshape_and_cache")


def pkv_paged_attention_workspace_size(cache: CacheDesc, num_seqs: int, num_q_heads: int, num_splits: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pkv_paged_attention_workspace_size(ctypes.byref(cache), int(num_seqs), int(num_q_heads),
                                                    int(num_splits), ctypes.byref(out)),
           "pkv_paged_attention_workspace_size")
    return int(out.value)


def pkv_paged_attention_decode(out, q, k_cache, v_cache, cache: CacheDesc, block_tables, context_lens,
                               scale: float, num_splits: int = 0, max_context_len: int = 0, workspace=None,
                               device_error=None, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pkv_paged_attention_decode(_ptr(out), _ptr(q), _dtype(q), _ptr(k_cache), _ptr(v_cache),
                                            ctypes.byref(cache), _ptr(block_tables), int(block_tables.shape[1]),
                                            _ptr(context_lens), int(q.shape[0]), int(q.shape[1]), float(scale),
                                            int(num_splits), int(max_context_len), _ptr(workspace), ws_bytes,
                                            _ptr(device_error), _stream(stream)),
           "pkv_paged_attention_decode")


def pkv_paged_attention_decode_shared(out, q, k_cache, v_cache, cache: CacheDesc, block_tables, context_lens,
                                      scale: float, num_splits: int = 0, max_context_len: int = 0, workspace=None,
                                      device_error=None, stream=None) -> None:
    """pkv_paged_attention_decode for a batch whose tables share physical blocks (same arguments)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pkv_paged_attention_decode_shared(_ptr(out), _ptr(q), _dtype(q), _ptr(k_cache), _ptr(v_cache),
                                                   ctypes.byref(cache), _ptr(block_tables),
                                                   int(block_tables.shape[1]), _ptr(context_lens), int(q.shape[0]),
                                                   int(q.shape[1]), float(scale), int(num_splits),
                                                   int(max_context_len), _ptr(workspace), ws_bytes,
                                                   _ptr(device_error), _stream(stream)),
           "pkv_paged_attention_decode_shared")


def pkv_paged_attention_decode_static_scratch(out, q, k_cache, v_cache, cache: CacheDesc, block_tables,
                                              context_lens, scale: float, num_splits: int = 0,
                                              max_context_len: int = 0, device_error=None, stream=None) -> None:
    """pkv_paged_attention_decode without a workspace argument: the library's static scratch is used."""
    _check(lib().pkv_paged_attention_decode_static_scratch(
        _ptr(out), _ptr(q), _dtype(q), _ptr(k_cache), _ptr(v_cache), ctypes.byref(cache), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(context_lens), int(q.shape[0]), int(q.shape[1]), float(scale),
        int(num_splits), int(max_context_len), _ptr(device_error), _stream(stream)),
        "pkv_paged_attention_decode_static_scratch")


def pkv_paged_prefill_chunk(out, q, q_start: int, k_cache, v_cache, cache: CacheDesc, block_table, kv_len: int,
                            scale: float, device_error=None, stream=None) -> None:
    _check(lib().pkv_paged_prefill_chunk(_ptr(out), _ptr(q), _dtype(q), int(q.shape[0]), int(q_start),
                                         _ptr(k_cache), _ptr(v_cache), ctypes.byref(cache), _ptr(block_table),
                                         int(kv_len), int(q.shape[1]), float(scale), _ptr(device_error),
                                         _stream(stream)),
           "pkv_paged_prefill_chunk")


def pkv_paged_attention_mixed_workspace_size(cache: CacheDesc, num_decode: int, num_q_heads: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pkv_paged_attention_mixed_workspace_size(ctypes.byref(cache), int(num_decode), int(num_q_heads),
                                                          ctypes.byref(out)),
           "pkv_paged_attention_mixed_workspace_size")
    return int(out.value)


def pkv_paged_attention_mixed(out, q, cu_q, q_starts, kv_lens, k_cache, v_cache, cache: CacheDesc, block_tables,
                              num_decode: int, scale: float, workspace=None, device_error=None, stream=None) -> None:
    """A mixed step in one launch: chunks [0, num_decode) are decode tokens, the rest prefill chunks (varlen arrays
    on the device, q/out [total_q_tokens][Hq][128])."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pkv_paged_attention_mixed(_ptr(out), _ptr(q), _dtype(q), int(q.shape[0]), _ptr(cu_q),
                                           _ptr(q_starts), _ptr(kv_lens), _ptr(k_cache), _ptr(v_cache),
                                           ctypes.byref(cache), _ptr(block_tables), int(block_tables.shape[1]),
                                           int(kv_lens.shape[0]), int(num_decode), int(q.shape[1]), float(scale),
                                           _ptr(workspace), ws_bytes, _ptr(device_error), _stream(stream)),
           "pkv_paged_attention_mixed")


def pkv_paged_prefill_varlen(out, q, cu_q, q_starts, kv_lens, k_cache, v_cache, cache: CacheDesc, block_tables,
                             scale: float, device_error=None, stream=None) -> None:
    """Several prefill chunks in one launch; q/out are [total_q_tokens][Hq][128], the index arrays on the device."""
    _check(lib().pkv_paged_prefill_varlen(_ptr(out), _ptr(q), _dtype(q), int(q.shape[0]), _ptr(cu_q),
                                          _ptr(q_starts), _ptr(kv_lens), _ptr(k_cache), _ptr(v_cache),
                                          ctypes.byref(cache), _ptr(block_tables), int(block_tables.shape[1]),
                                          int(kv_lens.shape[0]), int(q.shape[1]), float(scale),
                                          _ptr(device_error), _stream(stream)),
           "pkv_paged_prefill_varlen")


STATIC_SCRATCH_BYTES = 12 * 1024 * 1024  # PKV_STATIC_SCRATCH_BYTES in include/pkv.h


def pkv_copy_blocks(k_cache, v_cache, cache: CacheDesc, block_mapping, device_error=None, stream=None) -> None:
    _check(lib().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), ctypes.byref(cache), _ptr(block_mapping),
                                 int(block_mapping.shape[0]), _ptr(device_error), _stream(stream)),
           "pkv_copy_blocks")


def pkv_swap_blocks(src_k, src_v, dst_k, dst_v, cache: CacheDesc, block_mapping, device_error=None,
                    stream=None) -> None:
    """Whole-block copies between two pools (device or pinned host memory)."""
    _check(lib().pkv_swap_blocks(_ptr(src_k), _ptr(src_v), int(src_k.shape[0]), _ptr(dst_k), _ptr(dst_v),
                                 int(dst_k.shape[0]), ctypes.byref(cache), _ptr(block_mapping),
                                 int(block_mapping.shape[0]), _ptr(device_error), _stream(stream)),
           "pkv_swap_blocks")


def pkv_block_hashes(token_ids, cu_tokens, block_size: int, out_offsets, hashes, device_error=None,
                     stream=None) -> None:
    """Chained FNV-1a-64 content hashes of every full block (hashes: int64/uint64 device tensor)."""
    _check(lib().pkv_block_hashes(_ptr(token_ids), _ptr(cu_tokens), int(cu_tokens.shape[0]) - 1, int(block_size),
                                  _ptr(out_offsets), _ptr(hashes), int(hashes.numel()), _ptr(device_error),
                                  _stream(stream)),
           "pkv_block_hashes")


def pkv_status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def pkv_last_error() -> str:
    return (lib().pkv_last_error() or b"").decode()


def pkv_abi_version() -> int:
    return int(lib().pkv_abi_version())
