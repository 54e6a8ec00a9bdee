"""ctypes binding of libpkv (the C ABI in include/pkv.h).

Argument marshalling only: shapes and dtypes are read off torch tensors,
pointers are passed through, and every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if ``_lib/libpkv.so`` is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

PKV_OK = 0
PKV_ERR_UNSUPPORTED = 4
PKV_ERR_RANGE = 9
PKV_FP8_E4M3 = 3
PKV_INT8 = 4
_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
# 8-bit pools: uint8 tensors hold E4M3 codes, int8 tensors int8 codes
_POOL_DTYPES = {**_DTYPES, torch.uint8: PKV_FP8_E4M3, torch.int8: PKV_INT8}
_CODE_DTYPES = (torch.uint8, torch.int8)


class PkvError(RuntimeError):
    """A libpkv call returned a non-zero pkv_status."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed: {message} (status {status})")
        self.status = status


class DecodeOptions(ctypes.Structure):
    """Mirror of ``pkv_decode_options``."""
    _fields_ = [("window", ctypes.c_int32), ("num_sinks", ctypes.c_int32),
                ("tokens_per_split", ctypes.c_int32), ("k_new", ctypes.c_void_p),
                ("v_new", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p)]


class CacheLayout(ctypes.Structure):
    """Mirror of ``pkv_cache_layout``."""
    _fields_ = [("num_blocks", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class IndexErrorInfo(ctypes.Structure):
    """Mirror of ``pkv_index_error``."""
    _fields_ = [("what", ctypes.c_int32), ("row", ctypes.c_int64), ("col", ctypes.c_int64),
                ("value", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load libpkv.so (built by ``paged_kv_cache_24_gb300._build``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libpkv.so not found at {path}; build it with "
                "`python -m paged_kv_cache_24_gb300._build` (there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lay = ctypes.POINTER(CacheLayout)
        sig = {
            "pkv_slot_mapping": [vp, i32, i32, vp, i32, vp, vp],
            "pkv_stage_copy": [vp, vp, i64, vp],
            "pkv_append": [vp, vp, vp, i64, vp, vp, lay, vp],
            "pkv_decode": [vp, i32, i32, vp, vp, lay, vp, i32, vp, i32, f32, vp, vp],
            "pkv_decode_split": [vp, i32, i32, vp, vp, lay, vp, i32, vp, i32, f32, vp, i32, vp],
            "pkv_append_decode": [vp, vp, vp, i32, i32, vp, vp, lay, vp, i32, vp, i32, f32, vp,
                                  i32, vp],
            "pkv_decode_ex": [vp, i32, i32, vp, vp, lay, vp, i32, vp, f32, vp,
                              ctypes.POINTER(DecodeOptions), vp],
            "pkv_append_fp8": [vp, vp, i32, vp, i64, vp, vp, vp, vp, lay, vp],
            "pkv_append_int8": [vp, vp, i32, vp, i64, vp, vp, vp, vp, lay, vp],
            "pkv_prefill": [vp, vp, vp, vp, i32, i32, i32, vp, vp, lay, vp, i32, vp, i32, i32,
                            f32, vp, vp],
            "pkv_decode_plan": [i32, i32, lay, i32, i32, i32, i32, i32, ctypes.POINTER(i32),
                                ctypes.POINTER(i32)],
            "pkv_release_workspaces": [],
            "pkv_validate_indices": [vp, i32, i32, vp, vp, i64, i64, i32, vp,
                                     ctypes.POINTER(IndexErrorInfo)],
            "pkv_device_address": [vp, ctypes.POINTER(vp)],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.pkv_status_string.argtypes = [ctypes.c_int]
        lib.pkv_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(name: str, status: int) -> None:
    if status != PKV_OK:
        msg = load_library().pkv_status_string(status).decode()
        raise PkvError(name, status, msg)


def status_string(status: int) -> str:
    return load_library().pkv_status_string(status).decode()


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def cache_layout(cache: torch.Tensor) -> CacheLayout:
    """Layout of a head-major pool tensor [num_blocks, num_kv_heads, block_size, head_dim]
    (a uint8 pool holds FP8 E4M3 codes, an int8 pool int8 codes)."""
    if cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    if cache.dtype not in _POOL_DTYPES:
        raise TypeError(f"unsupported cache dtype {cache.dtype}")
    if not cache.is_contiguous():
        raise ValueError("cache must be contiguous")
    nb, hkv, bs, d = cache.shape
    return CacheLayout(nb, hkv, bs, d, _POOL_DTYPES[cache.dtype])


def _compute_dtype(cache: torch.Tensor):
    """dtype of q / out / new tokens for a pool (fp16 for 8-bit pools)."""
    return torch.float16 if cache.dtype in _CODE_DTYPES else cache.dtype


def _check_scales(k_cache, k_scale, v_scale):
    if k_cache.dtype not in _CODE_DTYPES:
        _require(k_scale is None and v_scale is None, "scales are only for 8-bit pools")
        return
    shape = tuple(k_cache.shape[:3])
    for sc in (k_scale, v_scale):
        _require(sc is not None and sc.dtype == torch.float32 and tuple(sc.shape) == shape
                 and sc.is_contiguous() and sc.device.type == "cuda",
                 f"8-bit pools need contiguous float32 scales of shape {shape}")


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _on_cuda(*ts) -> None:
    for t in ts:
        if t is not None and t.device.type != "cuda":
            raise ValueError("libpkv operates on CUDA tensors only")


def pkv_device_address(t: torch.Tensor) -> int | None:
    """The address through which the library's kernels reach t's memory (device
    memory, or pinned host memory), or None for pageable host memory."""
    addr = ctypes.c_void_p()
    rc = load_library().pkv_device_address(ctypes.c_void_p(t.data_ptr()), ctypes.byref(addr))
    if rc == PKV_ERR_UNSUPPORTED:
        return None
    _check("pkv_device_address", rc)
    return addr.value


def _address(t: torch.Tensor, what: str) -> int:
    """A decode's q, new K/V or output: a CUDA tensor, or a pinned host tensor
    the kernels read or write directly over the host link."""
    if t.device.type == "cuda":
        return t.data_ptr()
    _require(t.is_pinned(), f"{what} must be a CUDA tensor or pinned host memory")
    addr = pkv_device_address(t)
    _require(addr is not None, f"this GPU cannot address the pinned {what} buffer")
    return addr


def pkv_stage_copy(dst: torch.Tensor, src: torch.Tensor, nbytes: int | None = None,
                   stream=None) -> int:
    """Copy the first nbytes (default: all) of src into dst with a kernel; either
    tensor may live in pinned host memory.  Returns the library's status
    (PKV_ERR_UNSUPPORTED = 4 when a side is pageable host memory; nothing is
    launched then); other errors raise."""
    _require(src.is_contiguous() and dst.is_contiguous(), "src and dst must be contiguous")
    n = src.numel() * src.element_size() if nbytes is None else int(nbytes)
    _require(0 <= n <= src.numel() * src.element_size() and n <= dst.numel() * dst.element_size(),
             "nbytes exceeds a tensor")
    rc = load_library().pkv_stage_copy(_ptr(dst), _ptr(src), n, _stream(stream))
    if rc != PKV_ERR_UNSUPPORTED:
        _check("pkv_stage_copy", rc)
    return rc


def pkv_slot_mapping(block_tables: torch.Tensor, positions: torch.Tensor, block_size: int,
                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Slots of each sequence's new token (int64 [B], -1 = no slot)."""
    _on_cuda(block_tables, positions, out)
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2
             and block_tables.is_contiguous(), "block_tables must be contiguous int32 [B, MB]")
    _require(positions.dtype == torch.int64 and positions.is_contiguous()
             and positions.numel() == block_tables.shape[0], "positions must be int64 [B]")
    if out is None:
        out = torch.empty(block_tables.shape[0], dtype=torch.int64, device=block_tables.device)
    _check("pkv_slot_mapping", load_library().pkv_slot_mapping(
        _ptr(block_tables), block_tables.shape[0], block_tables.shape[1], _ptr(positions),
        int(block_size), _ptr(out), _stream(stream)))
    return out


def pkv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
               k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> None:
    """Write k[i], v[i] ([T, Hkv, D]) into cache slot slot_mapping[i] (int64, <0 skips).
    k and v may be pinned host tensors (read by the kernel over the host link)."""
    _on_cuda(slot_mapping, k_cache, v_cache)
    layout = cache_layout(k_cache)
    _require(v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype
             and v_cache.is_contiguous(), "v_cache must match k_cache")
    T = k.shape[0]
    shape = (T, layout.num_kv_heads, layout.head_dim)
    _require(tuple(k.shape) == shape and tuple(v.shape) == shape, f"k and v must be {shape}")
    _require(k.dtype == k_cache.dtype and v.dtype == k_cache.dtype, "k/v dtype must match cache")
    _require(k.is_contiguous() and v.is_contiguous(), "k and v must be contiguous")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == T
             and slot_mapping.is_contiguous(), "slot_mapping must be int64 [T]")
    _check("pkv_append", load_library().pkv_append(
        _address(k, "k"), _address(v, "v"), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache),
        ctypes.byref(layout), _stream(stream)))


def pkv_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               block_tables: torch.Tensor, context_lens: torch.Tensor, window: int,
               scale: float, out: torch.Tensor | None = None, tokens_per_split: int = 0,
               stream=None, num_sinks: int = 0, k_scale: torch.Tensor | None = None,
               v_scale: torch.Tensor | None = None) -> torch.Tensor:
    """Decode attention of q [B, Hq, D] over the paged context; returns out [B, Hq, D].
    With a window, ``num_sinks`` first positions are attended as well.  8-bit pools
    (uint8 E4M3 or int8 codes) take their row scales and fp16 q.  ``q`` and ``out``
    may be pinned host tensors: the kernels then read or write them straight
    over the host link."""
    _on_cuda(k_cache, v_cache, block_tables, context_lens, k_scale, v_scale)
    layout = cache_layout(k_cache)
    _require(v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype
             and v_cache.is_contiguous(), "v_cache must match k_cache")
    _check_scales(k_cache, k_scale, v_scale)
    _require(q.dim() == 3 and q.shape[2] == layout.head_dim and q.is_contiguous()
             and q.dtype == _compute_dtype(k_cache),
             "q must be contiguous [B, Hq, D] of the cache's compute dtype")
    B, Hq, D = q.shape
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2
             and block_tables.shape[0] == B and block_tables.is_contiguous(),
             "block_tables must be contiguous int32 [B, MB]")
    _require(context_lens.dtype == torch.int32 and context_lens.numel() == B
             and context_lens.is_contiguous(), "context_lens must be int32 [B]")
    if out is None:
        out = torch.empty_like(q, device=k_cache.device)
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(),
             "out must be contiguous and shaped like q")
    opts = DecodeOptions(int(window), int(num_sinks), int(tokens_per_split), None, None,
                         _ptr(k_scale) or None, _ptr(v_scale) or None)
    _check("pkv_decode", load_library().pkv_decode_ex(
        _address(q, "q"), B, Hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(layout),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), float(scale),
        _address(out, "out"), ctypes.byref(opts), _stream(stream)))
    return out


def _append_q8(fn: str, code_dtype, k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale,
               stream) -> None:
    _on_cuda(slot_mapping, k_cache, v_cache, k_scale, v_scale)
    layout = cache_layout(k_cache)
    _require(k_cache.dtype == code_dtype, f"{fn} writes {code_dtype} pools")
    _require(v_cache.shape == k_cache.shape and v_cache.dtype == code_dtype
             and v_cache.is_contiguous(), "v_cache must match k_cache")
    _check_scales(k_cache, k_scale, v_scale)
    T = k.shape[0]
    shape = (T, layout.num_kv_heads, layout.head_dim)
    _require(tuple(k.shape) == shape and tuple(v.shape) == shape and k.dtype == v.dtype
             and k.dtype in _DTYPES and k.is_contiguous() and v.is_contiguous(),
             f"k and v must be contiguous {shape} fp32/fp16/bf16")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == T
             and slot_mapping.is_contiguous(), "slot_mapping must be int64 [T]")
    _check(fn, getattr(load_library(), fn)(
        _address(k, "k"), _address(v, "v"), _DTYPES[k.dtype], _ptr(slot_mapping), T,
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), ctypes.byref(layout),
        _stream(stream)))


def pkv_append_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                   v_scale: torch.Tensor, stream=None) -> None:
    """Quantise k[i], v[i] ([T, Hkv, D], fp32/fp16/bf16) into the FP8 pools (uint8
    codes [NB, Hkv, bs, D], float32 row scales [NB, Hkv, bs]) at slot_mapping[i]."""
    _append_q8("pkv_append_fp8", torch.uint8, k, v, slot_mapping, k_cache, v_cache, k_scale,
               v_scale, stream)


def pkv_append_int8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                    k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor,
                    v_scale: torch.Tensor, stream=None) -> None:
    """Quantise k[i], v[i] ([T, Hkv, D], fp32/fp16/bf16) into the INT8 pools (int8
    codes [NB, Hkv, bs, D], float32 row scales [NB, Hkv, bs]) at slot_mapping[i]."""
    _append_q8("pkv_append_int8", torch.int8, k, v, slot_mapping, k_cache, v_cache, k_scale,
               v_scale, stream)


def pkv_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_q: torch.Tensor,
                k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                context_lens: torch.Tensor, window: int, scale: float, max_chunk: int,
                out: torch.Tensor | None = None, stream=None,
                num_sinks: int = 0) -> torch.Tensor:
    """Append each sequence's chunk (packed q/k/v, offsets cu_q) and compute its
    causal (optionally windowed, with attention sinks) attention over the
    paged cache; returns out like q."""
    _on_cuda(q, k, v, cu_q, k_cache, v_cache, block_tables, context_lens, out)
    layout = cache_layout(k_cache)
    _require(v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype
             and v_cache.is_contiguous(), "v_cache must match k_cache")
    T = q.shape[0]
    _require(q.dim() == 3 and q.shape[2] == layout.head_dim and q.dtype == k_cache.dtype
             and q.is_contiguous(), "q must be contiguous [T, Hq, D] of the cache dtype")
    shape = (T, layout.num_kv_heads, layout.head_dim)
    _require(tuple(k.shape) == shape and tuple(v.shape) == shape and k.dtype == q.dtype
             and v.dtype == q.dtype and k.is_contiguous() and v.is_contiguous(),
             f"k and v must be contiguous {shape}")
    B = block_tables.shape[0]
    _require(cu_q.dtype == torch.int32 and cu_q.numel() == B + 1 and cu_q.is_contiguous(),
             "cu_q must be int32 [B + 1]")
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2
             and block_tables.is_contiguous(), "block_tables must be contiguous int32 [B, MB]")
    _require(context_lens.dtype == torch.int32 and context_lens.numel() == B
             and context_lens.is_contiguous(), "context_lens must be int32 [B]")
    if out is None:
        out = torch.empty_like(q)
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(),
             "out must be contiguous and shaped like q")
    _check("pkv_prefill", load_library().pkv_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_q), B, q.shape[1], int(max_chunk), _ptr(k_cache),
        _ptr(v_cache), ctypes.byref(layout), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), int(window), int(num_sinks), float(scale), _ptr(out),
        _stream(stream)))
    return out


def pkv_append_decode(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, window: int, scale: float,
                      out: torch.Tensor | None = None, tokens_per_split: int = 0,
                      stream=None, num_sinks: int = 0) -> torch.Tensor:
    """Append each sequence's new token (at position context_lens[b] - 1) and
    decode, in one launch; same result as the separate calls.  ``q``, ``k_new``,
    ``v_new`` and ``out`` may be pinned host tensors, as for ``pkv_decode``."""
    _on_cuda(k_cache, v_cache, block_tables, context_lens)
    layout = cache_layout(k_cache)
    _require(v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype
             and v_cache.is_contiguous(), "v_cache must match k_cache")
    _require(q.dim() == 3 and q.shape[2] == layout.head_dim and q.is_contiguous()
             and q.dtype == k_cache.dtype, "q must be contiguous [B, Hq, D] of the cache dtype")
    B, Hq, D = q.shape
    shape = (B, layout.num_kv_heads, layout.head_dim)
    _require(tuple(k_new.shape) == shape and tuple(v_new.shape) == shape
             and k_new.dtype == q.dtype and v_new.dtype == q.dtype
             and k_new.is_contiguous() and v_new.is_contiguous(),
             f"k_new and v_new must be contiguous {shape} of the cache dtype")
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2
             and block_tables.shape[0] == B and block_tables.is_contiguous(),
             "block_tables must be contiguous int32 [B, MB]")
    _require(context_lens.dtype == torch.int32 and context_lens.numel() == B
             and context_lens.is_contiguous(), "context_lens must be int32 [B]")
    if out is None:
        out = torch.empty_like(q, device=k_cache.device)
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(),
             "out must be contiguous and shaped like q")
    opts = DecodeOptions(int(window), int(num_sinks), int(tokens_per_split),
                         _address(k_new, "k_new"), _address(v_new, "v_new"), None, None)
    _check("pkv_append_decode", load_library().pkv_decode_ex(
        _address(q, "q"), B, Hq, _ptr(k_cache), _ptr(v_cache), ctypes.byref(layout),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), float(scale),
        _address(out, "out"), ctypes.byref(opts), _stream(stream)))
    return out


def pkv_decode_plan(num_seqs: int, num_q_heads: int, layout: CacheLayout, max_blocks: int,
                    window: int, tokens_per_split: int = 0, num_sms: int = 0,
                    num_sinks: int = 0):
    """(tokens_per_split, num_splits) the library would use; host only."""
    tps, ns = ctypes.c_int32(0), ctypes.c_int32(0)
    _check("pkv_decode_plan", load_library().pkv_decode_plan(
        num_seqs, num_q_heads, ctypes.byref(layout), max_blocks, window, num_sinks,
        tokens_per_split, num_sms, ctypes.byref(tps), ctypes.byref(ns)))
    return tps.value, ns.value


INDEX_CHECKS = {1: "context_length", 2: "block_table_entry", 3: "slot", 4: "duplicate_slot"}


def pkv_validate_indices(block_tables, context_lens, num_blocks: int, block_size: int,
                         slot_mapping=None, stream=None):
    """Debug check of the indices the other calls trust (waits for the stream).

    Returns None when every index is in range, else (check, row, col, value)
    for the first failure: check is "context_length" (row = sequence),
    "block_table_entry" (row, col = sequence, block), "slot" (row = token) or
    "duplicate_slot" (row = token, col = the earlier token with that slot).
    """
    for t, dt, what in ((block_tables, torch.int32, "block_tables"),
                        (context_lens, torch.int32, "context_lens")):
        _require(t.dtype == dt and t.is_contiguous(), f"{what} must be contiguous {dt}")
    _require(block_tables.dim() == 2 and context_lens.numel() == block_tables.shape[0],
             "block_tables [B, MB] and context_lens [B]")
    if slot_mapping is not None:
        _require(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous(),
                 "slot_mapping must be contiguous int64")
    err = IndexErrorInfo()
    rc = load_library().pkv_validate_indices(
        _ptr(block_tables), block_tables.shape[0], block_tables.shape[1], _ptr(context_lens),
        _ptr(slot_mapping), 0 if slot_mapping is None else slot_mapping.numel(), num_blocks,
        block_size, _stream(stream), ctypes.byref(err))
    if rc == PKV_ERR_RANGE:
        return INDEX_CHECKS[err.what], err.row, err.col, err.value
    _check("pkv_validate_indices", rc)
    return None


def pkv_release_workspaces() -> None:
    _check("pkv_release_workspaces", load_library().pkv_release_workspaces())
