"""Float64 CPU oracle for paged-KV decode attention and the slot-mapping append.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this package.  The
product (``paged_kv_cache_24_gb300``) never imports it, and this package never
imports the product: the two share no code.

The arithmetic lives in ``pkv_oracle.c`` (plain C, double precision, libm
``exp``), written from the pages' statement of the method:

* "Build a Paged KV Cache in Pure Python", Step 3 (``PagedKVCache.append`` and
  ``retrieve``) and Step 4 (``scaled_dot_product_attention``);
* "Building a Streaming Sliding-Window Attention Engine in Pure Python",
  Step 3 (``sliding_window_attention``: attend over ``[max(0, T - w), T)``)
  and the StreamingLLM item of its "Extending" list (attention sinks: the
  first tokens are kept regardless of the window).

This module only marshals numpy / torch-CPU arrays into that library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32, F16, BF16 = 0, 1, 2
_ELEM_BYTES = {F32: 4, F16: 2, BF16: 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-Wall", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        # a host without libgomp still gets a (single-threaded) oracle
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_i32, c_i64, c_dbl, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_f16_to_double.restype = c_dbl
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = c_dbl
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_elements.restype = None
        lib.oracle_decode_elements.argtypes = [c_vp, c_i64, c_i32, c_vp]
        lib.oracle_slot_for_position.restype = c_i64
        lib.oracle_slot_for_position.argtypes = [c_vp, c_i32, c_i32, c_i64]
        lib.oracle_append.restype = ctypes.c_int
        lib.oracle_append.argtypes = [c_vp, c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i32, c_i32,
                                      c_i32, c_i32]
        lib.oracle_attend.restype = None
        lib.oracle_attend.argtypes = [c_vp, c_vp, c_vp, c_i64, c_i32, c_dbl, c_vp]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [c_vp, c_i32, c_i32, c_vp, c_vp, c_i64, c_i32, c_i32, c_i32,
                                      c_i32, c_vp, c_i32, c_vp, c_i32, c_i32, c_dbl, c_vp, c_i64,
                                      c_vp, c_i32]
        lib.oracle_e4m3_to_double.restype = c_dbl
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_encode_e4m3.restype = None
        lib.oracle_encode_e4m3.argtypes = [c_vp, c_i64, c_vp]
        lib.oracle_quantize_row.restype = ctypes.c_float
        lib.oracle_quantize_row.argtypes = [c_vp, c_i32, c_vp]
        lib.oracle_append_fp8.restype = ctypes.c_int
        lib.oracle_append_fp8.argtypes = [c_vp, c_vp, c_i32, c_vp, c_i64, c_vp, c_vp, c_vp, c_vp,
                                          c_i64, c_i32, c_i32, c_i32]
        lib.oracle_decode_fp8.restype = ctypes.c_int
        lib.oracle_decode_fp8.argtypes = [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp,
                                          c_i64, c_i32, c_i32, c_i32, c_vp, c_i32, c_vp, c_i32,
                                          c_i32, c_dbl, c_vp, c_i64, c_vp, c_i32]
        lib.oracle_quantize_row_int8.restype = ctypes.c_float
        lib.oracle_quantize_row_int8.argtypes = [c_vp, c_i32, c_vp]
        lib.oracle_append_int8.restype = ctypes.c_int
        lib.oracle_append_int8.argtypes = lib.oracle_append_fp8.argtypes
        lib.oracle_decode_int8.restype = ctypes.c_int
        lib.oracle_decode_int8.argtypes = lib.oracle_decode_fp8.argtypes
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_prefill.argtypes = [c_vp, c_i32, c_vp, c_i32, c_i32, c_vp, c_vp, c_i64, c_i32,
                                       c_i32, c_i32, c_vp, c_i32, c_vp, c_i32, c_i32, c_dbl, c_vp,
                                       c_i32]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# array marshalling (raw bits in, doubles out)


def _as_raw(x):
    """(numpy array of the raw element bits, dtype code) for a numpy or torch-CPU array."""
    mod = type(x).__module__
    if mod.startswith("torch"):
        import torch  # local: torch is only needed when torch tensors are passed

        if x.device.type != "cpu":
            raise ValueError("oracle inputs must live in host memory")
        x = x.contiguous()
        if x.dtype == torch.float32:
            return x.numpy(), F32
        if x.dtype == torch.float16:
            return x.view(torch.int16).numpy().view(np.uint16), F16
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        raise TypeError(f"unsupported oracle dtype {x.dtype}")
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float16:
        return x.view(np.uint16), F16
    raise TypeError(f"unsupported oracle dtype {x.dtype} (pass bf16 as a torch tensor)")


def _int_array(x, dtype):
    mod = type(x).__module__
    if mod.startswith("torch"):
        x = x.cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=dtype))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def decode_elements(bits: np.ndarray, dtype_code: int) -> np.ndarray:
    """Widen raw fp32 / fp16 / bf16 element bits to float64 with the oracle's decoder."""
    raw = np.ascontiguousarray(bits)
    out = np.empty(raw.size, dtype=np.float64)
    _load().oracle_decode_elements(_ptr(raw), raw.size, dtype_code, _ptr(out))
    return out.reshape(raw.shape)


def slot_for_position(block_table_row, block_size: int, pos: int) -> int:
    """Slot of logical position ``pos`` in a sequence with the given block list (-1 if none)."""
    row = _int_array(block_table_row, np.int32)
    return int(_load().oracle_slot_for_position(_ptr(row), row.size, block_size, pos))


def slot_mapping(block_tables, positions, block_size: int) -> np.ndarray:
    """Slots for each sequence's new token at ``positions[b]`` (int64, -1 for none)."""
    bt = _int_array(block_tables, np.int32)
    pos = _int_array(positions, np.int64)
    return np.array([slot_for_position(bt[b], block_size, int(pos[b])) for b in range(bt.shape[0])],
                    dtype=np.int64)


def append(k, v, slot_mapping_, k_cache, v_cache) -> None:
    """Write each token's K/V rows into its slot, in place on host arrays.

    ``k``, ``v``: [T, Hkv, D]; ``k_cache``, ``v_cache``: [NB, Hkv, bs, D] (numpy or
    torch-CPU, modified in place); ``slot_mapping_``: [T] int64, negative = skip.
    """
    kr, kd = _as_raw(k)
    vr, vd = _as_raw(v)
    if kd != vd:
        raise TypeError("k and v dtypes differ")
    for c in (k_cache, v_cache):
        contiguous = c.is_contiguous() if hasattr(c, "is_contiguous") else c.flags.c_contiguous
        if not contiguous:
            raise ValueError("caches must be contiguous so they can be written in place")
    kc, kcd = _as_raw(k_cache)
    vc, vcd = _as_raw(v_cache)
    if kcd != kd or vcd != kd:
        raise TypeError("cache dtype differs from k/v dtype")
    slots = _int_array(slot_mapping_, np.int64)
    nb, hkv, bs, d = kc.shape
    rc = _load().oracle_append(_ptr(kr), _ptr(vr), _ptr(slots), slots.size, _ptr(kc), _ptr(vc),
                               nb, hkv, bs, d, _ELEM_BYTES[kd])
    if rc != 0:
        raise ValueError(f"oracle_append failed with code {rc}")


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of one query [D] over a contiguous cache K, V [T, D] (float64)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    out = np.empty(q.shape[0], dtype=np.float64)
    _load().oracle_attend(_ptr(q), _ptr(K), _ptr(V), K.shape[0], q.shape[0], float(scale),
                          _ptr(out))
    return out


def decode(q, k_cache, v_cache, block_tables, context_lens, window: int, scale: float,
           pairs=None, threads: int = 0, check: bool = True, num_sinks: int = 0) -> np.ndarray:
    """Paged decode attention in float64.

    ``q`` [B, Hq, D]; caches [NB, Hkv, bs, D]; ``block_tables`` [B, MB] int32;
    ``context_lens`` [B] int32 (after the append); ``window`` <= 0 for none;
    ``num_sinks``: with a window, positions [0, num_sinks) are attended too.
    ``scale`` is used exactly as given (pass the float32 value the GPU sees).
    ``pairs``: optional [n, 2] array of (b, h); returns [n, D], else [B, Hq, D].
    """
    qr, qd = _as_raw(q)
    kc, kd = _as_raw(k_cache)
    vc, vd = _as_raw(v_cache)
    if not (qd == kd == vd):
        raise TypeError("q, k_cache and v_cache must share a dtype")
    bt = _int_array(block_tables, np.int32)
    lens = _int_array(context_lens, np.int32)
    B, Hq, D = qr.shape
    nb, hkv, bs, d2 = kc.shape
    if d2 != D:
        raise ValueError("head_dim mismatch")
    if pairs is None:
        pairs_arr = None
        n = B * Hq
    else:
        pairs_arr = _int_array(pairs, np.int32).reshape(-1, 2)
        n = pairs_arr.shape[0]
        if n == 0:
            return np.empty((0, D), dtype=np.float64)
    out = np.empty((n, D), dtype=np.float64)
    rc = _load().oracle_decode(_ptr(qr), B, Hq, _ptr(kc), _ptr(vc), nb, hkv, bs, D, qd,
                               _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0, _ptr(lens),
                               int(window), int(num_sinks), float(scale),
                               None if pairs_arr is None else _ptr(pairs_arr), n, _ptr(out),
                               int(threads))
    if check and rc != 0:
        raise ValueError(f"oracle_decode failed with code {rc}")
    return out if pairs is not None else out.reshape(B, Hq, D)


# ---------------------------------------------------------------------------
# FP8 (E4M3) cache: codes + one float32 scale per (token, kv head) row


F8 = 3


def _u8(x):
    if type(x).__module__.startswith("torch"):
        import torch
        x = x.contiguous()
        if x.dtype != torch.uint8:
            x = x.view(torch.uint8)
        return x.numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint8:
        raise TypeError("FP8 codes must be uint8")
    return x


def _f32(x):
    if type(x).__module__.startswith("torch"):
        x = x.contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("expected float32")
    return x


def e4m3_to_double(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8 array) in float64."""
    return decode_elements(_u8(codes), F8)


def encode_e4m3(x) -> np.ndarray:
    """Nearest E4M3 code (ties to even, saturating) of each float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_encode_e4m3(_ptr(x), x.size, _ptr(out))
    return out


def quantize_rows(x):
    """Quantise each row of a float32 matrix [n, D]: (codes uint8 [n, D], scales float32 [n])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n, d = x.shape
    codes = np.empty((n, d), dtype=np.uint8)
    scales = np.empty(n, dtype=np.float32)
    lib = _load()
    for i in range(n):
        scales[i] = lib.oracle_quantize_row(_ptr(x[i]), d, codes[i].ctypes.data)
    return codes, scales


def append_fp8(k, v, slot_mapping_, k_codes, v_codes, k_scale, v_scale) -> None:
    """Quantise and write each token's K/V rows ([T, Hkv, D], fp16/bf16/fp32) into
    FP8 pools ([NB, Hkv, bs, D] uint8 codes, [NB, Hkv, bs] float32 scales), in place."""
    kr, kd = _as_raw(k)
    vr, vd = _as_raw(v)
    if kd != vd:
        raise TypeError("k and v dtypes differ")
    for c in (k_codes, v_codes, k_scale, v_scale):
        contiguous = c.is_contiguous() if hasattr(c, "is_contiguous") else c.flags.c_contiguous
        if not contiguous:
            raise ValueError("pools must be contiguous so they can be written in place")
    kc, vc = _u8(k_codes), _u8(v_codes)
    ks, vs = _f32(k_scale), _f32(v_scale)
    slots = _int_array(slot_mapping_, np.int64)
    nb, hkv, bs, d = kc.shape
    rc = _load().oracle_append_fp8(_ptr(kr), _ptr(vr), kd, _ptr(slots), slots.size, _ptr(kc),
                                   _ptr(vc), _ptr(ks), _ptr(vs), nb, hkv, bs, d)
    if rc != 0:
        raise ValueError(f"oracle_append_fp8 failed with code {rc}")


def _codes8(x):
    """Raw bytes of an FP8 or INT8 code array (torch or numpy), sharing memory."""
    if type(x).__module__.startswith("torch"):
        import torch
        x = x.contiguous()
        return x.view(torch.uint8).numpy() if x.dtype != torch.uint8 else x.numpy()
    x = np.ascontiguousarray(x)
    if x.dtype not in (np.uint8, np.int8):
        raise TypeError("codes must be uint8 or int8")
    return x.view(np.uint8)


def quantize_rows_int8(x):
    """INT8-quantise each row of a float32 matrix [n, D]: (codes int8 [n, D], scales float32 [n])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n, d = x.shape
    codes = np.empty((n, d), dtype=np.int8)
    scales = np.empty(n, dtype=np.float32)
    lib = _load()
    for i in range(n):
        scales[i] = lib.oracle_quantize_row_int8(_ptr(x[i]), d, codes[i].ctypes.data)
    return codes, scales


def append_int8(k, v, slot_mapping_, k_codes, v_codes, k_scale, v_scale) -> None:
    """Quantise and write each token's K/V rows ([T, Hkv, D], fp16/bf16/fp32) into
    INT8 pools ([NB, Hkv, bs, D] int8 codes, [NB, Hkv, bs] float32 scales), in place."""
    kr, kd = _as_raw(k)
    vr, vd = _as_raw(v)
    if kd != vd:
        raise TypeError("k and v dtypes differ")
    for c in (k_codes, v_codes, k_scale, v_scale):
        contiguous = c.is_contiguous() if hasattr(c, "is_contiguous") else c.flags.c_contiguous
        if not contiguous:
            raise ValueError("pools must be contiguous so they can be written in place")
    kc, vc = _codes8(k_codes), _codes8(v_codes)
    ks, vs = _f32(k_scale), _f32(v_scale)
    slots = _int_array(slot_mapping_, np.int64)
    nb, hkv, bs, d = kc.shape
    rc = _load().oracle_append_int8(_ptr(kr), _ptr(vr), kd, _ptr(slots), slots.size, _ptr(kc),
                                    _ptr(vc), _ptr(ks), _ptr(vs), nb, hkv, bs, d)
    if rc != 0:
        raise ValueError(f"oracle_append_int8 failed with code {rc}")


def decode_int8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, window: int,
                scale: float, pairs=None, threads: int = 0, check: bool = True,
                num_sinks: int = 0) -> np.ndarray:
    """Paged decode over INT8 pools (stored value = code * row scale), in float64."""
    return _decode_codes("oracle_decode_int8", q, _codes8(k_codes), _codes8(v_codes), k_scale,
                         v_scale, block_tables, context_lens, window, scale, pairs, threads,
                         check, num_sinks)


def _decode_codes(fn, q, kc, vc, k_scale, v_scale, block_tables, context_lens, window, scale,
                  pairs, threads, check, num_sinks):
    qr, qd = _as_raw(q)
    ks, vs = _f32(k_scale), _f32(v_scale)
    bt = _int_array(block_tables, np.int32)
    lens = _int_array(context_lens, np.int32)
    B, Hq, D = qr.shape
    nb, hkv, bs, d2 = kc.shape
    if d2 != D:
        raise ValueError("head_dim mismatch")
    if pairs is None:
        pairs_arr, n = None, B * Hq
    else:
        pairs_arr = _int_array(pairs, np.int32).reshape(-1, 2)
        n = pairs_arr.shape[0]
        if n == 0:
            return np.empty((0, D), dtype=np.float64)
    out = np.empty((n, D), dtype=np.float64)
    rc = getattr(_load(), fn)(_ptr(qr), qd, B, Hq, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                              nb, hkv, bs, D, _ptr(bt), bt.shape[1], _ptr(lens), int(window),
                              int(num_sinks), float(scale),
                              None if pairs_arr is None else _ptr(pairs_arr), n, _ptr(out),
                              int(threads))
    if check and rc != 0:
        raise ValueError(f"{fn} failed with code {rc}")
    return out if pairs is not None else out.reshape(B, Hq, D)


def decode_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, window: int,
               scale: float, pairs=None, threads: int = 0, check: bool = True,
               num_sinks: int = 0) -> np.ndarray:
    """Paged decode over FP8 pools (stored value = code * row scale), in float64."""
    qr, qd = _as_raw(q)
    kc, vc = _u8(k_codes), _u8(v_codes)
    ks, vs = _f32(k_scale), _f32(v_scale)
    bt = _int_array(block_tables, np.int32)
    lens = _int_array(context_lens, np.int32)
    B, Hq, D = qr.shape
    nb, hkv, bs, d2 = kc.shape
    if d2 != D:
        raise ValueError("head_dim mismatch")
    if pairs is None:
        pairs_arr, n = None, B * Hq
    else:
        pairs_arr = _int_array(pairs, np.int32).reshape(-1, 2)
        n = pairs_arr.shape[0]
        if n == 0:
            return np.empty((0, D), dtype=np.float64)
    out = np.empty((n, D), dtype=np.float64)
    rc = _load().oracle_decode_fp8(_ptr(qr), qd, B, Hq, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                                   nb, hkv, bs, D, _ptr(bt), bt.shape[1], _ptr(lens),
                                   int(window), int(num_sinks), float(scale),
                                   None if pairs_arr is None else _ptr(pairs_arr), n, _ptr(out),
                                   int(threads))
    if check and rc != 0:
        raise ValueError(f"oracle_decode_fp8 failed with code {rc}")
    return out if pairs is not None else out.reshape(B, Hq, D)


def prefill(q, cu_q, k_cache, v_cache, block_tables, context_lens, window: int, scale: float,
            threads: int = 0, check: bool = True, num_sinks: int = 0) -> np.ndarray:
    """Chunked prefill over a paged cache (chunk already appended), float64.

    ``q`` [T, Hq, D] packed chunk queries; ``cu_q`` [B + 1] chunk offsets;
    ``context_lens`` [B] lengths including the chunk.  Query token at position
    p attends positions j <= p with p - j < window when window > 0, and, with a
    window, also the positions j < num_sinks (attention sinks).
    Returns [T, Hq, D]."""
    qr, qd = _as_raw(q)
    kc, kd = _as_raw(k_cache)
    vc, vd = _as_raw(v_cache)
    if not (qd == kd == vd):
        raise TypeError("q, k_cache and v_cache must share a dtype")
    cu = _int_array(cu_q, np.int32)
    bt = _int_array(block_tables, np.int32)
    lens = _int_array(context_lens, np.int32)
    T, Hq, D = qr.shape
    nb, hkv, bs, d2 = kc.shape
    out = np.empty((T, Hq, D), dtype=np.float64)
    rc = _load().oracle_prefill(_ptr(qr), qd, _ptr(cu), len(cu) - 1, Hq, _ptr(kc), _ptr(vc), nb,
                                hkv, bs, D, _ptr(bt), bt.shape[1], _ptr(lens), int(window),
                                int(num_sinks), float(scale), _ptr(out), int(threads))
    if check and rc != 0:
        raise ValueError(f"oracle_prefill failed with code {rc}")
    return out
