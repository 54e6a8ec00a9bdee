"""The C ABI on the host: every declared symbol is exported, and argument checks
return their status codes before anything touches a GPU."""
import ctypes
import os
import re

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(REPO, "include", "pkv.h")

OK, NULL, SHAPE, DTYPE, UNSUP, ALIGN = 0, 1, 2, 3, 4, 5


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pkv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_two_calls_of_the_method():
    names = declared_functions()
    assert "pkv_append" in names and "pkv_decode" in names


def test_library_exports_every_declared_symbol(pkv_lib):
    lib = ctypes.CDLL(pkv_lib.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings(pkv_lib):
    for code in range(10):
        assert pkv_lib.status_string(code).startswith("PKV_")
    assert "unknown" in pkv_lib.status_string(99)


def _layout(pkv, nb=64, hkv=8, bs=16, d=128, dt=1):
    return pkv.CacheLayout(nb, hkv, bs, d, dt)


FAKE = 0x100000  # a 16-byte aligned address that is never dereferenced


def _decode(pkv, layout, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, lens=FAKE, out=FAKE, B=4, hq=32,
            mb=8, window=0, tps=0):
    lib = pkv.load_library()
    return lib.pkv_decode_split(q, B, hq, k, v, ctypes.byref(layout), bt, mb, lens, window,
                                0.1, out, tps, None)


def test_decode_argument_checks(pkv_lib):
    pkv = pkv_lib
    assert _decode(pkv, _layout(pkv), q=0) == NULL
    assert _decode(pkv, _layout(pkv), out=0) == NULL
    assert _decode(pkv, _layout(pkv, dt=7)) == DTYPE
    assert _decode(pkv, _layout(pkv, d=96)) == UNSUP
    assert _decode(pkv, _layout(pkv, bs=8)) == UNSUP
    assert _decode(pkv, _layout(pkv, bs=24)) == UNSUP
    assert _decode(pkv, _layout(pkv), hq=12) == SHAPE           # 12 % 8 != 0
    assert _decode(pkv, _layout(pkv), B=-1) == SHAPE
    assert _decode(pkv, _layout(pkv, hkv=0)) == SHAPE
    assert _decode(pkv, _layout(pkv), q=FAKE + 8) == ALIGN
    assert _decode(pkv, _layout(pkv), lens=FAKE + 2) == ALIGN
    assert _decode(pkv, _layout(pkv), tps=24) == SHAPE          # not a multiple of 16
    assert _decode(pkv, _layout(pkv), tps=65536 + 16) == UNSUP  # more than 65536 per split
    assert _decode(pkv, _layout(pkv, nb=1 << 30)) == UNSUP      # TMA rows exceed int32
    # nothing to do: succeeds without touching the device
    assert _decode(pkv, _layout(pkv), B=0, q=0, out=0) == OK


def test_append_argument_checks(pkv_lib):
    pkv = pkv_lib
    lib = pkv.load_library()
    lay = _layout(pkv)

    def call(k=FAKE, v=FAKE, slots=FAKE, n=3, kc=FAKE, vc=FAKE, layout=lay):
        return lib.pkv_append(k, v, slots, n, kc, vc, ctypes.byref(layout), None)

    assert call(k=0) == NULL
    assert call(slots=0) == NULL
    assert call(n=-1) == SHAPE
    assert call(n=0, k=0, v=0) == OK
    assert call(layout=_layout(pkv, dt=-1)) == DTYPE
    assert call(layout=_layout(pkv, d=4)) == UNSUP   # 4 fp16 = 8 bytes: not 16-byte rows
    assert call(v=FAKE + 4) == ALIGN
    assert call(slots=FAKE + 4) == ALIGN


def test_slot_mapping_argument_checks(pkv_lib):
    lib = pkv_lib.load_library()
    assert lib.pkv_slot_mapping(FAKE, 4, 8, FAKE, 0, FAKE, None) == SHAPE
    assert lib.pkv_slot_mapping(0, 4, 8, FAKE, 16, FAKE, None) == NULL
    assert lib.pkv_slot_mapping(FAKE, 4, 8, FAKE + 4, 16, FAKE, None) == ALIGN
    assert lib.pkv_slot_mapping(0, 0, 8, 0, 16, 0, None) == OK


@pytest.mark.parametrize("cfg,expect", [
    # (num_seqs, hq, layout args, max_blocks, window) -> (tokens_per_split, num_splits)
    ((64, 32, (10000, 32, 16, 128, 1), 256, 0), (2048, 2)),
    ((256, 32, (44000, 8, 32, 128, 2), 256, 0), (2048, 4)),
    # fewer items than SMs (16-bit, head_dim 128): one wave of at most one
    # CTA per SM -- 128 or 96 windows one split each, a single 4096-token
    # sequence's 8 items in 19 pieces each
    ((16, 32, (30000, 8, 16, 128, 2), 2048, 4096), (4112, 1)),
    ((12, 32, (30000, 8, 16, 128, 2), 2048, 4096), (4112, 1)),
    ((1, 32, (4096, 8, 16, 128, 1), 256, 0), (224, 19)),
    ((4, 32, (4096, 8, 16, 128, 1), 256, 0), (1024, 4)),
    # the same few items at head_dim 64 keep the 4-CTAs-per-SM splits
    ((1, 32, (4096, 8, 16, 64, 1), 256, 0), (128, 32)),
    ((16, 32, (30000, 8, 16, 128, 2), 2048, 4097), (4128, 1)),
    ((4, 8, (32, 8, 16, 64, 0), 7, 0), (128, 1)),
    ((1, 8, (4096, 8, 16, 128, 1), 2048, 0), (1728, 19)),
    # 32+ items per SM and at most 257 units each: one split per item
    ((1024, 32, (50000, 8, 16, 128, 1), 130, 0), (2080, 1)),
    ((1024, 32, (50000, 8, 16, 128, 1), 256, 0), (4096, 1)),
    ((1024, 32, (50000, 8, 16, 128, 1), 257, 0), (4112, 1)),
    ((1024, 32, (50000, 8, 16, 128, 1), 258, 0), (2048, 3)),
    ((600, 32, (50000, 8, 16, 128, 1), 130, 0), (2048, 2)),
])
def test_plan(pkv_lib, cfg, expect):
    B, hq, lay, mb, window = cfg
    assert pkv_lib.pkv_decode_plan(B, hq, pkv_lib.CacheLayout(*lay), mb, window,
                                   num_sms=152) == expect


def _units_needed(L, window, sinks):
    """Units a length-L context attends: the sink units, then the window units
    (one range from unit 0 when they meet)."""
    if L == 0:
        return 0
    lo = max(0, L - window) if window > 0 else 0
    s = min(sinks, lo) if window > 0 else 0
    su, wu0 = -(-s // 16), lo // 16
    if su >= wu0:
        su = wu0 = 0
    return su + (L + 15) // 16 - wu0


def test_plan_covers_every_length(pkv_lib):
    """The grid's split count bounds the splits any valid length needs."""
    lay = pkv_lib.CacheLayout(5000, 8, 32, 128, 2)
    for mb in (1, 3, 17, 64):
        for window in (0, 1, 15, 16, 17, 100, 4096):
            for sinks in (0, 4, 16, 40):
                for tps in (0, 16, 64, 2048):
                    t, ns = pkv_lib.pkv_decode_plan(8, 32, lay, mb, window, tps, num_sms=152,
                                                    num_sinks=sinks)
                    units = t // 16
                    worst = max(-(-_units_needed(L, window, sinks) // units)
                                for L in range(0, mb * 32 + 1))
                    assert worst <= ns


def test_quantised_pool_argument_checks(pkv_lib):
    """8-bit pools (FP8 = 3, INT8 = 4): decode only at head_dim 128 and with row
    scales, appends only into the matching code format, no fixed-scratch decode."""
    pkv = pkv_lib
    lib = pkv.load_library()
    for dt in (3, 4):
        assert _decode(pkv, _layout(pkv, dt=dt, d=64)) == UNSUP
        assert _decode(pkv, _layout(pkv, dt=dt)) == NULL         # no scales given
        vp = ctypes.c_void_p
        assert lib.pkv_decode_noalloc(vp(FAKE), 4, 32, vp(FAKE), vp(FAKE),
                                      ctypes.byref(_layout(pkv, dt=dt)), vp(FAKE), 8, vp(FAKE),
                                      0, ctypes.c_float(0.1), vp(FAKE), None) == UNSUP
        # the options form takes the scales; without them: NULL, before any CUDA call
        lib.pkv_decode_noalloc_ex.argtypes = [vp, ctypes.c_int32, ctypes.c_int32, vp, vp,
                                              ctypes.POINTER(pkv.CacheLayout), vp,
                                              ctypes.c_int32, vp, ctypes.c_float, vp,
                                              ctypes.POINTER(pkv.DecodeOptions), vp]
        opts = pkv.DecodeOptions(0, 0, 0, None, None, None, None)
        assert lib.pkv_decode_noalloc_ex(vp(FAKE), 4, 32, vp(FAKE), vp(FAKE),
                                         ctypes.byref(_layout(pkv, dt=dt)), vp(FAKE), 8,
                                         vp(FAKE), ctypes.c_float(0.1), vp(FAKE),
                                         ctypes.byref(opts), None) == NULL
        assert lib.pkv_decode_noalloc_ex(vp(FAKE), 4, 32, vp(FAKE), vp(FAKE),
                                         ctypes.byref(_layout(pkv, dt=dt)), vp(FAKE), 8,
                                         vp(FAKE), ctypes.c_float(0.1), vp(FAKE), None,
                                         None) == NULL

    def app(fn, dt, in_dtype=1, ks=FAKE, n=3):
        lay = _layout(pkv, dt=dt)
        return getattr(lib, fn)(FAKE, FAKE, in_dtype, FAKE, n, FAKE, FAKE, ks, FAKE,
                                ctypes.byref(lay), None)

    assert app("pkv_append_int8", 3) == DTYPE      # an FP8 pool
    assert app("pkv_append_fp8", 4) == DTYPE       # an INT8 pool
    assert app("pkv_append_int8", 1) == DTYPE      # a 16-bit pool
    assert app("pkv_append_int8", 4, in_dtype=3) == DTYPE
    assert app("pkv_append_int8", 4, ks=0) == NULL
    assert app("pkv_append_int8", 4, n=-1) == SHAPE
    assert app("pkv_append_int8", 4, n=0) == OK
    assert _decode(pkv, _layout(pkv, dt=5)) == DTYPE


def test_prefill_argument_checks(pkv_lib):
    """pkv_prefill rejects bad shapes before touching memory: 8-bit or fp32
    pools, a negative sink count, more than 65534 sequences; no sequences or an
    empty chunk is a no-op."""
    lib = pkv_lib.load_library()

    def call(dt=1, num_seqs=4, max_chunk=64, sinks=0, window=16):
        lay = _layout(pkv_lib, dt=dt)
        return lib.pkv_prefill(FAKE, FAKE, FAKE, FAKE, num_seqs, 32, max_chunk, FAKE, FAKE,
                               ctypes.byref(lay), FAKE, 8, FAKE, window, sinks,
                               ctypes.c_float(0.1), FAKE, None)

    assert call(dt=0) == UNSUP
    assert call(dt=3) == UNSUP
    assert call(dt=4) == UNSUP
    assert call(sinks=-1) == SHAPE
    assert call(num_seqs=-1) == SHAPE
    assert call(num_seqs=65535) == UNSUP
    assert call(num_seqs=0) == OK
    assert call(max_chunk=0) == OK


def test_stage_copy_argument_checks(pkv_lib):
    """pkv_stage_copy checks its arguments before any CUDA call."""
    lib = pkv_lib.load_library()
    assert lib.pkv_stage_copy(FAKE, FAKE, -1, None) == SHAPE
    assert lib.pkv_stage_copy(FAKE, FAKE, 0, None) == OK
    assert lib.pkv_stage_copy(None, FAKE, 64, None) == NULL
    assert lib.pkv_stage_copy(FAKE, None, 64, None) == NULL
    assert lib.pkv_stage_copy(FAKE + 8, FAKE, 64, None) == ALIGN
    assert lib.pkv_stage_copy(FAKE, FAKE + 4, 64, None) == ALIGN


def test_validate_indices_argument_checks(pkv_lib):
    """pkv_validate_indices checks sizes and pointers before copying anything."""
    lib = pkv_lib.load_library()
    err = pkv_lib._binding.IndexErrorInfo()
    ref = ctypes.byref(err)
    assert lib.pkv_validate_indices(None, 0, 0, None, None, 0, 0, 16, None, ref) == OK
    assert err.what == 0
    assert lib.pkv_validate_indices(None, 0, 4, None, None, 0, 10, 16, None, None) == OK
    assert lib.pkv_validate_indices(FAKE, -1, 4, FAKE, None, 0, 10, 16, None, ref) == SHAPE
    assert lib.pkv_validate_indices(FAKE, 2, -4, FAKE, None, 0, 10, 16, None, ref) == SHAPE
    assert lib.pkv_validate_indices(FAKE, 2, 4, FAKE, None, -3, 10, 16, None, ref) == SHAPE
    assert lib.pkv_validate_indices(FAKE, 2, 4, FAKE, None, 0, -1, 16, None, ref) == SHAPE
    assert lib.pkv_validate_indices(FAKE, 2, 4, FAKE, None, 0, 10, 0, None, ref) == SHAPE
    assert lib.pkv_validate_indices(None, 2, 4, FAKE, None, 0, 10, 16, None, ref) == NULL
    assert lib.pkv_validate_indices(FAKE, 2, 4, None, None, 0, 10, 16, None, ref) == NULL
    assert lib.pkv_validate_indices(None, 0, 4, None, None, 3, 10, 16, None, ref) == NULL
