"""pkv_decode_noalloc: decode without any device allocation at call time.

Some callers cannot let a library call cudaMalloc: a serving engine that has
already handed all free HBM to its own KV-block pool, or a hot loop that must
not run into the device-wide synchronisation cudaMalloc / cudaFree can bring.
pkv_decode_noalloc serves them with a fixed scratch buffer that lives in the
library image.  These checks call it through the C ABI, on two calls in a
row (the second call runs over the first call's leftovers in the shared
buffer), with the device's free memory unchanged across them, and compare
its outputs with the float64 oracle and with pkv_decode, the entry point
that allocates its workspace.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

pytestmark = pytest.mark.gpu

PKV_ERR_SCRATCH = 8
TOL = {torch.float16: 2e-3, torch.bfloat16: 2e-3, torch.float32: 1e-5}


def _noalloc_fn(pkv):
    lib = pkv.load_library()
    fn = lib.pkv_decode_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [vp, i32, i32, vp, vp, ctypes.POINTER(pkv.CacheLayout), vp, i32, vp, i32,
                   ctypes.c_float, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(pkv, fn, q, kc, vc, bt, lens, window, scale, out, stream=None):
    layout = pkv.cache_layout(kc)
    st = (stream or torch.cuda.current_stream()).cuda_stream
    return fn(q.data_ptr(), q.shape[0], q.shape[1], kc.data_ptr(), vc.data_ptr(),
              ctypes.byref(layout), bt.data_ptr(), bt.shape[1], lens.data_ptr(), window,
              scale, out.data_ptr(), st)


def _close(a, b, dtype):
    a, b = a.double(), b.double()
    tol = TOL[dtype] + 0.5 * torch.finfo(dtype).eps * b.abs()
    assert torch.isfinite(a).all()
    assert ((a - b).abs() <= tol).all(), f"max diff {(a - b).abs().max().item():.3e}"


@pytest.mark.parametrize("dtype,window", [(torch.bfloat16, 0), (torch.float16, 4500),
                                          (torch.float32, 0)])
def test_noalloc_matches_allocating_decode_twice(pkv_lib, oracle_lib, dtype, window):
    """Two no-alloc calls in a row on a stream no allocating call has used,
    with the device's free memory unchanged across them; each output is
    compared with the float64 oracle and with pkv_decode's."""
    pkv = pkv_lib
    fn = _noalloc_fn(pkv)
    spec = config_spec(0, dtype=dtype, num_seqs=6, num_q_heads=16, num_kv_heads=4,
                       head_dim=128, block_size=16, lens=[1, 40, 700, 1500, 2600, 5000],
                       explicit_pool=None, lens_are_pre_append=False, window=window)
    w = make_workload(spec, device="cuda", poison=True)
    plan = pkv.pkv_decode_plan(spec.num_seqs, spec.num_q_heads, pkv.cache_layout(w.k_cache),
                               w.max_blocks, window)
    assert plan[1] > 1, "the case must use the split-K scratch"
    slots = pkv.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(), 16)
    pkv.pkv_append(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache)
    lens = w.lens_steps[0].contiguous()
    # the second call uses other queries and shorter contexts, over what the
    # first call left in the shared scratch
    qs = [w.q_steps[0], torch.flip(w.q_steps[0], dims=[0]).contiguous()]
    lns = [lens, torch.clamp(lens - 17, min=0).contiguous()]
    outs = [torch.full_like(q, float("nan")) for q in qs]
    warm_out = torch.full_like(qs[0], float("nan"))
    side, fresh = torch.cuda.Stream(), torch.cuda.Stream()
    # once on a side stream first: loads the kernels' code and looks up the
    # scratch buffer's address (the one-time set-up of the first call)
    with torch.cuda.stream(side):
        rc = _call_noalloc(pkv, fn, qs[1], w.k_cache, w.v_cache, w.block_tables, lns[1],
                           window, w.scale, warm_out, stream=side)
    assert rc == 0, pkv.status_string(rc)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for q, ln, out in zip(qs, lns, outs):
        rc = _call_noalloc(pkv, fn, q, w.k_cache, w.v_cache, w.block_tables, ln, window,
                           w.scale, out, stream=fresh)
        assert rc == 0, pkv.status_string(rc)
    fresh.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory was allocated"

    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    bt_h = w.block_tables.cpu().numpy()
    for q, ln, out in zip(qs, lns, outs):
        ref_oracle = oracle.decode(q.cpu(), kc_h, vc_h, bt_h, ln.cpu().numpy(), window, w.scale)
        _close(out.cpu(), torch.from_numpy(ref_oracle), dtype)
        ref = pkv.pkv_decode(q, w.k_cache, w.v_cache, w.block_tables, ln, window, w.scale)
        torch.cuda.synchronize()
        _close(out, ref, dtype)


def test_noalloc_rejects_problems_beyond_its_scratch(pkv_lib):
    pkv = pkv_lib
    fn = _noalloc_fn(pkv)
    B, hq, hkv, d, bs, mb = 1024, 32, 8, 128, 16, 300
    q = torch.zeros(B, hq, d, dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    kc = torch.zeros(4, hkv, bs, d, dtype=torch.float16, device="cuda")
    bt = torch.zeros(B, mb, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    tps, ns = pkv.pkv_decode_plan(B, hq, pkv.cache_layout(kc), mb, 0)
    need = B * hq * ns * (d * 4 + 8)
    assert need > 32 * 1024 * 1024
    rc = _call_noalloc(pkv, fn, q, kc, kc, bt, lens, 0, 0.1, out)
    assert rc == PKV_ERR_SCRATCH
    assert "scratch" in pkv.status_string(rc)


def _noalloc_ex(pkv):
    lib = pkv.load_library()
    fn = lib.pkv_decode_noalloc_ex
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [vp, i32, i32, vp, vp, ctypes.POINTER(pkv.CacheLayout), vp, i32, vp,
                   ctypes.c_float, vp, ctypes.POINTER(pkv.DecodeOptions), vp]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.parametrize("kind", ["sinks_window", "fused_append", "fp8", "int8"])
def test_noalloc_ex_matches_decode_ex_bit_for_bit(pkv_lib, oracle_lib, kind):
    """The options form runs the same plan and kernels as pkv_decode_ex, only
    with the library's scratch: the outputs (and pools) agree bit for bit."""
    pkv = pkv_lib
    fn = _noalloc_ex(pkv)
    q8 = kind in ("fp8", "int8")
    spec = config_spec(0, dtype=torch.float16, num_seqs=5, num_q_heads=16, num_kv_heads=4,
                       head_dim=128, block_size=16, lens=[1, 60, 900, 2500, 4100],
                       explicit_pool=None, lens_are_pre_append=False,
                       window=700 if kind == "sinks_window" else 0,
                       num_sinks=5 if kind == "sinks_window" else 0,
                       kv_fp8=kind == "fp8", kv_int8=kind == "int8")
    outs, pools = [], []
    for noalloc in (False, True):
        w = make_workload(spec, device="cuda", poison=True)
        lens = w.lens_steps[0].contiguous()
        fused = kind == "fused_append"
        if not fused:
            slots = pkv.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(), 16)
            if q8:
                app = pkv.pkv_append_fp8 if kind == "fp8" else pkv.pkv_append_int8
                app(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache, w.k_scale,
                    w.v_scale)
            else:
                pkv.pkv_append(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache)
        opts = pkv.DecodeOptions(spec.window, spec.num_sinks, 512,
                                 w.k_steps[0].data_ptr() if fused else None,
                                 w.v_steps[0].data_ptr() if fused else None,
                                 w.k_scale.data_ptr() if q8 else None,
                                 w.v_scale.data_ptr() if q8 else None)
        out = torch.full_like(w.q_steps[0], float("nan"))
        layout = pkv.cache_layout(w.k_cache)
        call = fn if noalloc else pkv.load_library().pkv_decode_ex
        rc = call(w.q_steps[0].data_ptr(), spec.num_seqs, spec.num_q_heads,
                  w.k_cache.data_ptr(), w.v_cache.data_ptr(), ctypes.byref(layout),
                  w.block_tables.data_ptr(), w.block_tables.shape[1], lens.data_ptr(),
                  ctypes.c_float(w.scale), out.data_ptr(), ctypes.byref(opts),
                  torch.cuda.current_stream().cuda_stream)
        assert rc == 0, pkv.status_string(rc)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        outs.append(out.cpu())
        pools.append((w.k_cache.cpu(), w.v_cache.cpu()))
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    for a, b in zip(pools[0], pools[1]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
