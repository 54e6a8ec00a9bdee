"""The two calls the pages' statement of the problem names, driven through
the C ABI exactly as include/pkv.h declares them -- ``pkv_append(k, v,
slot_mapping, T, k_cache, v_cache, layout, stream)`` and ``pkv_decode(q, B,
Hq, k_cache, v_cache, layout, block_tables, MB, context_lens, window, scale,
out, stream)`` -- with no Python wrapper in between ("Build a Paged KV Cache in
Pure Python", Step 3 ``append`` and Step 4 ``scaled_dot_product_attention``).

The pool after the append must equal the oracle's bit for bit, and every
decode output must be within the oracle tolerance (2e-3 / 1e-5 plus half an
output ulp).  Each case is sized so the library's own plan splits the
contexts (split-K partials plus the log-sum-exp combine).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

pytestmark = pytest.mark.gpu

BASE = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 2e-3}

CASES = [
    # name, dtype, Hq, Hkv, D, bs, lens, window
    ("fp32_d128_g4", torch.float32, 8, 2, 128, 16, [1, 33, 700, 2100], 0),
    ("fp16_d128_mha", torch.float16, 4, 4, 128, 16, [5, 300, 1777, 4100], 0),
    ("bf16_d128_g4_window", torch.bfloat16, 16, 4, 128, 32, [2, 64, 999, 6000], 1500),
    ("bf16_d64_g8", torch.bfloat16, 16, 2, 64, 16, [17, 513, 3000], 0),
]


@pytest.mark.parametrize("name,dtype,hq,hkv,d,bs,lens,window", CASES, ids=[c[0] for c in CASES])
def test_plain_append_and_decode_symbols(pkv_lib, oracle_lib, name, dtype, hq, hkv, d, bs, lens,
                                         window):
    pkv = pkv_lib
    lib = pkv.load_library()
    spec = config_spec(0, dtype=dtype, num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv,
                       head_dim=d, block_size=bs, lens=lens, explicit_pool=None,
                       lens_are_pre_append=False, window=window, seed=len(name))
    w = make_workload(spec, device="cuda", poison_outside_window=True)
    layout = pkv.cache_layout(w.k_cache)
    tps, ns = pkv.pkv_decode_plan(spec.num_seqs, hq, layout, w.max_blocks, window)
    assert ns > 1, "the case must split its contexts"

    bt_h = w.block_tables.cpu().numpy()
    slots_h = oracle.slot_mapping(bt_h, w.pos_steps[0].cpu().numpy(), bs)
    slots = torch.from_numpy(slots_h).to("cuda")
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    oracle.append(w.k_steps[0].cpu(), w.v_steps[0].cpu(), slots_h, kc_h, vc_h)
    lens_d = w.lens_steps[0].contiguous()
    ref = oracle.decode(w.q_steps[0].cpu(), kc_h, vc_h, bt_h, lens_d.cpu().numpy(), window,
                        w.scale)

    stream = torch.cuda.current_stream().cuda_stream
    k, v, q = w.k_steps[0].contiguous(), w.v_steps[0].contiguous(), w.q_steps[0].contiguous()
    rc = lib.pkv_append(ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                        ctypes.c_void_p(slots.data_ptr()), ctypes.c_int64(spec.num_seqs),
                        ctypes.c_void_p(w.k_cache.data_ptr()),
                        ctypes.c_void_p(w.v_cache.data_ptr()), ctypes.byref(layout),
                        ctypes.c_void_p(stream))
    assert rc == 0, pkv.status_string(rc)
    out = torch.full_like(q, float("nan"))
    rc = lib.pkv_decode(ctypes.c_void_p(q.data_ptr()), ctypes.c_int32(spec.num_seqs),
                        ctypes.c_int32(hq), ctypes.c_void_p(w.k_cache.data_ptr()),
                        ctypes.c_void_p(w.v_cache.data_ptr()), ctypes.byref(layout),
                        ctypes.c_void_p(w.block_tables.data_ptr()),
                        ctypes.c_int32(w.block_tables.shape[1]),
                        ctypes.c_void_p(lens_d.data_ptr()), ctypes.c_int32(window),
                        ctypes.c_float(w.scale), ctypes.c_void_p(out.data_ptr()),
                        ctypes.c_void_p(stream))
    assert rc == 0, pkv.status_string(rc)
    torch.cuda.synchronize()

    bits = (lambda t: t.view(torch.int32)) if dtype == torch.float32 else (
        lambda t: t.view(torch.int16))
    assert torch.equal(bits(w.k_cache.cpu()), bits(kc_h))
    assert torch.equal(bits(w.v_cache.cpu()), bits(vc_h))
    g = out.double().cpu().numpy()
    assert np.isfinite(g).all()
    err = np.abs(g - ref)
    tol = BASE[dtype] + 0.5 * torch.finfo(dtype).eps * np.abs(ref)
    assert (err <= tol).all(), f"max err {err.max():.3e}"
