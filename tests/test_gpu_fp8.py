"""FP8 (E4M3) KV pools on the GPU against the oracle: the quantising append is
bit-exact (codes and scales), decode over FP8 pools matches the oracle's
decode of the stored values (code * row scale) within the fp16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

pytestmark = pytest.mark.gpu


def _close(out, ref, plain=False):
    g = out.double().cpu().numpy()
    err = np.abs(g - ref)
    tol = 2e-3 + 0.5 * torch.finfo(torch.float16).eps * np.abs(ref)
    assert not np.isnan(g).any()
    assert (err <= tol).all(), f"max err {err.max():.3e}"
    if plain:
        assert err.max() <= 2e-3


@pytest.mark.parametrize("in_dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
def test_append_fp8_bit_exact(pkv_lib, oracle_lib, in_dtype, d):
    torch.manual_seed(0)
    nb, hkv, bs, T = 40, 4, 16, 37
    kc = torch.randint(0, 256, (nb, hkv, bs, d), dtype=torch.uint8, device="cuda")
    vc = torch.randint(0, 256, (nb, hkv, bs, d), dtype=torch.uint8, device="cuda")
    ks = torch.rand(nb, hkv, bs, device="cuda")
    vs = torch.rand(nb, hkv, bs, device="cuda")
    k = (torch.randn(T, hkv, d, device="cuda") * 3).to(in_dtype)
    v = (torch.randn(T, hkv, d, device="cuda") * 0.01).to(in_dtype)
    k[0] = 0                       # all-zero rows: scale 1, zero codes
    k[1, :, ::2] = -0.0            # signed zeros next to values
    k[2] = 1000 if in_dtype != torch.float16 else 60000   # large magnitudes
    v[3, :, 5] = 1e-4              # one non-zero value per row
    v[3, :, :5] = 0
    slots = torch.randperm(nb * bs, device="cuda")[:T].to(torch.int64)
    slots[7] = -1
    slots[9] = nb * bs + 3         # beyond the pool: skipped
    h = [x.cpu() for x in (kc, vc, ks, vs)]
    pkv_lib.pkv_append_fp8(k, v, slots, kc, vc, ks, vs)
    o_slots = slots.cpu().numpy().copy()
    o_slots[9] = -1
    oracle.append_fp8(k.cpu(), v.cpu(), o_slots, *h)
    torch.cuda.synchronize()
    assert torch.equal(kc.cpu(), h[0]) and torch.equal(vc.cpu(), h[1])
    assert torch.equal(ks.cpu().view(torch.int32), h[2].view(torch.int32))
    assert torch.equal(vs.cpu().view(torch.int32), h[3].view(torch.int32))


CASES = [
    ("mha_small", dict(num_seqs=5, num_q_heads=4, num_kv_heads=4, lens=[1, 16, 17, 700, 1399]),
     0, 0, (0, 16, 64)),
    ("gqa4_bs32", dict(num_seqs=5, num_q_heads=8, num_kv_heads=2, block_size=32,
                       lens=[2, 32, 33, 64, 2500]), 0, 0, (0, 16, 2048)),
    ("g16", dict(num_seqs=3, num_q_heads=32, num_kv_heads=2, lens=[5, 250, 777]), 0, 0, (0, 48)),
    ("g32_chunks", dict(num_seqs=2, num_q_heads=32, num_kv_heads=1, lens=[40, 900]), 0, 0,
     (0, 32)),
    ("window_sinks", dict(num_seqs=6, num_q_heads=8, num_kv_heads=2,
                          lens=[1, 20, 100, 101, 317, 2000]), 37, 4, (0, 16)),
    ("long_split", dict(num_seqs=3, num_q_heads=8, num_kv_heads=2, lens=[100, 3000, 6000]),
     0, 0, (4096, 65536)),
    ("window_sinks_long_split", dict(num_seqs=2, num_q_heads=8, num_kv_heads=2,
                                     lens=[2600, 6000]), 2500, 4, (2528,)),
]


@pytest.mark.parametrize("name,over,window,sinks,splits", CASES, ids=[c[0] for c in CASES])
def test_decode_fp8_small(pkv_lib, oracle_lib, name, over, window, sinks, splits):
    spec = config_spec(0, dtype=torch.float16, head_dim=128, explicit_pool=None,
                       lens_are_pre_append=False, kv_fp8=True, window=window, num_sinks=sinks,
                       **over)
    w = make_workload(spec, device="cuda", poison_outside_window=True)
    # the step: quantise the new token in, then decode
    slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                     spec.block_size)
    h = [x.cpu() for x in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    o_slots = oracle.slot_mapping(w.block_tables.cpu().numpy(), w.pos_steps[0].cpu().numpy(),
                                  spec.block_size)
    oracle.append_fp8(w.k_steps[0].cpu(), w.v_steps[0].cpu(), o_slots, *h)
    ref = oracle.decode_fp8(w.q_steps[0].cpu(), *h, w.block_tables.cpu().numpy(),
                            w.lens_steps[0].cpu().numpy(), window, w.scale, num_sinks=sinks)
    pkv_lib.pkv_append_fp8(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache, w.k_scale,
                           w.v_scale)
    for tps in splits:
        out = pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables,
                                 w.lens_steps[0].contiguous(), window, w.scale,
                                 tokens_per_split=tps, num_sinks=sinks, k_scale=w.k_scale,
                                 v_scale=w.v_scale)
        torch.cuda.synchronize()
        _close(out, ref)
    assert torch.equal(w.k_cache.cpu(), h[0]) and torch.equal(w.v_cache.cpu(), h[1])


@pytest.mark.parametrize("name", ["mha_fp8", "gqa_fp8"])
def test_decode_fp8_benchmark_size(pkv_lib, oracle_lib, name):
    from paged_kv_cache_24_gb300.workloads import CONFIGS
    w = make_workload(config_spec(CONFIGS[name]), device="cuda")
    spec = w.spec
    slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                     spec.block_size)
    pkv_lib.pkv_append_fp8(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache, w.k_scale,
                           w.v_scale)
    out = pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables,
                             w.lens_steps[0].contiguous(), 0, w.scale, k_scale=w.k_scale,
                             v_scale=w.v_scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    pairs = np.stack([rng.integers(0, spec.num_seqs, 96), rng.integers(0, spec.num_q_heads, 96)],
                     1).astype(np.int32)
    h = [x.cpu() for x in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    ref = oracle.decode_fp8(w.q_steps[0].cpu(), *h, w.block_tables.cpu().numpy(),
                            w.lens_steps[0].cpu().numpy(), 0, w.scale, pairs=pairs)
    got = out[torch.from_numpy(pairs[:, 0]).long(), torch.from_numpy(pairs[:, 1]).long()]
    _close(got, ref, plain=True)
    assert torch.isfinite(out.float()).all()


def test_fp8_rejects_fused_append_and_missing_scales(pkv_lib):
    w = make_workload(config_spec(0, dtype=torch.float16, head_dim=128, num_q_heads=8,
                                  num_kv_heads=8, kv_fp8=True), device="cuda")
    with pytest.raises(ValueError):
        pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables,
                           w.lens_steps[0].contiguous(), 0, w.scale)
    with pytest.raises(pkv_lib.PkvError):
        lib = pkv_lib.load_library()
        import ctypes
        opts = pkv_lib.DecodeOptions(0, 0, 0, w.k_steps[0].data_ptr(), w.v_steps[0].data_ptr(),
                                     w.k_scale.data_ptr(), w.v_scale.data_ptr())
        out = torch.empty_like(w.q_steps[0])
        rc = lib.pkv_decode_ex(w.q_steps[0].data_ptr(), 4, 8, w.k_cache.data_ptr(),
                               w.v_cache.data_ptr(), ctypes.byref(pkv_lib.cache_layout(w.k_cache)),
                               w.block_tables.data_ptr(), w.block_tables.shape[1],
                               w.lens_steps[0].contiguous().data_ptr(), w.scale, out.data_ptr(),
                               ctypes.byref(opts), None)
        if rc != 0:
            raise pkv_lib.PkvError("pkv_decode_ex", rc, pkv_lib.status_string(rc))
