"""INT8 KV pools on the GPU against the oracle: the quantising append is
bit-exact (codes and scales), decode over INT8 pools matches the oracle's
decode of the stored values (code * row scale) within the fp16 tolerance, and
the public step (DecodeStep) runs over them."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import CONFIGS, config_spec, make_workload

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
def test_append_int8_bit_exact(pkv_lib, oracle_lib, in_dtype, d):
    torch.manual_seed(1)
    nb, hkv, bs, T = 40, 4, 16, 37
    kc = torch.randint(-128, 128, (nb, hkv, bs, d), dtype=torch.int8, device="cuda")
    vc = torch.randint(-128, 128, (nb, hkv, bs, d), dtype=torch.int8, device="cuda")
    ks = torch.rand(nb, hkv, bs, device="cuda")
    vs = torch.rand(nb, hkv, bs, device="cuda")
    k = (torch.randn(T, hkv, d, device="cuda") * 3).to(in_dtype)
    v = (torch.randn(T, hkv, d, device="cuda") * 0.01).to(in_dtype)
    k[0] = 0                       # all-zero rows: scale 1, zero codes
    k[1, :, ::2] = -0.0            # signed zeros next to values
    k[2] = 1000 if in_dtype != torch.float16 else 60000   # large magnitudes
    v[3, :, 5] = 1e-4              # one non-zero value per row
    v[3, :, :5] = 0
    # exact halves of the step: ties, which round to even
    k[4, :, :] = 0
    k[4, :, 0] = 127.0
    k[4, :, 1:9] = torch.tensor([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, 126.5]).to(in_dtype)
    slots = torch.randperm(nb * bs, device="cuda")[:T].to(torch.int64)
    slots[7] = -1
    slots[9] = nb * bs + 3         # beyond the pool: skipped
    h = [x.cpu() for x in (kc, vc, ks, vs)]
    pkv_lib.pkv_append_int8(k, v, slots, kc, vc, ks, vs)
    o_slots = slots.cpu().numpy().copy()
    o_slots[9] = -1
    oracle.append_int8(k.cpu(), v.cpu(), o_slots, *h)
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
def test_decode_int8_small(pkv_lib, oracle_lib, name, over, window, sinks, splits):
    spec = config_spec(0, dtype=torch.float16, head_dim=128, explicit_pool=None,
                       lens_are_pre_append=False, kv_int8=True, window=window, num_sinks=sinks,
                       **over)
    w = make_workload(spec, device="cuda", poison_outside_window=True)
    # the step: quantise the new token in, then decode
    slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                     spec.block_size)
    h = [x.cpu() for x in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    o_slots = oracle.slot_mapping(w.block_tables.cpu().numpy(), w.pos_steps[0].cpu().numpy(),
                                  spec.block_size)
    oracle.append_int8(w.k_steps[0].cpu(), w.v_steps[0].cpu(), o_slots, *h)
    ref = oracle.decode_int8(w.q_steps[0].cpu(), *h, w.block_tables.cpu().numpy(),
                             w.lens_steps[0].cpu().numpy(), window, w.scale, num_sinks=sinks)
    pkv_lib.pkv_append_int8(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache, w.k_scale,
                            w.v_scale)
    for tps in splits:
        out = pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables,
                                 w.lens_steps[0].contiguous(), window, w.scale,
                                 tokens_per_split=tps, num_sinks=sinks, k_scale=w.k_scale,
                                 v_scale=w.v_scale)
        torch.cuda.synchronize()
        _close(out, ref)
    assert torch.equal(w.k_cache.cpu(), h[0]) and torch.equal(w.v_cache.cpu(), h[1])


def test_decode_int8_extreme_codes(pkv_lib, oracle_lib):
    """Codes at +-127 and 0 in every row (the whole conversion range) and
    scales spanning eight octaves."""
    spec = config_spec(0, dtype=torch.float16, head_dim=128, explicit_pool=None,
                       lens_are_pre_append=False, kv_int8=True, num_seqs=3, num_q_heads=8,
                       num_kv_heads=2, lens=[3, 64, 300])
    w = make_workload(spec, device="cuda", poison=False)
    g = torch.Generator(device="cuda").manual_seed(9)
    pattern = torch.tensor([127, -127, 0, 1, -1, 64, -64, 100], dtype=torch.int8, device="cuda")
    w.k_cache.copy_(pattern.repeat(w.k_cache.numel() // 8).view_as(w.k_cache))
    w.v_cache.copy_(pattern.flip(0).repeat(w.v_cache.numel() // 8).view_as(w.v_cache))
    w.k_scale.copy_(2.0 ** (torch.rand(w.k_scale.shape, generator=g, device="cuda") * 8 - 10))
    w.v_scale.copy_(2.0 ** (torch.rand(w.v_scale.shape, generator=g, device="cuda") * 8 - 8))
    h = [x.cpu() for x in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    ref = oracle.decode_int8(w.q_steps[0].cpu(), *h, w.block_tables.cpu().numpy(),
                             w.lens_steps[0].cpu().numpy(), 0, w.scale)
    out = pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables,
                             w.lens_steps[0].contiguous(), 0, w.scale, k_scale=w.k_scale,
                             v_scale=w.v_scale)
    torch.cuda.synchronize()
    _close(out, ref)


@pytest.mark.parametrize("name", ["mha_int8", "gqa_int8"])
def test_decode_int8_benchmark_size(pkv_lib, oracle_lib, name):
    w = make_workload(config_spec(CONFIGS[name]), device="cuda")
    spec = w.spec
    slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                     spec.block_size)
    pkv_lib.pkv_append_int8(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache,
                            w.k_scale, w.v_scale)
    out = pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables,
                             w.lens_steps[0].contiguous(), 0, w.scale, k_scale=w.k_scale,
                             v_scale=w.v_scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    pairs = np.stack([rng.integers(0, spec.num_seqs, 96), rng.integers(0, spec.num_q_heads, 96)],
                     1).astype(np.int32)
    h = [x.cpu() for x in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    ref = oracle.decode_int8(w.q_steps[0].cpu(), *h, w.block_tables.cpu().numpy(),
                             w.lens_steps[0].cpu().numpy(), 0, w.scale, pairs=pairs)
    got = out[torch.from_numpy(pairs[:, 0]).long(), torch.from_numpy(pairs[:, 1]).long()]
    _close(got, ref, plain=True)
    assert torch.isfinite(out.float()).all()


def test_decode_step_over_int8_pools(pkv_lib, oracle_lib):
    """The public step: pinned staging in, quantising append + decode in one
    CUDA graph, output back."""
    spec = config_spec(0, dtype=torch.float16, head_dim=128, explicit_pool=None,
                       lens_are_pre_append=False, kv_int8=True, num_seqs=4, num_q_heads=8,
                       num_kv_heads=2, lens=[5, 33, 200, 1000])
    w = make_workload(spec, device="cuda", poison=False)
    h = [x.cpu() for x in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
    step = pkv_lib.DecodeStep(w.k_cache, w.v_cache, spec.num_seqs, spec.num_q_heads,
                              w.max_blocks, 0, w.scale, fused=False, k_scale=w.k_scale,
                              v_scale=w.v_scale)
    hb = step.host[0]
    hb["q"].copy_(w.q_steps[0]); hb["k"].copy_(w.k_steps[0]); hb["v"].copy_(w.v_steps[0])
    hb["positions"].copy_(w.pos_steps[0]); hb["context_lens"].copy_(w.lens_steps[0])
    hb["block_tables"].copy_(w.block_tables)
    out = step.run(0).clone()
    o_slots = oracle.slot_mapping(w.block_tables.cpu().numpy(), w.pos_steps[0].cpu().numpy(),
                                  spec.block_size)
    oracle.append_int8(w.k_steps[0].cpu(), w.v_steps[0].cpu(), o_slots, *h)
    ref = oracle.decode_int8(w.q_steps[0].cpu(), *h, w.block_tables.cpu().numpy(),
                             w.lens_steps[0].cpu().numpy(), 0, w.scale)
    _close(out, ref)
    assert torch.equal(w.k_cache.cpu(), h[0]) and torch.equal(w.v_cache.cpu(), h[1])
