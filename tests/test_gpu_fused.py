"""pkv_append_decode (append + decode in one launch) against the separate calls
(bit-identical pools and outputs) and against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

pytestmark = pytest.mark.gpu

BASE_TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 2e-3}


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _separate(pkv, w, s, kc, vc, tps):
    slots = pkv.pkv_slot_mapping(w.block_tables, w.pos_steps[s].contiguous(), w.spec.block_size)
    pkv.pkv_append(w.k_steps[s], w.v_steps[s], slots, kc, vc)
    return pkv.pkv_decode(w.q_steps[s], kc, vc, w.block_tables, w.lens_steps[s].contiguous(),
                          w.spec.window, w.scale, tokens_per_split=tps)


def _fused(pkv, w, s, kc, vc, tps):
    return pkv.pkv_append_decode(w.q_steps[s], w.k_steps[s], w.v_steps[s], kc, vc,
                                 w.block_tables, w.lens_steps[s].contiguous(), w.spec.window,
                                 w.scale, tokens_per_split=tps)


def _oracle_step(w, s, kc_h, vc_h, pairs=None):
    bt = w.block_tables.cpu().numpy()
    slots = oracle.slot_mapping(bt, w.pos_steps[s].cpu().numpy(), w.spec.block_size)
    oracle.append(w.k_steps[s].cpu(), w.v_steps[s].cpu(), slots, kc_h, vc_h)
    return oracle.decode(w.q_steps[s].cpu(), kc_h, vc_h, bt, w.lens_steps[s].cpu().numpy(),
                         w.spec.window, w.scale, pairs=pairs)


def _check_oracle(out, ref, dtype, plain=False):
    g = out.double().cpu().numpy()
    err = np.abs(g - ref)
    tol = BASE_TOL[dtype] + 0.5 * torch.finfo(dtype).eps * np.abs(ref)
    assert (err <= tol).all(), f"max err {err.max():.3e}"
    if plain:
        assert err.max() <= BASE_TOL[dtype]


CASES = [
    ("tiny_fp32", dict(), (0, 16)),
    ("fp32_d128_g4", dict(dtype=torch.float32, head_dim=128, num_q_heads=8, num_kv_heads=2,
                          num_seqs=4, lens=[0, 1, 100, 517], explicit_pool=None), (0, 32)),
    ("fp16_mha", dict(dtype=torch.float16, num_seqs=5, num_q_heads=4, num_kv_heads=4,
                      head_dim=128, lens=[1, 16, 17, 700, 1399], explicit_pool=None,
                      lens_are_pre_append=False), (0, 16, 64)),
    ("bf16_gqa_bs32", dict(dtype=torch.bfloat16, num_seqs=5, num_q_heads=8, num_kv_heads=2,
                           head_dim=128, block_size=32, lens=[2, 32, 33, 64, 2500],
                           explicit_pool=None, lens_are_pre_append=False), (0, 16, 2048)),
    ("bf16_d64_g16", dict(dtype=torch.bfloat16, num_seqs=3, num_q_heads=32, num_kv_heads=2,
                          head_dim=64, lens=[5, 250, 777], explicit_pool=None,
                          lens_are_pre_append=False), (0, 48)),
    ("fp16_g32_chunks", dict(dtype=torch.float16, num_seqs=2, num_q_heads=32, num_kv_heads=1,
                             head_dim=128, lens=[40, 900], explicit_pool=None,
                             lens_are_pre_append=False), (0, 32)),
    ("bf16_window", dict(dtype=torch.bfloat16, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, block_size=16, lens=[1, 20, 100, 101, 317, 2000],
                         window=37, explicit_pool=None, lens_are_pre_append=False), (0, 16)),
]


@pytest.mark.parametrize("name,over,splits", CASES, ids=[c[0] for c in CASES])
def test_fused_equals_separate_and_oracle(pkv_lib, oracle_lib, name, over, splits):
    spec = config_spec(0, **over)
    base = make_workload(spec, device="cuda", poison_outside_window=True)
    kc_h, vc_h = base.k_cache.cpu(), base.v_cache.cpu()
    ref = _oracle_step(base, 0, kc_h, vc_h)
    for tps in splits:
        ka, va = base.k_cache.clone(), base.v_cache.clone()
        kb, vb = base.k_cache.clone(), base.v_cache.clone()
        out_a = _separate(pkv_lib, base, 0, ka, va, tps)
        out_b = _fused(pkv_lib, base, 0, kb, vb, tps)
        torch.cuda.synchronize()
        assert torch.equal(_bits(ka), _bits(kb)) and torch.equal(_bits(va), _bits(vb))
        assert torch.equal(_bits(out_a), _bits(out_b))
        assert torch.equal(_bits(kb.cpu()), _bits(kc_h)) and torch.equal(_bits(vb.cpu()), _bits(vc_h))
        _check_oracle(out_b, ref, spec.dtype)


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_fused_benchmark_workloads(pkv_lib, oracle_lib, idx):
    w = make_workload(config_spec(idx), device="cuda", poison_outside_window=True)
    ka, va = w.k_cache.clone(), w.v_cache.clone()
    out_a = _separate(pkv_lib, w, 0, ka, va, 0)
    del ka, va
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    out_b = _fused(pkv_lib, w, 0, w.k_cache, w.v_cache, 0)
    torch.cuda.synchronize()
    assert torch.equal(_bits(out_a), _bits(out_b))
    rng = np.random.default_rng(idx)
    pairs = np.stack([rng.integers(0, w.spec.num_seqs, 64),
                      rng.integers(0, w.spec.num_q_heads, 64)], 1).astype(np.int32)
    ref = _oracle_step(w, 0, kc_h, vc_h, pairs=pairs)
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(kc_h))
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(vc_h))
    got = out_b[torch.from_numpy(pairs[:, 0]).long(), torch.from_numpy(pairs[:, 1]).long()]
    _check_oracle(got, ref, w.spec.dtype, plain=True)


def test_fused_serving_32_steps(pkv_lib, oracle_lib):
    w = make_workload(config_spec(4), device="cuda")
    ka, va = w.k_cache.clone(), w.v_cache.clone()
    for s in range(w.steps):
        out_a = _separate(pkv_lib, w, s, ka, va, 0)
        out_b = _fused(pkv_lib, w, s, w.k_cache, w.v_cache, 0)
        assert torch.equal(_bits(out_a), _bits(out_b))
    torch.cuda.synchronize()
    assert torch.equal(_bits(ka), _bits(w.k_cache)) and torch.equal(_bits(va), _bits(w.v_cache))


def test_fused_empty_context_writes_nothing(pkv_lib):
    dt = torch.float16
    q = torch.randn(2, 4, 128, device="cuda").to(dt)
    kc = torch.full((3, 2, 16, 128), float("nan"), device="cuda", dtype=dt)
    vc = kc.clone()
    kn = torch.randn(2, 2, 128, device="cuda").to(dt)
    vn = torch.randn_like(kn)
    bt = torch.tensor([[0, 1], [2, 1]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    out = pkv_lib.pkv_append_decode(q, kn, vn, kc, vc, bt, lens, 0, 0.1)
    torch.cuda.synchronize()
    assert (out[0] == 0).all()
    # sequence 1: its single token is the new one, written to block 2 row 0
    assert torch.equal(kc[2, :, 0], kn[1]) and torch.equal(vc[2, :, 0], vn[1])
    assert torch.equal(out[1], vn[1].repeat_interleave(2, dim=0))
    assert torch.isnan(kc[0]).all() and torch.isnan(kc[1]).all()
