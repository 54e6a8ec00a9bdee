"""Seeded random sweep of the CUDA path against the oracle: decode over fp32,
fp16, bf16, FP8 and INT8 pools (separate or fused append), and the chunked
prefill (with windows and sinks), on shapes drawn from the supported ranges -- head dims, GQA groups,
page sizes, ragged lengths, windows, attention sinks and split sizes.  Every
output and the whole pool after the append are compared; a failing case
names its seed."""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

pytestmark = pytest.mark.gpu

BASE_TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 2e-3}
# seeds per sweep; a longer sweep sets these (e.g. PKV_RANDOM_DECODE_SEEDS=5000)
N_DECODE = int(os.environ.get("PKV_RANDOM_DECODE_SEEDS", "30"))
N_PREFILL = int(os.environ.get("PKV_RANDOM_PREFILL_SEEDS", "24"))
N_WIDE = int(os.environ.get("PKV_RANDOM_WIDE_SEEDS", "12"))
KINDS = ("fp32", "fp16", "bf16", "fp8", "int8")
DTYPE = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16,
         "fp8": torch.float16, "int8": torch.float16}


def _bits(t):
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    if t.element_size() == 1:
        return t.view(torch.uint8)
    return t.view(torch.int16)


def _close(out, ref, dtype, what):
    g = out.double().cpu().numpy()
    err = np.abs(g - ref)
    tol = BASE_TOL[dtype] + 0.5 * torch.finfo(dtype).eps * np.abs(ref)
    assert not np.isnan(g).any(), f"{what}: NaN in the output"
    assert (err <= tol).all(), f"{what}: max err {err.max():.3e}"


def _decode_case(seed):
    r = np.random.default_rng(1000 + seed)
    kind = KINDS[seed % len(KINDS)]
    d = 128 if kind in ("fp8", "int8") else int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2, 4]))
    g = int(r.choice([1, 2, 3, 4, 6, 8, 16]))
    bs = int(r.choice([16, 32, 48, 64, 128, 256]))
    B = int(r.integers(1, 7))
    lens = r.integers(1, 2500, B)
    # a few lengths on and next to page edges
    for i in range(B):
        if r.random() < 0.3:
            lens[i] = max(1, bs * int(r.integers(1, 6)) + int(r.choice([-1, 0, 1])))
    window = 0 if r.random() < 0.4 else int(r.integers(1, 600))
    sinks = 0 if window == 0 else int(r.choice([0, 1, 4, 17]))
    tps = int(r.choice([0, 16, 48, 256, 2048, 4096, 65536]))
    fused = kind in ("fp32", "fp16", "bf16") and r.random() < 0.5
    over = dict(dtype=DTYPE[kind], num_seqs=B, num_q_heads=hkv * g, num_kv_heads=hkv,
                head_dim=d, block_size=bs, lens=[int(x) for x in lens], window=window,
                num_sinks=sinks, explicit_pool=None, lens_are_pre_append=False,
                seed=2000 + seed, kv_fp8=kind == "fp8", kv_int8=kind == "int8")
    return kind, over, tps, fused


@pytest.mark.parametrize("seed", range(N_DECODE))
def test_random_decode(pkv_lib, oracle_lib, seed):
    kind, over, tps, fused = _decode_case(seed)
    what = f"seed {seed}: {kind} {over} tps={tps} fused={fused}"
    spec = config_spec(0, **over)
    w = make_workload(spec, device="cuda", poison_outside_window=True)
    bt = w.block_tables.cpu().numpy()
    lens = w.lens_steps[0].contiguous()
    o_slots = oracle.slot_mapping(bt, w.pos_steps[0].cpu().numpy(), spec.block_size)
    if kind in ("fp8", "int8"):
        h = [x.cpu() for x in (w.k_cache, w.v_cache, w.k_scale, w.v_scale)]
        app, dec = ((oracle.append_fp8, oracle.decode_fp8) if kind == "fp8"
                    else (oracle.append_int8, oracle.decode_int8))
        app(w.k_steps[0].cpu(), w.v_steps[0].cpu(), o_slots, *h)
        ref = dec(w.q_steps[0].cpu(), *h, bt, lens.cpu().numpy(), spec.window, w.scale,
                  num_sinks=spec.num_sinks)
        slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                         spec.block_size)
        append = pkv_lib.pkv_append_fp8 if kind == "fp8" else pkv_lib.pkv_append_int8
        append(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache, w.k_scale, w.v_scale)
        out = pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables, lens,
                                 spec.window, w.scale, tokens_per_split=tps,
                                 num_sinks=spec.num_sinks, k_scale=w.k_scale, v_scale=w.v_scale)
        torch.cuda.synchronize()
        assert torch.equal(w.k_scale.cpu().view(torch.int32), h[2].view(torch.int32)), what
        assert torch.equal(w.v_scale.cpu().view(torch.int32), h[3].view(torch.int32)), what
    else:
        h = [w.k_cache.cpu(), w.v_cache.cpu()]
        oracle.append(w.k_steps[0].cpu(), w.v_steps[0].cpu(), o_slots, *h)
        ref = oracle.decode(w.q_steps[0].cpu(), *h, bt, lens.cpu().numpy(), spec.window,
                            w.scale, num_sinks=spec.num_sinks)
        if fused:
            out = pkv_lib.pkv_append_decode(w.q_steps[0], w.k_steps[0], w.v_steps[0],
                                             w.k_cache, w.v_cache, w.block_tables, lens,
                                             spec.window, w.scale, tokens_per_split=tps,
                                             num_sinks=spec.num_sinks)
        else:
            slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                             spec.block_size)
            pkv_lib.pkv_append(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache)
            out = pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables, lens,
                                     spec.window, w.scale, tokens_per_split=tps,
                                     num_sinks=spec.num_sinks)
        torch.cuda.synchronize()
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(h[0])), what
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(h[1])), what
    _close(out, ref, spec.dtype, what)


def _prefill_case(seed):
    r = np.random.default_rng(3000 + seed)
    dtype = (torch.float16, torch.bfloat16)[seed % 2]
    d = int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2, 4]))
    g = int(r.choice([1, 2, 3, 4, 6, 8, 16]))
    bs = int(r.choice([16, 32, 64]))
    B = int(r.integers(1, 6))
    prefixes = [int(x) for x in r.integers(0, 1500, B)]
    chunks = [int(x) for x in r.integers(1, 400, B)]
    window = 0 if r.random() < 0.5 else int(r.integers(1, 700))
    sinks = 0 if window == 0 else int(r.choice([0, 0, 1, 4, 19, 200]))
    return dtype, d, hkv, g, bs, prefixes, chunks, window, sinks


@pytest.mark.parametrize("seed", range(N_PREFILL))
def test_random_prefill(pkv_lib, oracle_lib, seed):
    dtype, d, hkv, g, bs, prefixes, chunks, window, sinks = _prefill_case(seed)
    what = (f"seed {seed}: {dtype} d={d} hkv={hkv} g={g} bs={bs} {prefixes} {chunks} "
            f"w={window} sinks={sinks}")
    lens = [p + n for p, n in zip(prefixes, chunks)]
    spec = config_spec(0, dtype=dtype, num_seqs=len(lens), num_q_heads=hkv * g,
                       num_kv_heads=hkv, head_dim=d, block_size=bs, lens=lens,
                       explicit_pool=None, lens_are_pre_append=False, window=0, seed=4000 + seed)
    w = make_workload(spec, device="cuda")
    bt = w.block_tables.cpu().numpy()
    # the chunk's own slots start as NaN: the prefill must write them first
    slots = np.array([oracle.slot_for_position(bt[b], bs, t)
                      for b, (p, L) in enumerate(zip(prefixes, lens)) for t in range(p, L)],
                     np.int64)
    blk = torch.from_numpy(slots // bs).to("cuda")
    row = torch.from_numpy(slots % bs).to("cuda")
    w.k_cache[blk, :, row] = float("nan")
    w.v_cache[blk, :, row] = float("nan")
    gen = torch.Generator(device="cuda").manual_seed(5000 + seed)
    T = sum(chunks)
    q = torch.randn(T, hkv * g, d, generator=gen, device="cuda").to(dtype)
    k = torch.randn(T, hkv, d, generator=gen, device="cuda").to(dtype)
    v = torch.randn(T, hkv, d, generator=gen, device="cuda").to(dtype)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32, device="cuda")
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    oracle.append(k.cpu(), v.cpu(), slots, kc_h, vc_h)
    ref = oracle.prefill(q.cpu(), cu.cpu().numpy(), kc_h, vc_h, bt, np.array(lens, np.int32),
                         window, w.scale, num_sinks=sinks)
    out = torch.full_like(q, float("nan"))
    pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, L, window, w.scale,
                        max_chunk=max(chunks), out=out, num_sinks=sinks)
    torch.cuda.synchronize()
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(kc_h)), what
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(vc_h)), what
    _close(out, ref, dtype, what)


@pytest.mark.parametrize("seed", range(N_WIDE))
def test_random_prefill_bf16_wide_range(pkv_lib, oracle_lib, seed):
    """bf16 prefills whose (sequence, kv head) pairs each hold V at their own
    scale, 10^-30 .. 10^30 (some pairs also one value 10^12 times larger than
    the rest), in random shapes: the outputs match the oracle's relative to
    each pair's scale -- through both the scaled-fp16 product and the exact
    bf16 one (the outlier is capped at 1e37, inside bf16's range)."""
    _, d, hkv, g, bs, prefixes, chunks, window, sinks = _prefill_case(seed + 100)
    dtype = torch.bfloat16
    r = np.random.default_rng(7000 + seed)
    what = (f"seed {seed}: d={d} hkv={hkv} g={g} bs={bs} {prefixes} {chunks} "
            f"w={window} sinks={sinks}")
    lens = [p + n for p, n in zip(prefixes, chunks)]
    B = len(lens)
    spec = config_spec(0, dtype=dtype, num_seqs=B, num_q_heads=hkv * g, num_kv_heads=hkv,
                       head_dim=d, block_size=bs, lens=lens, explicit_pool=None,
                       lens_are_pre_append=False, window=0, seed=8000 + seed)
    w = make_workload(spec, device="cuda")
    bt = w.block_tables.cpu().numpy()
    gen = torch.Generator(device="cuda").manual_seed(9000 + seed)
    T = sum(chunks)
    q = torch.randn(T, hkv * g, d, generator=gen, device="cuda").to(dtype)
    k = torch.randn(T, hkv, d, generator=gen, device="cuda").to(dtype)
    v = torch.randn(T, hkv, d, generator=gen, device="cuda").to(dtype)
    starts = np.concatenate([[0], np.cumsum(chunks)])
    scale = np.ones((B, hkv))
    for b in range(B):
        prefix_slots = np.array([oracle.slot_for_position(bt[b], bs, t)
                                 for t in range(prefixes[b])], np.int64)
        for h in range(hkv):
            s = 10.0 ** int(r.integers(-30, 31))
            scale[b, h] = s
            if prefix_slots.size:
                blk = torch.from_numpy(prefix_slots // bs).to("cuda")
                row = torch.from_numpy(prefix_slots % bs).to("cuda")
                w.v_cache[blk, h, row] = (w.v_cache[blk, h, row].double() * s).to(dtype)
            v[starts[b]:starts[b + 1], h] = (v[starts[b]:starts[b + 1], h].double() * s).to(dtype)
            if r.random() < 0.3:  # one value far above the pair's others (finite in bf16)
                t = int(r.integers(0, lens[b]))
                c = int(r.integers(0, d))
                big = min(1.0e12 * s, 1.0e37)
                if t < prefixes[b]:
                    sl = oracle.slot_for_position(bt[b], bs, t)
                    w.v_cache[sl // bs, h, sl % bs, c] = big
                else:
                    v[starts[b] + t - prefixes[b], h, c] = big
    # the chunk's own slots start as NaN: the prefill must write them first
    slots = np.array([oracle.slot_for_position(bt[b], bs, t)
                      for b, (p, L) in enumerate(zip(prefixes, lens)) for t in range(p, L)],
                     np.int64)
    w.k_cache[torch.from_numpy(slots // bs).to("cuda"), :,
              torch.from_numpy(slots % bs).to("cuda")] = float("nan")
    w.v_cache[torch.from_numpy(slots // bs).to("cuda"), :,
              torch.from_numpy(slots % bs).to("cuda")] = float("nan")
    cu = torch.tensor(starts, dtype=torch.int32, device="cuda")
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    oracle.append(k.cpu(), v.cpu(), slots, kc_h, vc_h)
    ref = oracle.prefill(q.cpu(), cu.cpu().numpy(), kc_h, vc_h, bt, np.array(lens, np.int32),
                         window, w.scale, num_sinks=sinks)
    out = torch.full_like(q, float("nan"))
    pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, L, window, w.scale,
                        max_chunk=max(chunks), out=out, num_sinks=sinks)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all(), what
    # every output row of sequence b, query head hq is in units of its pair's scale
    row_scale = np.repeat(np.repeat(scale, g, axis=1)[:, None, :], 1, axis=1)
    tok_b = np.repeat(np.arange(B), chunks)
    s = row_scale[tok_b][:, 0, :, None]          # [T, Hq, 1]
    err = np.abs(got - ref) / s
    tol = 2e-3 + 0.5 * torch.finfo(dtype).eps * np.abs(ref) / s
    assert (err <= tol).all(), f"{what}: max scaled err {err.max():.3e}"
