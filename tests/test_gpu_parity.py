"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Bar: slot mapping, append and the whole pool after it are bit-exact; decode
outputs are within max-abs error 2e-3 (fp16 / bf16 inputs, fp32 accumulation)
or 1e-5 (fp32) of the oracle.  Outputs are rounded into their 16-bit dtype,
which by itself can cost half an ulp (up to 2^-8 = 3.9e-3 at |x| in [1, 2) for
bf16), so small-context cases, whose outputs are O(1), compare with
    |gpu - oracle| <= base + eps(dtype) / 2 * |oracle|,
base = 2e-3 or 1e-5.  The benchmark-size workloads (long contexts, |out| << 1)
must also meet the plain base bound.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

pytestmark = pytest.mark.gpu

BASE_TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 2e-3}


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def check_close(gpu_out, ref, dtype, plain=False):
    g = gpu_out.detach().double().cpu().numpy()
    base = BASE_TOL[dtype]
    err = np.abs(g - ref)
    tol = base + 0.5 * torch.finfo(dtype).eps * np.abs(ref)
    assert not np.isnan(g).any(), "NaN in GPU output"
    worst = np.argmax(err - tol)
    assert (err <= tol).all(), (f"max err {err.max():.3e}; worst {err.flat[worst]:.3e} > tol "
                                f"{tol.flat[worst]:.3e} at ref {ref.flat[worst]:.4f}")
    if plain:
        assert err.max() <= base, f"max abs err {err.max():.3e} > {base}"
    return float(err.max())


class HostMirror:
    """Host copy of a workload's state that the oracle advances step by step."""

    def __init__(self, w):
        self.w = w
        self.kc = w.k_cache.cpu()
        self.vc = w.v_cache.cpu()
        self.bt = w.block_tables.cpu().numpy()

    def step(self, s, pairs=None):
        w = self.w
        pos = w.pos_steps[s].cpu().numpy()
        slots = oracle.slot_mapping(self.bt, pos, w.spec.block_size)
        oracle.append(w.k_steps[s].cpu(), w.v_steps[s].cpu(), slots, self.kc, self.vc)
        ref = oracle.decode(w.q_steps[s].cpu(), self.kc, self.vc, self.bt,
                            w.lens_steps[s].cpu().numpy(), w.spec.window, w.scale, pairs=pairs)
        return slots, ref


def gpu_step(pkv, w, s, tokens_per_split=0, stream=None):
    slots = pkv.pkv_slot_mapping(w.block_tables, w.pos_steps[s].contiguous(), w.spec.block_size,
                                 stream=stream)
    pkv.pkv_append(w.k_steps[s], w.v_steps[s], slots, w.k_cache, w.v_cache, stream=stream)
    out = pkv.pkv_decode(w.q_steps[s], w.k_cache, w.v_cache, w.block_tables,
                         w.lens_steps[s].contiguous(), w.spec.window, w.scale,
                         tokens_per_split=tokens_per_split, stream=stream)
    return slots, out


# ---------------------------------------------------------------------------
# small and mid-size cases: every output compared


SMALL = [
    # name, spec overrides, tokens_per_split values to try
    ("tiny_fp32", dict(), (0, 16, 32)),
    ("fp32_d128_gqa", dict(dtype=torch.float32, head_dim=128, num_q_heads=12, num_kv_heads=3,
                           num_seqs=5, lens=[1, 17, 100, 300, 513], explicit_pool=None), (0, 64)),
    ("mha_fp16_small", dict(dtype=torch.float16, num_seqs=6, num_q_heads=4, num_kv_heads=4,
                            head_dim=128, lens=[1, 2, 16, 17, 600, 1333], explicit_pool=None,
                            lens_are_pre_append=False), (0, 16, 128)),
    ("gqa_bf16_bs32", dict(dtype=torch.bfloat16, num_seqs=5, num_q_heads=8, num_kv_heads=2,
                           head_dim=128, block_size=32, lens=[3, 31, 32, 33, 1500],
                           explicit_pool=None, lens_are_pre_append=False), (0, 16, 2048)),
    ("bf16_d64_g16", dict(dtype=torch.bfloat16, num_seqs=3, num_q_heads=32, num_kv_heads=2,
                          head_dim=64, block_size=16, lens=[5, 250, 777], explicit_pool=None,
                          lens_are_pre_append=False), (0, 48)),
    ("fp16_d64_g6_bs64", dict(dtype=torch.float16, num_seqs=4, num_q_heads=12, num_kv_heads=2,
                              head_dim=64, block_size=64, lens=[64, 65, 129, 1000],
                              explicit_pool=None, lens_are_pre_append=False), (0, 80)),
    ("window_bf16", dict(dtype=torch.bfloat16, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, block_size=16, lens=[1, 20, 100, 101, 317, 2000],
                         window=37, explicit_pool=None, lens_are_pre_append=False), (0, 16)),
    ("window_16_fp16", dict(dtype=torch.float16, num_seqs=3, num_q_heads=4, num_kv_heads=1,
                            head_dim=128, block_size=16, lens=[15, 16, 47], window=16,
                            explicit_pool=None, lens_are_pre_append=False), (0,)),
    ("g32_two_chunks", dict(dtype=torch.bfloat16, num_seqs=2, num_q_heads=32, num_kv_heads=1,
                            head_dim=128, block_size=16, lens=[40, 900], explicit_pool=None,
                            lens_are_pre_append=False), (0, 32)),
]


# enough (sequence, kv head) items for the launcher to pick two ring stages and
# three CTAs per SM (at least 16 items per SM: 2432 on 152 SMs)
_r = np.random.default_rng(41)
SMALL.append(("many_short_fp16", dict(dtype=torch.float16, num_seqs=640, num_q_heads=8,
                                      num_kv_heads=4, head_dim=128, block_size=16,
                                      lens=_r.integers(1, 160, 640).tolist(), explicit_pool=None,
                                      lens_are_pre_append=False), (0, 32)))
SMALL.append(("many_short_bf16_bs32", dict(dtype=torch.bfloat16, num_seqs=700, num_q_heads=16,
                                           num_kv_heads=4, head_dim=128, block_size=32,
                                           lens=_r.integers(1, 120, 700).tolist(),
                                           explicit_pool=None, lens_are_pre_append=False), (0,)))


# more work items than SMs and fewer than 16 per SM
SMALL.append(("mid_grid_fp16", dict(dtype=torch.float16, num_seqs=40, num_q_heads=8,
                                    num_kv_heads=4, head_dim=128, block_size=16,
                                    lens=_r.integers(1, 600, 40).tolist(), explicit_pool=None,
                                    lens_are_pre_append=False), (0, 64)))
SMALL.append(("mid_grid_bf16_bs64", dict(dtype=torch.bfloat16, num_seqs=20, num_q_heads=16,
                                         num_kv_heads=8, head_dim=128, block_size=64,
                                         lens=_r.integers(1, 900, 20).tolist(),
                                         explicit_pool=None, lens_are_pre_append=False),
                      (0, 32)))

# the largest batch the decode grid takes (65535 sequences), with empty and
# one-token contexts among them
SMALL.append(("max_sequences_fp16_d64", dict(dtype=torch.float16, num_seqs=65535, num_q_heads=2,
                                             num_kv_heads=1, head_dim=64, block_size=16,
                                             lens=_r.integers(0, 33, 65535).tolist(),
                                             explicit_pool=None, lens_are_pre_append=False),
                      (0,)))

# splits longer than 32 units per warp: each warp resolves its pages 32 units
# at a time
SMALL.append(("long_split_fp16", dict(dtype=torch.float16, num_seqs=5, num_q_heads=4,
                                      num_kv_heads=4, head_dim=128, block_size=16,
                                      lens=[1, 700, 2100, 5000, 9000], explicit_pool=None,
                                      lens_are_pre_append=False), (4096, 65536)))
SMALL.append(("long_split_bf16_d64_window", dict(dtype=torch.bfloat16, num_seqs=4,
                                                 num_q_heads=16, num_kv_heads=2, head_dim=64,
                                                 block_size=32, lens=[2999, 3001, 3003, 7000],
                                                 window=3000, explicit_pool=None,
                                                 lens_are_pre_append=False), (0, 3008, 65536)))


@pytest.mark.parametrize("name,over,splits", SMALL, ids=[s[0] for s in SMALL])
def test_small_cases_all_outputs(pkv_lib, oracle_lib, name, over, splits):
    spec = config_spec(0, **over)
    for tps in splits:
        w = make_workload(spec, device="cuda", poison_outside_window=True)
        mirror = HostMirror(w)
        o_slots, ref = mirror.step(0)
        g_slots, out = gpu_step(pkv_lib, w, 0, tokens_per_split=tps)
        torch.cuda.synchronize()
        assert np.array_equal(g_slots.cpu().numpy(), o_slots)
        assert torch.equal(_bits(w.k_cache.cpu()), _bits(mirror.kc))
        assert torch.equal(_bits(w.v_cache.cpu()), _bits(mirror.vc))
        check_close(out, ref, spec.dtype)


SINKS = [
    # name, spec overrides, num_sinks, tokens_per_split values
    ("bf16_g4_w37_s4", dict(dtype=torch.bfloat16, num_seqs=8, num_q_heads=8, num_kv_heads=2,
                            head_dim=128, block_size=16,
                            lens=[1, 5, 20, 37, 38, 41, 700, 2000], window=37), 4, (0, 16, 64)),
    ("fp16_d64_bs32_w100_s20", dict(dtype=torch.float16, num_seqs=5, num_q_heads=4,
                                    num_kv_heads=4, head_dim=64, block_size=32,
                                    lens=[19, 110, 121, 130, 1500], window=100), 20, (0, 32)),
    ("fp32_w16_s4", dict(dtype=torch.float32, num_seqs=4, num_q_heads=8, num_kv_heads=2,
                         head_dim=128, lens=[3, 17, 21, 400], window=16), 4, (0, 16)),
    ("bf16_s16_aligned", dict(dtype=torch.bfloat16, num_seqs=3, num_q_heads=32, num_kv_heads=2,
                              head_dim=128, lens=[33, 64, 999], window=32), 16, (0, 16)),
    ("fp16_w2500_s20_long_split", dict(dtype=torch.float16, num_seqs=3, num_q_heads=8,
                                       num_kv_heads=2, head_dim=128, lens=[2600, 3000, 6000],
                                       window=2500), 20, (0, 2528, 65536)),
]


@pytest.mark.parametrize("name,over,sinks,splits", SINKS, ids=[c[0] for c in SINKS])
def test_attention_sinks(pkv_lib, oracle_lib, name, over, sinks, splits):
    spec = config_spec(0, explicit_pool=None, lens_are_pre_append=False, num_sinks=sinks,
                       **over)
    w = make_workload(spec, device="cuda", poison_outside_window=True)
    slots = pkv_lib.pkv_slot_mapping(w.block_tables, w.pos_steps[0].contiguous(),
                                     spec.block_size)
    pkv_lib.pkv_append(w.k_steps[0], w.v_steps[0], slots, w.k_cache, w.v_cache)
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    ref = oracle.decode(w.q_steps[0].cpu(), kc_h, vc_h, w.block_tables.cpu().numpy(),
                        w.lens_steps[0].cpu().numpy(), spec.window, w.scale, num_sinks=sinks)
    for tps in splits:
        out = pkv_lib.pkv_decode(w.q_steps[0], w.k_cache, w.v_cache, w.block_tables,
                                 w.lens_steps[0].contiguous(), spec.window, w.scale,
                                 tokens_per_split=tps, num_sinks=sinks)
        torch.cuda.synchronize()
        check_close(out, ref, spec.dtype)
    # fused append + decode with sinks, from the pre-append pool
    w2 = make_workload(spec, device="cuda", poison_outside_window=True)
    out = pkv_lib.pkv_append_decode(w2.q_steps[0], w2.k_steps[0], w2.v_steps[0], w2.k_cache,
                                    w2.v_cache, w2.block_tables, w2.lens_steps[0].contiguous(),
                                    spec.window, w2.scale, num_sinks=sinks)
    torch.cuda.synchronize()
    check_close(out, ref, spec.dtype)
    assert torch.equal(_bits(w2.k_cache.cpu()), _bits(kc_h))


def test_single_token_is_exact(pkv_lib, oracle_lib):
    for dt in (torch.float16, torch.bfloat16, torch.float32):
        spec = config_spec(0, dtype=dt, num_seqs=3, num_q_heads=4, num_kv_heads=2,
                           head_dim=128, lens=[1, 1, 1], explicit_pool=None,
                           lens_are_pre_append=False)
        w = make_workload(spec, device="cuda")
        _, out = gpu_step(pkv_lib, w, 0)
        # one token: weight exactly 1, out = v of that token for every query head
        expect = w.v_steps[0].repeat_interleave(2, dim=1)
        assert torch.equal(_bits(out), _bits(expect))


def test_empty_context_gives_zeros(pkv_lib):
    for dt in (torch.float16, torch.float32):
        q = torch.randn(3, 8, 128, device="cuda").to(dt)
        kc = torch.full((4, 2, 16, 128), float("nan"), device="cuda", dtype=dt)
        bt = torch.tensor([[0, 1], [2, 3], [1, 0]], dtype=torch.int32, device="cuda")
        lens = torch.tensor([0, 5, 0], dtype=torch.int32, device="cuda")
        kc[2, :, :5] = 1.0
        out = pkv_lib.pkv_decode(q, kc, kc.clone(), bt, lens, 0, 0.1)
        assert (out[0] == 0).all() and (out[2] == 0).all()
        assert torch.allclose(out[1].float(), torch.ones_like(out[1]).float())


def test_invalid_indices_give_nan_rows_only(pkv_lib):
    dt = torch.bfloat16
    q = torch.randn(4, 8, 128, device="cuda").to(dt)
    kc = torch.randn(6, 2, 16, 128, device="cuda").to(dt)
    vc = torch.randn_like(kc)
    bt = torch.tensor([[0, 1], [2, 99], [3, -5], [4, 5]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([20, 20, 20, 33], dtype=torch.int32, device="cuda")  # 33 > 2 * 16
    for tps in (0, 16):
        out = pkv_lib.pkv_decode(q, kc, vc, bt, lens, 0, 0.1, tokens_per_split=tps)
        torch.cuda.synchronize()
        assert torch.isfinite(out[0].float()).all()
        assert torch.isnan(out[1].float()).all()
        assert torch.isnan(out[2].float()).all()
        assert torch.isnan(out[3].float()).all()


def test_uniform_keys_give_mean_of_window_at_scale(pkv_lib):
    """Property at any size: equal keys -> the output is the mean of V over the window."""
    torch.manual_seed(0)
    B, hkv, G, d, bs, L, win = 4, 2, 4, 128, 16, 3000, 1111
    nb = B * (L // bs + 1)
    kc = torch.randn(1, hkv, 1, d, device="cuda").to(torch.bfloat16).expand(nb, hkv, bs, d).contiguous()
    vc = torch.randn(nb, hkv, bs, d, device="cuda").to(torch.bfloat16)
    bt = torch.randperm(nb, device="cuda").to(torch.int32).view(B, -1)
    lens = torch.tensor([L, L - 7, 200, 1], dtype=torch.int32, device="cuda")
    q = torch.randn(B, hkv * G, d, device="cuda").to(torch.bfloat16)
    out = pkv_lib.pkv_decode(q, kc, vc, bt, lens, win, 0.08)
    for b in range(B):
        Lb = int(lens[b])
        t = torch.arange(max(0, Lb - win), Lb, device="cuda")
        rows = vc[bt[b, t // bs].long(), :, t % bs].double()   # [T, hkv, d]
        mean = rows.mean(0).repeat_interleave(G, dim=0)
        err = (out[b].double() - mean).abs().max().item()
        assert err <= 2e-3 + 0.5 * torch.finfo(torch.bfloat16).eps * mean.abs().max().item()


def test_nondefault_stream(pkv_lib, oracle_lib):
    spec = config_spec(0, dtype=torch.float16, num_seqs=4, num_q_heads=8, num_kv_heads=2,
                       head_dim=128, lens=[100, 700, 33, 2000], explicit_pool=None,
                       lens_are_pre_append=False)
    w = make_workload(spec, device="cuda")
    mirror = HostMirror(w)
    _, ref = mirror.step(0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _, out = gpu_step(pkv_lib, w, 0, tokens_per_split=64, stream=s)
    s.synchronize()
    check_close(out, ref, spec.dtype)


def test_two_streams_concurrently(pkv_lib, oracle_lib):
    """Two workloads decoded at the same time on two streams, each with
    split-K partials (so each uses its own stream's workspace), launched
    interleaved for several rounds with no synchronisation between the
    streams: every round's outputs equal the oracle's and the pools end bit
    for bit as the oracle's."""
    ws, mirrors, refs = [], [], []
    for seed, dtype in ((11, torch.float16), (12, torch.bfloat16)):
        spec = config_spec(0, dtype=dtype, num_seqs=6, num_q_heads=8, num_kv_heads=2,
                           head_dim=128, lens=[1, 90, 700, 1500, 3000, 4097], explicit_pool=None,
                           lens_are_pre_append=False, seed=seed)
        w = make_workload(spec, device="cuda")
        mirror = HostMirror(w)
        _, ref = mirror.step(0)
        ws.append(w)
        mirrors.append(mirror)
        refs.append(ref)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    outs = []
    for _ in range(4):
        for i, st in enumerate(streams):
            with torch.cuda.stream(st):
                # the same step again: its append rewrites the same rows
                outs.append((i, gpu_step(pkv_lib, ws[i], 0, tokens_per_split=128, stream=st)[1]))
    torch.cuda.synchronize()
    for i, out in outs:
        check_close(out, refs[i], ws[i].spec.dtype)
    for w, mirror in zip(ws, mirrors):
        assert torch.equal(_bits(w.k_cache.cpu()), _bits(mirror.kc))
        assert torch.equal(_bits(w.v_cache.cpu()), _bits(mirror.vc))


# ---------------------------------------------------------------------------
# benchmark-size workloads: whole pool bit-exact after the append, and every
# output compared with the oracle (at these sizes the float64 oracle takes
# seconds on the host cores)


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_benchmark_workload(pkv_lib, oracle_lib, idx):
    spec = config_spec(idx)
    w = make_workload(spec, device="cuda", poison_outside_window=True)
    mirror = HostMirror(w)
    o_slots, ref = mirror.step(0)
    g_slots, out = gpu_step(pkv_lib, w, 0)
    torch.cuda.synchronize()
    assert np.array_equal(g_slots.cpu().numpy(), o_slots)
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(mirror.kc))
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(mirror.vc))
    # the long-context workloads' outputs are far below 1: the plain bound holds
    check_close(out, ref, spec.dtype, plain=(idx > 0))


def test_fused_benchmark_workload_all_outputs(pkv_lib, oracle_lib):
    """The benchmark's own launch (fused append + decode, the library's plan)
    on the GQA workload: the whole pool bit-exact and every output within the
    plain 2e-3 of the oracle."""
    spec = config_spec(2)
    w = make_workload(spec, device="cuda", poison_outside_window=True)
    mirror = HostMirror(w)
    _, ref = mirror.step(0)
    out = pkv_lib.pkv_append_decode(w.q_steps[0], w.k_steps[0], w.v_steps[0], w.k_cache,
                                    w.v_cache, w.block_tables, w.lens_steps[0].contiguous(),
                                    spec.window, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(mirror.kc))
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(mirror.vc))
    check_close(out, ref, spec.dtype, plain=True)


def test_serving_mix_32_steps(pkv_lib, oracle_lib):
    """All 32 append + decode steps of the serving mix; every output of 8
    steps spread over the run (first, last and six between) compared with the
    oracle, and the whole pool bit-exact at the end."""
    spec = config_spec(4)
    w = make_workload(spec, device="cuda")
    mirror = HostMirror(w)
    checked = {0, 4, 9, 13, 18, 22, 27, spec.steps - 1}
    for s in range(spec.steps):
        check = s in checked
        o_slots, ref = mirror.step(s, pairs=None if check else np.zeros((0, 2), np.int32))
        g_slots, out = gpu_step(pkv_lib, w, s)
        assert np.array_equal(g_slots.cpu().numpy(), o_slots)
        if check:
            torch.cuda.synchronize()
            check_close(out, ref, spec.dtype, plain=True)
    torch.cuda.synchronize()
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(mirror.kc))
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(mirror.vc))


@pytest.mark.parametrize("tps", [0, 64])
def test_decode_bf16_wide_range(pkv_lib, oracle_lib, tps):
    """bf16 pools whose (sequence, kv head) pairs each hold V at their own
    scale, 10^-30 .. 10^30, some with one value 10^12 above the rest (capped
    inside bf16's range): every output matches the oracle relative to its
    pair's scale (V stays bf16 in the decode's products; P is carried as hi +
    lo parts), with and without split contexts."""
    dtype = torch.bfloat16
    B, hq, hkv, d = 6, 16, 4, 128
    spec = config_spec(0, dtype=dtype, num_seqs=B, num_q_heads=hq, num_kv_heads=hkv,
                       head_dim=d, block_size=16, lens=[1, 17, 300, 777, 1500, 2100],
                       explicit_pool=None, lens_are_pre_append=False, seed=77)
    w = make_workload(spec, device="cuda", poison_outside_window=True)
    r = np.random.default_rng(78)
    bt = w.block_tables.cpu().numpy()
    lens = w.lens_steps[0].cpu().numpy()
    scale = np.ones((B, hkv))
    for b in range(B):
        sl = np.array([oracle.slot_for_position(bt[b], 16, t) for t in range(lens[b] - 1)],
                      np.int64)
        for h in range(hkv):
            s = 10.0 ** int(r.integers(-30, 31))
            scale[b, h] = s
            if sl.size:
                blk, row = torch.from_numpy(sl // 16).cuda(), torch.from_numpy(sl % 16).cuda()
                w.v_cache[blk, h, row] = (w.v_cache[blk, h, row].double() * s).to(dtype)
            w.v_steps[0][b, h] = (w.v_steps[0][b, h].double() * s).to(dtype)
            if sl.size and r.random() < 0.4:
                t = int(r.integers(0, sl.size))
                w.v_cache[sl[t] // 16, h, sl[t] % 16, int(r.integers(0, d))] = min(1e12 * s, 1e37)
    mirror = HostMirror(w)
    _, ref = mirror.step(0)
    _, out = gpu_step(pkv_lib, w, 0, tokens_per_split=tps)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    s = np.repeat(scale, hq // hkv, axis=1)[:, :, None]     # [B, Hq, 1]
    err = np.abs(got - ref) / s
    tol = 2e-3 + 0.5 * torch.finfo(dtype).eps * np.abs(ref) / s
    assert (err <= tol).all(), f"max scaled err {err.max():.3e}"
