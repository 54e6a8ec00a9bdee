"""Pins of the oracle's FP8 (E4M3) cache: the element format against torch's
float8_e4m3fn, round-to-nearest-even encoding, the per-row quantiser's closed
forms and error bound, and decode over a quantised pool against float64 SDPA
of the dequantised values.  ("Building a Memory-Compressed Attention Engine
with KV Caching", Extending, item 2: INT8 or FP8 quantisation of the cached
keys and values.)"""
import math

import numpy as np
import pytest
import torch

import oracle


def _torch_e4m3(codes):
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_decoder_all_codes(oracle_lib):
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    mine = oracle.e4m3_to_double(codes)
    ref = _torch_e4m3(codes)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))
    assert np.nanmax(mine) == 448.0 and np.nanmin(np.abs(mine[mine != 0])) == 2.0 ** -9


def test_e4m3_encoder_matches_torch_round_to_nearest_even(oracle_lib):
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_to_double(finite)
    order = np.argsort(vals)
    sv = np.unique(vals[order])
    mids = (sv[:-1] + sv[1:]) / 2                       # exact ties
    rng = np.random.default_rng(0)
    rand = rng.uniform(-448, 448, 20000)
    small = rng.uniform(-0.03, 0.03, 20000)             # subnormal range
    x = np.concatenate([sv, mids, rand, small]).astype(np.float32)
    mine = oracle.encode_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, f"first mismatches: {x[bad[:5]]} -> {mine[bad[:5]]} vs {ref[bad[:5]]}"


def test_e4m3_encoder_saturates(oracle_lib):
    codes = oracle.encode_e4m3(np.array([500.0, 1e30, -1e9, np.inf, -np.inf], np.float32))
    assert list(oracle.e4m3_to_double(codes)) == [448.0, 448.0, -448.0, 448.0, -448.0]


def test_quantize_row_closed_forms(oracle_lib):
    # representable values with absmax 448: scale 1, codes exact
    codes, scales = oracle.quantize_rows(np.array([[448, -224, 1, 0, -0.5, 2 ** -9]], np.float32))
    assert scales[0] == 1.0
    assert list(oracle.e4m3_to_double(codes[0])) == [448, -224, 1, 0, -0.5, 2 ** -9]
    # all-zero row: scale 1, zero codes
    codes, scales = oracle.quantize_rows(np.zeros((1, 8), np.float32))
    assert scales[0] == 1.0 and not oracle.e4m3_to_double(codes[0]).any()
    # a power-of-two rescaling keeps the codes and scales the scale
    x = np.random.default_rng(1).standard_normal((4, 64)).astype(np.float32)
    c1, s1 = oracle.quantize_rows(x)
    c2, s2 = oracle.quantize_rows(x * np.float32(8.0))
    assert np.array_equal(c1, c2) and np.array_equal(s2, s1 * 8)


def test_quantize_row_error_bound(oracle_lib):
    """Round to nearest: |x - code * scale| <= half the E4M3 spacing at x / scale
    (relative 2^-4 for normals, absolute 2^-10 * scale in the subnormal range)."""
    x = np.random.default_rng(2).standard_normal((200, 128)).astype(np.float32)
    codes, scales = oracle.quantize_rows(x)
    deq = oracle.e4m3_to_double(codes) * scales[:, None].astype(np.float64)
    y = np.abs(x.astype(np.float64) / scales[:, None])
    half_spacing = np.where(y >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(y, 1e-30))) - 4),
                            2.0 ** -10)
    err = np.abs(deq - x) / scales[:, None]
    assert (err <= half_spacing * (1 + 1e-6)).all()
    assert np.all(np.abs(oracle.e4m3_to_double(codes)).max(axis=1) == 448.0)


def test_decode_fp8_matches_sdpa_on_dequantized_values(oracle_lib):
    rng = np.random.default_rng(3)
    B, hq, hkv, d, bs = 3, 4, 2, 16, 4
    lens = [1, 9, 14]
    nb = 12
    perm = rng.permutation(nb)
    table = np.full((B, 4), -1, np.int32)
    kc = np.full((nb, hkv, bs, d), 0x7F, np.uint8)     # NaN codes outside the contexts
    vc = kc.copy()
    ksc = np.full((nb, hkv, bs), np.nan, np.float32)
    vsc = ksc.copy()
    logical = []
    cur = 0
    for b, L in enumerate(lens):
        n = -(-L // bs)
        table[b, :n] = perm[cur:cur + n]
        cur += n
        Kl = rng.integers(0, 0x7E, (L, hkv, d)).astype(np.uint8) | (rng.integers(0, 2, (L, hkv, d)) << 7).astype(np.uint8)
        Vl = rng.integers(0, 0x7E, (L, hkv, d)).astype(np.uint8)
        Ks = rng.uniform(0.001, 0.01, (L, hkv)).astype(np.float32)
        Vs = rng.uniform(0.001, 0.01, (L, hkv)).astype(np.float32)
        for t in range(L):
            kc[table[b, t // bs], :, t % bs] = Kl[t]
            vc[table[b, t // bs], :, t % bs] = Vl[t]
            ksc[table[b, t // bs], :, t % bs] = Ks[t]
            vsc[table[b, t // bs], :, t % bs] = Vs[t]
        logical.append((Kl, Vl, Ks, Vs))
    q = torch.randn(B, hq, d).to(torch.float16)
    for window, sinks in ((0, 0), (5, 2)):
        out = oracle.decode_fp8(q, kc, vc, ksc, vsc, table, np.array(lens, np.int32), window,
                                0.25, num_sinks=sinks)
        for b, L in enumerate(lens):
            Kl, Vl, Ks, Vs = logical[b]
            Kd = torch.from_numpy(_torch_e4m3(Kl) * Ks[..., None].astype(np.float64))
            Vd = torch.from_numpy(_torch_e4m3(Vl) * Vs[..., None].astype(np.float64))
            G = hq // hkv
            Kh = Kd.permute(1, 0, 2).repeat_interleave(G, 0)
            Vh = Vd.permute(1, 0, 2).repeat_interleave(G, 0)
            mask = None
            if window > 0:
                pos = torch.arange(L)
                mask = ((pos >= max(0, L - window)) | (pos < sinks)).view(1, 1, 1, L)
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[b].double().view(1, hq, 1, d), Kh[None], Vh[None], attn_mask=mask,
                scale=0.25).view(hq, d).numpy()
            np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_append_fp8_writes_quantised_rows(oracle_lib):
    rng = np.random.default_rng(4)
    nb, hkv, bs, d, T = 5, 2, 4, 32, 6
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = kc.copy()
    ks = np.zeros((nb, hkv, bs), np.float32)
    vs = ks.copy()
    k = torch.randn(T, hkv, d).to(torch.float16)
    v = torch.randn(T, hkv, d).to(torch.float16)
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int64)
    slots[2] = -1
    oracle.append_fp8(k, v, slots, kc, vc, ks, vs)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        blk, r = s // bs, s % bs
        for h in range(hkv):
            codes, scale = oracle.quantize_rows(k[i, h].float().numpy()[None])
            assert np.array_equal(kc[blk, h, r], codes[0]) and ks[blk, h, r] == scale[0]
            codes, scale = oracle.quantize_rows(v[i, h].float().numpy()[None])
            assert np.array_equal(vc[blk, h, r], codes[0]) and vs[blk, h, r] == scale[0]
    written = {(s // bs, s % bs) for s in slots if s >= 0}
    for blk in range(nb):
        for r in range(bs):
            if (blk, r) not in written:
                assert not kc[blk, :, r].any() and not ks[blk, :, r].any()
