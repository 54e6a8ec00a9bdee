"""Pins of the oracle's INT8 cache: the per-row quantiser's closed forms, its
round-to-nearest-even rule and error bound, the same quantity computed with
torch's float32 arithmetic, the append into INT8 pools, and decode over a
quantised pool against float64 SDPA of the dequantised values.
("Building a Memory-Compressed Attention Engine with KV Caching", Extending,
item 2: INT8 or FP8 quantisation of the cached keys and values.)"""
import numpy as np
import torch

import oracle


def test_quantize_int8_closed_forms(oracle_lib):
    # absmax 127: scale 1, codes are the values rounded to nearest, ties to even
    row = np.array([[127, 0.5, 1.5, 2.5, -0.5, -1.5, -126.4, 3.0]], np.float32)
    codes, scales = oracle.quantize_rows_int8(row)
    assert scales[0] == 1.0
    assert list(codes[0]) == [127, 0, 2, 2, 0, -2, -126, 3]
    # all-zero row: scale 1, zero codes
    codes, scales = oracle.quantize_rows_int8(np.zeros((1, 8), np.float32))
    assert scales[0] == 1.0 and not codes[0].any()
    # the absmax element always gets +-127 and -128 is never produced
    rng = np.random.default_rng(1)
    x = rng.standard_normal((200, 64)).astype(np.float32)
    codes, _ = oracle.quantize_rows_int8(x)
    am = np.abs(x).argmax(axis=1)
    assert np.array_equal(np.abs(codes[np.arange(200), am]), np.full(200, 127))
    assert codes.min() >= -127
    # scaling a row by a power of two keeps its codes and scales its scale
    c2, s2 = oracle.quantize_rows_int8(x * 8)
    c1, s1 = oracle.quantize_rows_int8(x)
    assert np.array_equal(c1, c2) and np.array_equal(s2, s1 * 8)


def test_quantize_int8_matches_float32_torch(oracle_lib):
    """The same definition in torch's float32 ops: scale = absmax / 127,
    code = round_half_even(x * (127 / absmax)) clamped to [-127, 127]."""
    rng = np.random.default_rng(2)
    rows = np.concatenate([
        rng.standard_normal((300, 128)),
        rng.uniform(-1e-30, 1e-30, (50, 128)),
        rng.uniform(-6e4, 6e4, (50, 128)),
    ]).astype(np.float32)
    codes, scales = oracle.quantize_rows_int8(rows)
    x = torch.from_numpy(rows)
    absmax = x.abs().amax(dim=1, keepdim=True)
    ref_scale = absmax / torch.tensor(127.0)
    inv = torch.tensor(127.0) / absmax
    ref_codes = torch.round(x * inv).clamp(-127, 127).to(torch.int8)
    assert np.array_equal(scales, ref_scale[:, 0].numpy())
    assert np.array_equal(codes, ref_codes.numpy())


def test_quantize_int8_error_bound(oracle_lib):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((500, 64)) * rng.uniform(1e-3, 1e3, (500, 1))).astype(np.float32)
    codes, scales = oracle.quantize_rows_int8(x)
    err = np.abs(codes.astype(np.float64) * scales[:, None].astype(np.float64) - x)
    # half a step, with room for the two float32 roundings of scale and x / scale
    assert (err <= scales[:, None] * (0.5 + 1e-5)).all()


def test_decode_int8_matches_sdpa_on_dequantized_values(oracle_lib):
    rng = np.random.default_rng(5)
    B, hq, hkv, d, bs = 3, 4, 2, 16, 4
    lens = [1, 9, 14]
    nb = 12
    perm = rng.permutation(nb)
    table = np.full((B, 4), -1, np.int32)
    kc = np.full((nb, hkv, bs, d), -128, np.int8)       # never-produced code outside contexts
    vc = kc.copy()
    ksc = np.full((nb, hkv, bs), np.nan, np.float32)
    vsc = ksc.copy()
    logical = []
    cur = 0
    for b, L in enumerate(lens):
        n = -(-L // bs)
        table[b, :n] = perm[cur:cur + n]
        cur += n
        Kl = rng.integers(-127, 128, (L, hkv, d)).astype(np.int8)
        Vl = rng.integers(-127, 128, (L, hkv, d)).astype(np.int8)
        Ks = rng.uniform(0.001, 0.03, (L, hkv)).astype(np.float32)
        Vs = rng.uniform(0.001, 0.03, (L, hkv)).astype(np.float32)
        for t in range(L):
            kc[table[b, t // bs], :, t % bs] = Kl[t]
            vc[table[b, t // bs], :, t % bs] = Vl[t]
            ksc[table[b, t // bs], :, t % bs] = Ks[t]
            vsc[table[b, t // bs], :, t % bs] = Vs[t]
        logical.append((Kl, Vl, Ks, Vs))
    q = torch.randn(B, hq, d).to(torch.float16)
    for window, sinks in ((0, 0), (5, 2)):
        out = oracle.decode_int8(q, kc, vc, ksc, vsc, table, np.array(lens, np.int32), window,
                                 0.25, num_sinks=sinks)
        for b, L in enumerate(lens):
            Kl, Vl, Ks, Vs = logical[b]
            Kd = torch.from_numpy(Kl.astype(np.float64) * Ks[..., None].astype(np.float64))
            Vd = torch.from_numpy(Vl.astype(np.float64) * Vs[..., None].astype(np.float64))
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


def test_append_int8_writes_quantised_rows(oracle_lib):
    rng = np.random.default_rng(4)
    nb, hkv, bs, d, T = 5, 2, 4, 32, 6
    kc = np.zeros((nb, hkv, bs, d), np.int8)
    vc = kc.copy()
    ks = np.zeros((nb, hkv, bs), np.float32)
    vs = ks.copy()
    k = torch.randn(T, hkv, d).to(torch.bfloat16)
    v = torch.randn(T, hkv, d).to(torch.bfloat16)
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int64)
    slots[3] = -1
    oracle.append_int8(k, v, slots, kc, vc, ks, vs)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        blk, r = s // bs, s % bs
        for h in range(hkv):
            codes, scale = oracle.quantize_rows_int8(k[i, h].float().numpy()[None])
            assert np.array_equal(kc[blk, h, r], codes[0]) and ks[blk, h, r] == scale[0]
            codes, scale = oracle.quantize_rows_int8(v[i, h].float().numpy()[None])
            assert np.array_equal(vc[blk, h, r], codes[0]) and vs[blk, h, r] == scale[0]
    written = {(s // bs, s % bs) for s in slots if s >= 0}
    for blk in range(nb):
        for r in range(bs):
            if (blk, r) not in written:
                assert not kc[blk, :, r].any() and not ks[blk, :, r].any()
