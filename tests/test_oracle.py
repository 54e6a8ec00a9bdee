"""Pins of the float64 oracle against what the pages and the mathematics fix.

Every test here runs on the CPU.  None of them re-types the oracle's formula:
they check closed forms worked out by hand (tests/golden), a library routine
the definition reduces to (torch's float64 scaled_dot_product_attention on the
logical, contiguous sequence), brute force at 40 significant digits (mpmath),
exact decoders of the element formats, and invariants (block permutation,
window == truncation, GQA == replicated MHA).
"""
import json
import math
import os
import zlib

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def paged_from_logical(x_log, block_table, block_size, num_blocks, fill=np.nan):
    """Place logical tokens x_log [L, Hkv, D] into a head-major pool [NB, Hkv, bs, D]:
    token t goes to block block_table[t // bs], row t % bs (the page's layout)."""
    L, hkv, d = x_log.shape
    pool = np.full((num_blocks, hkv, block_size, d), fill, dtype=x_log.dtype)
    for t in range(L):
        pool[block_table[t // block_size], :, t % block_size, :] = x_log[t]
    return pool


# ---------------------------------------------------------------------------
# element decoders: every one of the 65536 bit patterns


def _same(a, b):
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(
        a[~np.isnan(a)], b[~np.isnan(b)]) and np.array_equal(
        np.signbit(a[~np.isnan(a)]), np.signbit(b[~np.isnan(b)]))


def test_f16_decoder_all_bit_patterns(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode_elements(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float64)
    assert _same(mine, ref)


def test_bf16_decoder_all_bit_patterns(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode_elements(bits, oracle.BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert _same(mine, ref)


def test_f32_decoder_is_exact(oracle_lib):
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.decode_elements(x, oracle.F32), x.astype(np.float64))


# ---------------------------------------------------------------------------
# hand-derived closed forms


CASES = _load("attention_closed_forms.json")["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_closed_form_cases(oracle_lib, case):
    d = len(case["q"])
    L = len(case["K"])
    K = np.asarray(case["K"], dtype=np.float32).reshape(L, 1, d)
    V = np.asarray(case["V"], dtype=np.float32).reshape(L, 1, d)
    bs, nb = case["block_size"], case["num_blocks"]
    table = np.full((1, max(1, len(case["block_table"]))), -1, dtype=np.int32)
    table[0, :len(case["block_table"])] = case["block_table"]
    kc = paged_from_logical(K, table[0], bs, nb)
    vc = paged_from_logical(V, table[0], bs, nb)
    q = np.asarray(case["q"], dtype=np.float32).reshape(1, 1, d)
    out = oracle.decode(q, kc, vc, table, np.array([L], np.int32), case["window"], case["scale"],
                        num_sinks=case.get("sinks", 0))
    np.testing.assert_allclose(out[0, 0], case["expected"], rtol=0, atol=case["tol"])


def test_attend_contiguous_two_tokens(oracle_lib):
    # the contiguous form of the first closed form
    c = CASES[0]
    out = oracle.attend(np.array(c["q"]), np.array(c["K"]), np.array(c["V"]), c["scale"])
    np.testing.assert_allclose(out, c["expected"], atol=c["tol"], rtol=0)


# ---------------------------------------------------------------------------
# the definition reduces to a library routine on the logical sequence


def _random_problem(rng, B, hq, hkv, d, bs, lens, dtype, nb_extra=3):
    """Random logical K/V per sequence, placed through a shuffled block pool."""
    need = [(L + bs - 1) // bs for L in lens]
    nb = sum(need) + nb_extra
    perm = rng.permutation(nb)
    mb = max(max(need), 1)
    table = np.full((B, mb), -1, dtype=np.int32)
    kc = np.full((nb, hkv, bs, d), np.nan, dtype=np.float32)
    vc = np.full((nb, hkv, bs, d), np.nan, dtype=np.float32)
    logical = []
    cur = 0
    for b, L in enumerate(lens):
        table[b, :need[b]] = perm[cur:cur + need[b]]
        cur += need[b]
        Kl = rng.standard_normal((L, hkv, d)).astype(np.float32)
        Vl = rng.standard_normal((L, hkv, d)).astype(np.float32)
        for t in range(L):
            kc[table[b, t // bs], :, t % bs] = Kl[t]
            vc[table[b, t // bs], :, t % bs] = Vl[t]
        logical.append((Kl, Vl))
    q = rng.standard_normal((B, hq, d)).astype(np.float32)
    to = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    qt, kt, vt = (torch.from_numpy(a).to(to) for a in (q, kc, vc))
    # logical data as the dtype sees it (exactly widened to float64 by torch)
    logical_t = [(torch.from_numpy(Kl).to(to).double(), torch.from_numpy(Vl).to(to).double())
                 for Kl, Vl in logical]
    return qt, kt, vt, table, logical_t


def _sdpa_reference(q_b, Kl, Vl, G, window, scale, sinks=0):
    """torch float64 SDPA of one sequence: q_b [Hq, D], Kl/Vl [L, Hkv, D]."""
    L = Kl.shape[0]
    hq, d = q_b.shape
    if L == 0:
        return torch.zeros(hq, d, dtype=torch.float64)
    Kh = Kl.permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, D]
    Vh = Vl.permute(1, 0, 2).repeat_interleave(G, dim=0)
    mask = None
    if window > 0:
        pos = torch.arange(L)
        mask = (pos >= max(0, L - window)) | (pos < sinks)
        mask = mask.view(1, 1, 1, L)
    out = torch.nn.functional.scaled_dot_product_attention(
        q_b.view(1, hq, 1, d), Kh.unsqueeze(0), Vh.unsqueeze(0), attn_mask=mask, scale=scale)
    return out.view(hq, d)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("hq,hkv,window,bs,sinks", [(4, 4, 0, 4, 0), (8, 2, 0, 8, 0),
                                                     (6, 2, 5, 4, 0), (4, 1, 3, 16, 0),
                                                     (3, 3, 100, 2, 0), (4, 2, 6, 4, 4),
                                                     (2, 1, 9, 8, 2), (4, 4, 0, 4, 3)])
def test_matches_torch_sdpa(oracle_lib, dtype, hq, hkv, window, bs, sinks):
    rng = np.random.default_rng(zlib.crc32(repr((dtype, hq, hkv, window, bs)).encode()))
    lens = [1, 7, 13, 0, 29]
    d = 16
    scale = float(np.float32(1 / math.sqrt(d)))
    q, kc, vc, table, logical = _random_problem(rng, len(lens), hq, hkv, d, bs, lens, dtype)
    out = oracle.decode(q, kc, vc, table, np.array(lens, np.int32), window, scale,
                        num_sinks=sinks)
    for b, L in enumerate(lens):
        ref = _sdpa_reference(q[b].double(), *logical[b], hq // hkv, window, scale,
                              sinks).numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# invariants


def test_block_permutation_invariance(oracle_lib):
    """The same logical sequences through two different block assignments give
    bit-identical results (the order of summation does not depend on layout)."""
    rng = np.random.default_rng(7)
    lens = [5, 33, 64, 17]
    q, kc, vc, table, logical = _random_problem(rng, 4, 4, 2, 8, 8, lens, "f32")
    out1 = oracle.decode(q, kc, vc, table, np.array(lens, np.int32), 0, 0.3)
    rng2 = np.random.default_rng(8)
    need = [(L + 7) // 8 for L in lens]
    nb2 = sum(need) + 11
    perm = rng2.permutation(nb2)
    table2 = np.full_like(table, -1)
    kc2 = np.full((nb2, 2, 8, 8), np.nan, np.float32)
    vc2 = np.full_like(kc2, np.nan)
    cur = 0
    for b, L in enumerate(lens):
        table2[b, :need[b]] = perm[cur:cur + need[b]]
        cur += need[b]
        Kl, Vl = (x.float().numpy() for x in logical[b])
        for t in range(L):
            kc2[table2[b, t // 8], :, t % 8] = Kl[t]
            vc2[table2[b, t // 8], :, t % 8] = Vl[t]
    out2 = oracle.decode(q, kc2, vc2, table2, np.array(lens, np.int32), 0, 0.3)
    assert np.array_equal(out1, out2)
    assert not np.isnan(out1).any()  # poisoned slots were never read


def test_window_equals_truncated_cache(oracle_lib):
    rng = np.random.default_rng(3)
    lens = [40, 41, 9]
    w = 11
    q, kc, vc, table, logical = _random_problem(rng, 3, 2, 2, 8, 4, lens, "f32")
    out_w = oracle.decode(q, kc, vc, table, np.array(lens, np.int32), w, 0.25)
    for b, L in enumerate(lens):
        keep = min(w, L)
        Kl, Vl = (x.float().numpy()[L - keep:] for x in logical[b])
        tab = np.arange((keep + 3) // 4, dtype=np.int32)[None, :]
        k2 = paged_from_logical(Kl, tab[0], 4, tab.shape[1])
        v2 = paged_from_logical(Vl, tab[0], 4, tab.shape[1])
        ref = oracle.decode(q[b:b + 1], k2, v2, tab, np.array([keep], np.int32), 0, 0.25)
        assert np.array_equal(out_w[b], ref[0])


def test_gqa_equals_replicated_mha(oracle_lib):
    rng = np.random.default_rng(11)
    lens = [19, 3]
    q, kc, vc, table, logical = _random_problem(rng, 2, 6, 2, 8, 4, lens, "f32")
    out = oracle.decode(q, kc, vc, table, np.array(lens, np.int32), 0, 0.5)
    # MHA pool whose kv head h holds the data of GQA kv head h // 3
    kc_m = np.repeat(kc.numpy(), 3, axis=1)
    vc_m = np.repeat(vc.numpy(), 3, axis=1)
    out_m = oracle.decode(q, kc_m, vc_m, table, np.array(lens, np.int32), 0, 0.5)
    assert np.array_equal(out, out_m)


def test_uniform_keys_give_mean_of_window(oracle_lib):
    rng = np.random.default_rng(5)
    L, w, d = 50, 20, 16
    K = np.tile(rng.standard_normal((1, 1, d)).astype(np.float32), (L, 1, 1))
    V = rng.standard_normal((L, 1, d)).astype(np.float32)
    tab = rng.permutation(13)[:13].astype(np.int32)[None, :]
    kc = paged_from_logical(K, tab[0], 4, 13)
    vc = paged_from_logical(V, tab[0], 4, 13)
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    out = oracle.decode(q, kc, vc, tab, np.array([L], np.int32), w, 0.7)
    np.testing.assert_allclose(out[0, 0], V[L - w:, 0].astype(np.float64).mean(0), atol=1e-13)


# ---------------------------------------------------------------------------
# brute force at 40 digits


def test_bruteforce_mpmath(oracle_lib):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    rng = np.random.default_rng(17)
    for trial in range(20):
        L = int(rng.integers(1, 6))
        d = 3
        w = int(rng.integers(0, 6))
        scale = float(rng.uniform(0.1, 2.0))
        K = rng.standard_normal((L, 1, d)).astype(np.float32)
        V = rng.standard_normal((L, 1, d)).astype(np.float32)
        q = rng.standard_normal((1, 1, d)).astype(np.float32)
        tab = rng.permutation(4).astype(np.int32)[None, :]
        kc = paged_from_logical(K, tab[0], 2, 4)
        vc = paged_from_logical(V, tab[0], 2, 4)
        out = oracle.decode(q, kc, vc, tab, np.array([L], np.int32), w, scale)[0, 0]
        lo = max(0, L - w) if w > 0 else 0
        s = [mp.mpf(scale) * mp.fsum(mp.mpf(float(q[0, 0, i])) * mp.mpf(float(K[t, 0, i]))
                                     for i in range(d)) for t in range(lo, L)]
        e = [mp.e ** x for x in s]  # no max-subtraction: exact arithmetic needs none
        z = mp.fsum(e)
        ref = [mp.fsum(e[j] * mp.mpf(float(V[lo + j, 0, i])) for j in range(len(e))) / z
               for i in range(d)]
        for i in range(d):
            assert abs(out[i] - float(ref[i])) <= 1e-14 * max(1.0, abs(float(ref[i])))


# ---------------------------------------------------------------------------
# append and slot mapping ("Build a Paged KV Cache in Pure Python", Step 3)


def test_slot_mapping_example(oracle_lib):
    ex = _load("p2_allocator_and_slots.json")["slot_mapping_example"]
    got = [oracle.slot_for_position(ex["block_table"], ex["block_size"], p)
           for p in ex["positions"]]
    assert got == ex["slots"]


def test_append_35_tokens_across_blocks(oracle_lib):
    """The page's append/retrieve test: 35 tokens, block_size 16, 8 heads x 64."""
    g = _load("p2_allocator_and_slots.json")["append_retrieve"]
    bs, h, d, n = g["block_size"], g["num_heads"], g["head_dim"], g["tokens"]
    rng = np.random.default_rng(0)
    nb = g["total_blocks"]
    table = rng.permutation(nb)[:g["blocks_used"]].astype(np.int32)
    kc = np.full((nb, h, bs, d), np.nan, np.float32)
    vc = np.full_like(kc, np.nan)
    K = rng.standard_normal((n, h, d)).astype(np.float32)
    V = rng.standard_normal((n, h, d)).astype(np.float32)
    for pos in range(n):  # one append per token, like the page's loop
        slot = oracle.slot_for_position(table, bs, pos)
        oracle.append(K[pos:pos + 1], V[pos:pos + 1], np.array([slot]), kc, vc)
    # retrieve: the blocks in list order, min(bs, n - start) rows each
    rows = np.concatenate([kc[table[j], :, :min(bs, n - j * bs)].transpose(1, 0, 2)
                           for j in range(len(table))])
    assert rows.shape == (g["retrieved_tokens"], h, d)
    assert np.array_equal(rows, K)
    # nothing else was written
    mask = np.ones(nb * bs, bool)
    for pos in range(n):
        mask[oracle.slot_for_position(table, bs, pos)] = False
    flat = kc.transpose(0, 2, 1, 3).reshape(nb * bs, h, d)
    assert np.isnan(flat[mask]).all()


def test_append_bit_copy_and_skips(oracle_lib):
    rng = np.random.default_rng(2)
    nb, hkv, bs, d, T = 6, 3, 4, 8, 9
    kc = torch.randn(nb, hkv, bs, d).to(torch.bfloat16)
    vc = torch.randn(nb, hkv, bs, d).to(torch.bfloat16)
    k0, v0 = kc.clone(), vc.clone()
    k = torch.randn(T, hkv, d).to(torch.bfloat16)
    v = torch.randn(T, hkv, d).to(torch.bfloat16)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[[1, 5]] = -1
    oracle.append(k, v, slots, kc, vc)
    kb, vb = kc.view(torch.int16), vc.view(torch.int16)
    touched = np.zeros((nb, bs), bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        touched[s // bs, s % bs] = True
        assert torch.equal(kb[s // bs, :, s % bs], k.view(torch.int16)[i])
        assert torch.equal(vb[s // bs, :, s % bs], v.view(torch.int16)[i])
    t = torch.from_numpy(touched)
    assert torch.equal(kc.view(torch.int16).permute(0, 2, 1, 3)[~t],
                       k0.view(torch.int16).permute(0, 2, 1, 3)[~t])
    assert torch.equal(vc.view(torch.int16).permute(0, 2, 1, 3)[~t],
                       v0.view(torch.int16).permute(0, 2, 1, 3)[~t])


def test_invalid_block_id_is_reported(oracle_lib):
    kc = np.zeros((2, 1, 2, 4), np.float32)
    table = np.array([[0, 7]], np.int32)
    out = oracle.decode(np.ones((1, 1, 4), np.float32), kc, kc, table, np.array([3], np.int32),
                        0, 1.0, check=False)
    assert np.isnan(out).all()
    with pytest.raises(ValueError):
        oracle.decode(np.ones((1, 1, 4), np.float32), kc, kc, table, np.array([3], np.int32),
                      0, 1.0)
