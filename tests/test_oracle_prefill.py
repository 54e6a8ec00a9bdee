"""Pins of the oracle's paged (chunked) prefill: the sliding-window causal mask
of "Building a Streaming Sliding-Window Attention Engine in Pure Python",
Step 3 (prefill_attention: (i - j) < window and j <= i, softmax per row),
against torch's float64 SDPA with that mask on the logical sequence, and a
closed form (uniform keys -> mean of V over each row's attended range)."""
import math

import numpy as np
import pytest
import torch

import oracle


def _paged(seqs_k, seqs_v, bs, rng, extra=5):
    """Place per-sequence logical K/V [L, Hkv, D] into a shuffled head-major pool."""
    need = [-(-k.shape[0] // bs) for k in seqs_k]
    nb = sum(need) + extra
    perm = rng.permutation(nb)
    hkv, d = seqs_k[0].shape[1:]
    table = np.full((len(seqs_k), max(max(need), 1)), -1, np.int32)
    kc = torch.full((nb, hkv, bs, d), float("nan"), dtype=seqs_k[0].dtype)
    vc = kc.clone()
    cur = 0
    for b, (K, V) in enumerate(zip(seqs_k, seqs_v)):
        table[b, :need[b]] = perm[cur:cur + need[b]]
        cur += need[b]
        for t in range(K.shape[0]):
            kc[table[b, t // bs], :, t % bs] = K[t]
            vc[table[b, t // bs], :, t % bs] = V[t]
    return kc, vc, table


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("hq,hkv,window,bs,sinks", [(4, 4, 0, 4, 0), (8, 2, 0, 8, 0),
                                                     (4, 2, 6, 4, 0), (2, 1, 1, 16, 0),
                                                     (4, 2, 6, 4, 3), (2, 1, 1, 16, 1),
                                                     (4, 4, 4, 8, 7), (8, 2, 2, 4, 30)])
def test_prefill_matches_sdpa_with_causal_window_mask(oracle_lib, dtype, hq, hkv, window, bs,
                                                      sinks):
    """Mask of query position p over key j: j <= p, and with a window
    (p - j < window or j < sinks) -- the window of Step 3 plus the sink
    positions of the StreamingLLM item."""
    rng = np.random.default_rng(hq * 100 + hkv * 10 + window + bs + 1000 * sinks)
    d = 16
    lens = [9, 23, 5]          # lengths after the chunk
    chunks = [9, 7, 3]         # first sequence: pure prefill; others: cached prefix + chunk
    Ks = [torch.randn(L, hkv, d).to(dtype) for L in lens]
    Vs = [torch.randn(L, hkv, d).to(dtype) for L in lens]
    kc, vc, table = _paged(Ks, Vs, bs, rng)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = torch.randn(int(cu[-1]), hq, d).to(dtype)
    scale = float(np.float32(1 / math.sqrt(d)))
    out = oracle.prefill(q, cu, kc, vc, table, np.array(lens, np.int32), window, scale,
                         num_sinks=sinks)
    G = hq // hkv
    for b, (L, n) in enumerate(zip(lens, chunks)):
        pos = torch.arange(L - n, L)                       # query positions
        key = torch.arange(L)
        mask = key[None, :] <= pos[:, None]
        if window > 0:
            mask &= ((pos[:, None] - key[None, :]) < window) | (key[None, :] < sinks)
        Kh = Ks[b].double().permute(1, 0, 2).repeat_interleave(G, 0)
        Vh = Vs[b].double().permute(1, 0, 2).repeat_interleave(G, 0)
        qb = q[cu[b]:cu[b + 1]].double().permute(1, 0, 2)  # [Hq, n, D]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qb[None], Kh[None], Vh[None], attn_mask=mask[None, None], scale=scale)[0]
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=1e-12, atol=1e-12)


def test_prefill_uniform_keys_closed_form(oracle_lib):
    rng = np.random.default_rng(0)
    L, n, w, d = 12, 6, 4, 8
    K = torch.ones(L, 1, d) * 0.5
    V = torch.randn(L, 1, d)
    kc, vc, table = _paged([K], [V], 4, rng)
    q = torch.randn(n, 1, d)
    out = oracle.prefill(q, np.array([0, n], np.int32), kc, vc, table, np.array([L], np.int32),
                         w, 0.3)
    for i in range(n):
        p = L - n + i
        lo = max(0, p - w + 1)
        np.testing.assert_allclose(out[i, 0], V[lo:p + 1, 0].double().mean(0).numpy(),
                                   atol=1e-13)


def test_prefill_sinks_uniform_keys_closed_form(oracle_lib):
    """Equal keys: each row is the mean of V over its sinks and its window."""
    rng = np.random.default_rng(1)
    L, n, w, sinks, d = 20, 9, 3, 4, 8
    K = torch.ones(L, 1, d) * 0.25
    V = torch.randn(L, 1, d)
    kc, vc, table = _paged([K], [V], 4, rng)
    q = torch.randn(n, 1, d)
    out = oracle.prefill(q, np.array([0, n], np.int32), kc, vc, table, np.array([L], np.int32),
                         w, 0.7, num_sinks=sinks)
    for i in range(n):
        p = L - n + i
        keys = sorted(set(range(min(sinks, p + 1))) | set(range(max(0, p - w + 1), p + 1)))
        np.testing.assert_allclose(out[i, 0], V[keys, 0].double().mean(0).numpy(), atol=1e-13)


def test_prefill_sinks_without_window_change_nothing(oracle_lib):
    """Sinks only act with a window: window 0 attends every earlier position."""
    rng = np.random.default_rng(2)
    K, V = torch.randn(30, 2, 8), torch.randn(30, 2, 8)
    kc, vc, table = _paged([K], [V], 8, rng)
    q = torch.randn(10, 4, 8)
    args = (q, np.array([0, 10], np.int32), kc, vc, table, np.array([30], np.int32), 0, 0.35)
    np.testing.assert_array_equal(oracle.prefill(*args), oracle.prefill(*args, num_sinks=5))
