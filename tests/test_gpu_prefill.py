"""pkv_prefill (chunked prefill over the paged cache) against the oracle: the
chunk's rows land bit-exactly in their slots, and every query row's output is
within the fp16 / bf16 tolerance of the oracle's prefill."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_24_gb300.workloads import config_spec, make_workload

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16)


def _prefill_case(dtype, hq, hkv, d, bs, prefixes, chunks, window, seed):
    """Pools holding each sequence's prefix (everything else NaN) and the packed chunk."""
    lens = [p + n for p, n in zip(prefixes, chunks)]
    spec = config_spec(0, dtype=dtype, num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv,
                       head_dim=d, block_size=bs, lens=lens, explicit_pool=None,
                       lens_are_pre_append=False, window=0, seed=seed)
    w = make_workload(spec, device="cuda")
    bt = w.block_tables.cpu().numpy()
    # positions prefix .. L-1 belong to the chunk: poison them before the call
    kc, vc = w.k_cache, w.v_cache
    for b, (p, L) in enumerate(zip(prefixes, lens)):
        for t in range(p, L):
            s = oracle.slot_for_position(bt[b], bs, t)
            kc[s // bs, :, s % bs] = float("nan")
            vc[s // bs, :, s % bs] = float("nan")
    g = torch.Generator(device="cuda").manual_seed(seed + 7)
    T = sum(chunks)
    q = torch.randn(T, hq, d, generator=g, device="cuda").to(dtype)
    k = torch.randn(T, hkv, d, generator=g, device="cuda").to(dtype)
    v = torch.randn(T, hkv, d, generator=g, device="cuda").to(dtype)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32, device="cuda")
    return w, q, k, v, cu, torch.tensor(lens, dtype=torch.int32, device="cuda")


def _oracle_prefill(w, q, k, v, cu, lens, chunks, window):
    kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
    bt = w.block_tables.cpu().numpy()
    cu_h, lens_h = cu.cpu().numpy(), lens.cpu().numpy()
    slots = []
    for b, n in enumerate(chunks):
        for i in range(n):
            slots.append(oracle.slot_for_position(bt[b], w.spec.block_size, lens_h[b] - n + i))
    oracle.append(k.cpu(), v.cpu(), np.array(slots, np.int64), kc, vc)
    out = oracle.prefill(q.cpu(), cu_h, kc, vc, bt, lens_h, window, w.scale)
    return out, kc, vc


CASES = [
    # name, dtype, hq, hkv, d, bs, prefixes, chunks, window
    ("mha_pure", torch.float16, 4, 4, 128, 16, [0, 0, 0], [1, 70, 129], 0),
    ("mha_chunked", torch.float16, 4, 4, 128, 16, [15, 300, 2], [17, 64, 200], 0),
    ("gqa4_bs32", torch.bfloat16, 8, 2, 128, 32, [0, 33, 500], [50, 31, 100], 0),
    ("gqa8", torch.bfloat16, 8, 1, 128, 16, [7, 100], [9, 40], 0),
    ("g6_chunks", torch.float16, 12, 2, 128, 16, [20, 0], [13, 30], 0),
    ("g32", torch.bfloat16, 32, 1, 128, 16, [40, 5], [11, 6], 0),
    ("d64", torch.bfloat16, 8, 4, 64, 16, [3, 90], [60, 45], 0),
    ("window37", torch.bfloat16, 8, 2, 128, 16, [0, 100, 7], [80, 50, 30], 37),
    ("window1", torch.float16, 4, 4, 128, 16, [5, 0], [20, 33], 1),
    ("window_large", torch.float16, 4, 2, 128, 16, [10, 60], [30, 20], 5000),
    # rows whose first key tiles are wholly outside their window
    ("window5_long", torch.bfloat16, 4, 4, 128, 16, [0, 200], [300, 260], 5),
    ("window16_d64", torch.float16, 8, 2, 64, 16, [100], [500], 16),
    # many key tiles, several CTAs per (sequence, kv head)
    ("long_prefix", torch.bfloat16, 8, 2, 128, 16, [3000, 1], [300, 700], 0),
    ("long_prefix_fp16", torch.float16, 16, 2, 128, 32, [2047], [513], 0),
]
# more (sequence, token chunk) work items than the planner's block has threads,
# of many different sizes, so its counting sort loops and fills many bins
_r = np.random.default_rng(29)
CASES.append(("many_seqs", torch.float16, 8, 2, 128, 16, _r.integers(0, 600, 300).tolist(),
              _r.integers(1, 140, 300).tolist(), 0))
# the largest batch the prefill takes (65534 sequences): one work item each,
# prefixes from empty up
CASES.append(("max_sequences", torch.float16, 2, 1, 64, 16, _r.integers(0, 40, 65534).tolist(),
              _r.integers(1, 4, 65534).tolist(), 0))
# more than 1024 work items (16 tokens per CTA at 16 query heads per kv head):
# the planner sizes the items past its per-thread register cache twice
CASES.append(("many_items", torch.bfloat16, 16, 1, 128, 16, _r.integers(0, 300, 90).tolist(),
              [199] + _r.integers(1, 200, 89).tolist(), 0))


@pytest.mark.parametrize("name,dtype,hq,hkv,d,bs,prefixes,chunks,window", CASES,
                         ids=[c[0] for c in CASES])
def test_prefill_matches_oracle(pkv_lib, oracle_lib, name, dtype, hq, hkv, d, bs, prefixes,
                                chunks, window):
    w, q, k, v, cu, lens = _prefill_case(dtype, hq, hkv, d, bs, prefixes, chunks, window,
                                         seed=len(name))
    ref, kc_h, vc_h = _oracle_prefill(w, q, k, v, cu, lens, chunks, window)
    # every row must be written: a work item left out would leave NaN behind
    out = torch.full_like(q, float("nan"))
    pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, lens, window,
                        w.scale, max_chunk=max(chunks), out=out)
    torch.cuda.synchronize()
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(kc_h))
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(vc_h))
    g = out.double().cpu().numpy()
    assert not np.isnan(g).any()
    err = np.abs(g - ref)
    tol = 2e-3 + 0.5 * torch.finfo(dtype).eps * np.abs(ref)
    assert (err <= tol).all(), f"max err {err.max():.3e}"


SINK_CASES = [
    # name, dtype, hq, hkv, d, bs, prefixes, chunks, window, sinks
    ("w37_s4", torch.bfloat16, 8, 2, 128, 16, [0, 100, 7], [80, 50, 30], 37, 4),
    # more sinks than the window, not a whole unit
    ("w5_s20_long", torch.bfloat16, 4, 4, 128, 16, [0, 200], [300, 260], 5, 20),
    ("w16_s16_d64", torch.float16, 8, 2, 64, 16, [100], [500], 16, 16),
    # sinks reaching into the window of the chunk's first rows
    ("w100_s150_bs32", torch.float16, 8, 2, 128, 32, [400, 10], [300, 200], 100, 150),
    ("w1_s1", torch.float16, 4, 4, 128, 16, [5, 0], [20, 33], 1, 1),
    # the sink tile far ahead of the window tiles
    ("w300_s3_far", torch.bfloat16, 16, 2, 128, 16, [3000], [700], 300, 3),
    ("w2000_s7_g4", torch.bfloat16, 8, 2, 128, 16, [3000, 1], [300, 700], 2000, 7),
    ("w64_s130_g8", torch.float16, 16, 2, 128, 16, [900, 129], [200, 64], 64, 130),
]


def _poison_unattended(w, prefixes, chunks, window, sinks):
    """NaN into every prefix slot no chunk row attends: past the sinks and
    before the first chunk row's window."""
    bs = w.spec.block_size
    bt = w.block_tables.cpu().numpy()
    slots = []
    for b, (p, n) in enumerate(zip(prefixes, chunks)):
        first_lo = max(0, p - window + 1)
        slots += [oracle.slot_for_position(bt[b], bs, t) for t in range(sinks, first_lo)]
    if slots:
        s = np.array(slots, np.int64)
        blk = torch.from_numpy(s // bs).to("cuda")
        row = torch.from_numpy(s % bs).to("cuda")
        w.k_cache[blk, :, row] = float("nan")
        w.v_cache[blk, :, row] = float("nan")


@pytest.mark.parametrize("name,dtype,hq,hkv,d,bs,prefixes,chunks,window,sinks", SINK_CASES,
                         ids=[c[0] for c in SINK_CASES])
def test_prefill_with_sinks_matches_oracle(pkv_lib, oracle_lib, name, dtype, hq, hkv, d, bs,
                                           prefixes, chunks, window, sinks):
    w, q, k, v, cu, lens = _prefill_case(dtype, hq, hkv, d, bs, prefixes, chunks, window,
                                         seed=len(name) + 100)
    _poison_unattended(w, prefixes, chunks, window, sinks)
    kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
    bt = w.block_tables.cpu().numpy()
    lens_h = lens.cpu().numpy()
    slots = [oracle.slot_for_position(bt[b], bs, lens_h[b] - n + i)
             for b, n in enumerate(chunks) for i in range(n)]
    oracle.append(k.cpu(), v.cpu(), np.array(slots, np.int64), kc, vc)
    ref = oracle.prefill(q.cpu(), cu.cpu().numpy(), kc, vc, bt, lens_h, window, w.scale,
                         num_sinks=sinks)
    out = torch.full_like(q, float("nan"))
    pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, lens, window,
                        w.scale, max_chunk=max(chunks), out=out, num_sinks=sinks)
    torch.cuda.synchronize()
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(kc))
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(vc))
    g = out.double().cpu().numpy()
    assert not np.isnan(g).any()
    err = np.abs(g - ref)
    tol = 2e-3 + 0.5 * torch.finfo(dtype).eps * np.abs(ref)
    assert (err <= tol).all(), f"max err {err.max():.3e}"


def test_prefill_last_row_equals_decode_with_sinks(pkv_lib):
    """The last chunk token attends exactly what a decode of length L with the
    same window and sinks attends."""
    w, q, k, v, cu, lens = _prefill_case(torch.bfloat16, 8, 2, 128, 16, [700, 90], [100, 40], 0,
                                         seed=5)
    out = pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, lens, 50,
                              w.scale, max_chunk=100, num_sinks=6)
    last = cu[1:].long() - 1
    dec = pkv_lib.pkv_decode(q[last].contiguous(), w.k_cache, w.v_cache, w.block_tables, lens, 50,
                             w.scale, num_sinks=6)
    torch.cuda.synchronize()
    diff = (out[last].double() - dec.double()).abs().max().item()
    assert diff <= 2e-3 + 0.5 * torch.finfo(torch.bfloat16).eps * dec.double().abs().max().item()


def test_prefill_last_row_equals_decode(pkv_lib):
    """The last chunk token attends exactly what a decode of length L attends."""
    w, q, k, v, cu, lens = _prefill_case(torch.bfloat16, 8, 2, 128, 16, [100, 37], [40, 12], 0,
                                         seed=3)
    out = pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, lens, 0,
                              w.scale, max_chunk=40)
    last = cu[1:].long() - 1
    dec = pkv_lib.pkv_decode(q[last].contiguous(), w.k_cache, w.v_cache, w.block_tables, lens, 0,
                             w.scale)
    torch.cuda.synchronize()
    diff = (out[last].double() - dec.double()).abs().max().item()
    assert diff <= 2e-3 + 0.5 * torch.finfo(torch.bfloat16).eps * dec.double().abs().max().item()


@pytest.mark.parametrize("scale", [0.0, -0.0625])
def test_prefill_nonpositive_scale(pkv_lib, oracle_lib, scale):
    """A zero scale gives the mean of the visible V rows; a negative one flips
    which keys dominate.  Both take the kernel's scale-first path."""
    chunks, prefixes = [70, 130], [40, 0]
    w, q, k, v, cu, lens = _prefill_case(torch.bfloat16, 8, 2, 128, 16, prefixes, chunks, 0,
                                         seed=11)
    kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
    bt = w.block_tables.cpu().numpy()
    lens_h = lens.cpu().numpy()
    slots = [oracle.slot_for_position(bt[b], w.spec.block_size, lens_h[b] - n + i)
             for b, n in enumerate(chunks) for i in range(n)]
    oracle.append(k.cpu(), v.cpu(), np.array(slots, np.int64), kc, vc)
    ref = oracle.prefill(q.cpu(), cu.cpu().numpy(), kc, vc, bt, lens_h, 0, scale)
    out = pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, lens, 0, scale,
                              max_chunk=max(chunks))
    torch.cuda.synchronize()
    g = out.double().cpu().numpy()
    err = np.abs(g - ref)
    assert (err <= 2e-3 + 0.5 * torch.finfo(torch.bfloat16).eps * np.abs(ref)).all(), err.max()


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("mode", ["dense", "sparse", "one_pair"])
@pytest.mark.parametrize("window,sinks", [(0, 0), (90, 5)])
def test_prefill_bf16_extreme_values_match_oracle(pkv_lib, oracle_lib, window, sinks, mode, d):
    """bf16 caches are exact over bf16's whole range: V values far beyond the
    fp16 range (7e4, 1e6, 1e30, 1e35 -- the last past 2^100, where the sums
    of weights times values need the weights scaled down to stay finite in
    fp32) and far below fp16's normal range (3e-6, 1e-30), in cached prefix
    keys and in the chunk's own keys, give the oracle's output within the
    usual tolerance.
    dense: every key holds them (every key tile takes the bf16 product), and
    the columns that hold them (all of one sign, so no cancellation hides an
    error) are also within a relative 2^-7.
    sparse: a few keys hold them.
    one_pair: only kv head 1 of the second sequence holds them (in a few
    keys), so one launch mixes pairs whose V scales into fp16 exactly with
    pairs that need the bf16 product."""
    dtype = torch.bfloat16
    prefixes, chunks = [30, 300], [10, 200]
    w, q, k, v, cu, lens = _prefill_case(dtype, 8, 2, d, 16, prefixes, chunks, window,
                                         seed=17)
    g = torch.Generator(device="cuda").manual_seed(23)

    def pos(shape, scale):  # positive values of one magnitude
        return ((1.0 + torch.rand(shape, generator=g, device="cuda")) * scale).to(dtype)

    bt = w.block_tables.cpu().numpy()
    bs = w.spec.block_size
    # (kv head, column) -> magnitude
    special = {(0, 3): 1.0e6, (0, 11): 1.0e-30, (0, 20): 1.0e35, (1, 7): 1.0e30,
               (1, 12): 3.0e-6, (1, 40): 7.0e4}
    if mode == "one_pair":
        special = {(h, c): mag for (h, c), mag in special.items() if h == 1}
    for b, (p, n) in enumerate(zip(prefixes, chunks)):
        if mode == "one_pair" and b != 1:
            continue
        ts = list(range(p)) if mode == "dense" else [t for t in (5, p - 1) if 0 <= t < p]
        s_pref = [oracle.slot_for_position(bt[b], bs, t) for t in ts]
        if s_pref:
            s_arr = torch.tensor(s_pref, device="cuda")
            for (h, c), mag in special.items():
                w.v_cache[s_arr // bs, h, s_arr % bs, c] = pos(len(s_pref), mag)
    rows = (torch.arange(v.shape[0], device="cuda") if mode == "dense"
            else torch.tensor([150] if mode == "one_pair" else [3, 150], device="cuda"))
    for (h, c), mag in special.items():
        v[rows, h, c] = pos(rows.numel(), mag)
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    lens_h = lens.cpu().numpy()
    slots = [oracle.slot_for_position(bt[b], bs, lens_h[b] - n + i)
             for b, n in enumerate(chunks) for i in range(n)]
    oracle.append(k.cpu(), v.cpu(), np.array(slots, np.int64), kc_h, vc_h)
    ref = oracle.prefill(q.cpu(), cu.cpu().numpy(), kc_h, vc_h, bt, lens_h, window, w.scale,
                         num_sinks=sinks)
    out = torch.full_like(q, float("nan"))
    pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, lens, window,
                        w.scale, max_chunk=max(chunks), out=out, num_sinks=sinks)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    tol = 2e-3 + 0.5 * torch.finfo(dtype).eps * np.abs(ref)
    assert (err <= tol).all(), f"max err {err.max():.3e}"
    if mode == "dense":
        G = 4  # query heads per kv head
        for (h, c), mag in special.items():
            r = ref[:, h * G:(h + 1) * G, c]
            e = err[:, h * G:(h + 1) * G, c]
            assert (r > 0).all()
            assert (e <= 2.0 ** -7 * r).all(), (h, c, float((e / r).max()))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_prefill_invalid_indices_give_nan_rows_only(pkv_lib, dtype):
    """A block id outside the pool in a sequence's table, or a length the
    table cannot hold, makes that sequence's rows NaN (never a trap, never a
    read outside the pool); the other sequences' rows are exactly those of a
    run without the bad sequences (bf16: the V-range scan skips the bad
    rows too)."""
    prefixes, chunks = [40, 70, 20], [10, 30, 25]
    w, q, k, v, cu, lens = _prefill_case(dtype, 8, 2, 128, 16, prefixes, chunks, 0, seed=9)
    good = pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache.clone(), w.v_cache.clone(),
                               w.block_tables, lens, 0, w.scale, max_chunk=max(chunks))
    bt = w.block_tables.clone()
    bt[0, 1] = w.num_blocks + 7          # a prefix block of sequence 0 past the pool
    bad_lens = lens.clone()
    bad_lens[2] = bt.shape[1] * w.spec.block_size + 1   # longer than sequence 2's table
    out = pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, bt, bad_lens, 0, w.scale,
                              max_chunk=max(chunks))
    torch.cuda.synchronize()
    o, r = out.float().cpu(), good.float().cpu()
    c = cu.cpu().tolist()
    assert torch.isnan(o[c[0]:c[1]]).all()
    assert torch.isnan(o[c[2]:c[3]]).all()
    assert torch.equal(o[c[1]:c[2]], r[c[1]:c[2]])


def test_prefill_bf16_long_table_scan_sees_every_row(pkv_lib, oracle_lib):
    """A block table longer than 64 row blocks of 128 (here 10,040 tokens)
    is scanned in longer blocks; a single V value of 1e30 near its end must
    still be found (else it would be converted to fp16, an infinity), and the
    output matches the oracle."""
    dtype = torch.bfloat16
    prefixes, chunks = [10000], [40]
    w, q, k, v, cu, lens = _prefill_case(dtype, 8, 2, 128, 16, prefixes, chunks, 0, seed=31)
    bt = w.block_tables.cpu().numpy()
    s = oracle.slot_for_position(bt[0], 16, 9500)
    w.v_cache[s // 16, 1, s % 16, 5] = 1.0e30
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    lens_h = lens.cpu().numpy()
    slots = [oracle.slot_for_position(bt[0], 16, lens_h[0] - 40 + i) for i in range(40)]
    oracle.append(k.cpu(), v.cpu(), np.array(slots, np.int64), kc_h, vc_h)
    ref = oracle.prefill(q.cpu(), cu.cpu().numpy(), kc_h, vc_h, bt, lens_h, 0, w.scale)
    out = pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, lens, 0,
                              w.scale, max_chunk=40)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert (err <= 2e-3 + 0.5 * torch.finfo(dtype).eps * np.abs(ref)).all(), err.max()


@pytest.mark.parametrize("workload", ["prefill_bf16", "prefill_fp16"])
def test_prefill_benchmark_workload_sampled(pkv_lib, oracle_lib, workload):
    """The bench's prefill workloads at their full size (4 sequences, a
    1024-token chunk each after a 2048-6144-token cached prefix, 32 query / 8
    kv heads, head_dim 128, block size 16), in the call the bench times: the
    pools after the chunk's append equal the oracle's bit for bit, and sampled
    rows -- every query head of each sequence's first and last chunk token and
    of 30 random ones -- match the float64 oracle.  Without a window, the row
    of the token at position p attends keys 0 .. p ("Building a Streaming
    Sliding-Window Attention Engine in Pure Python", Step 3,
    prefill_attention, read row-wise): the oracle's decode of that query with
    context length p + 1."""
    import bench

    w, q, k, v, cu, L, chunk, _ = bench.prefill_inputs(workload)
    spec = w.spec
    bs, dtype = spec.block_size, spec.dtype
    kc_h, vc_h = w.k_cache.cpu(), w.v_cache.cpu()
    bt = w.block_tables.cpu().numpy()
    lens, cu_h = L.cpu().numpy(), cu.cpu().numpy()
    out = torch.full_like(q, float("nan"))
    pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache, w.block_tables, L, 0, w.scale,
                        max_chunk=chunk, out=out)
    torch.cuda.synchronize()
    slots = [oracle.slot_for_position(bt[b], bs, int(lens[b]) - chunk + i)
             for b in range(spec.num_seqs) for i in range(chunk)]
    oracle.append(k.cpu(), v.cpu(), np.array(slots, np.int64), kc_h, vc_h)
    assert torch.equal(_bits(w.k_cache.cpu()), _bits(kc_h))
    assert torch.equal(_bits(w.v_cache.cpu()), _bits(vc_h))

    r = np.random.default_rng(41)
    toks = []
    for b in range(spec.num_seqs):
        sel = {0, chunk - 1} | set(r.choice(chunk, 30, replace=False).tolist())
        toks += [(b, i) for i in sorted(sel)]
    rows = torch.tensor([int(cu_h[b]) + i for b, i in toks], device=q.device)
    ctx = np.array([int(lens[b]) - chunk + i + 1 for b, i in toks], np.int32)
    ref = oracle.decode(q[rows].cpu(), kc_h, vc_h, np.stack([bt[b] for b, _ in toks]), ctx, 0,
                        w.scale)
    g = out[rows].double().cpu().numpy()
    assert np.isfinite(g).all()
    err = np.abs(g - ref)
    tol = 2e-3 + 0.5 * torch.finfo(dtype).eps * np.abs(ref)
    assert (err <= tol).all(), f"max err {err.max():.3e}"


def test_prefill_two_streams_concurrently(pkv_lib, oracle_lib):
    """Two prefills at the same time on two streams (each stream has its own
    workspace: work order, counters, V ranges), launched interleaved for
    several rounds without synchronisation between the streams: every
    round's rows match the oracle and the pools end bit for bit as its."""
    cases = [(torch.float16, [300, 40, 0], [200, 77, 130], 0, 51),
             (torch.bfloat16, [1000, 5], [64, 300], 0, 52)]
    prepared = []
    for dtype, prefixes, chunks, window, seed in cases:
        w, q, k, v, cu, lens = _prefill_case(dtype, 8, 2, 128, 16, prefixes, chunks, window, seed)
        ref, kc_h, vc_h = _oracle_prefill(w, q, k, v, cu, lens, chunks, window)
        prepared.append((w, q, k, v, cu, lens, chunks, window, ref, kc_h, vc_h, dtype))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    outs = []
    for _ in range(3):
        for i, st in enumerate(streams):
            w, q, k, v, cu, lens, chunks, window = prepared[i][:8]
            with torch.cuda.stream(st):
                # the same chunk again: its append rewrites the same rows
                outs.append((i, pkv_lib.pkv_prefill(q, k, v, cu, w.k_cache, w.v_cache,
                                                    w.block_tables, lens, window, w.scale,
                                                    max_chunk=max(chunks), stream=st)))
    torch.cuda.synchronize()
    for i, out in outs:
        ref, dtype = prepared[i][8], prepared[i][11]
        g = out.double().cpu().numpy()
        assert np.isfinite(g).all()
        err = np.abs(g - ref)
        assert (err <= 2e-3 + 0.5 * torch.finfo(dtype).eps * np.abs(ref)).all(), err.max()
    for p_ in prepared:
        w, kc_h, vc_h = p_[0], p_[9], p_[10]
        assert torch.equal(_bits(w.k_cache.cpu()), _bits(kc_h))
        assert torch.equal(_bits(w.v_cache.cpu()), _bits(vc_h))
