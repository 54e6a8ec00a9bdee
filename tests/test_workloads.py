"""Host-side checks of the seeded workload generator and the LIFO free-block stack."""
import json
import os

import numpy as np
import pytest
import torch

from paged_kv_cache_24_gb300.workloads import FreeBlockStack, config_spec, make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _p2():
    with open(os.path.join(GOLDEN, "p2_allocator_and_slots.json")) as f:
        return json.load(f)


def test_allocator_counts_from_the_page():
    g = _p2()["allocator"]
    a = FreeBlockStack(g["total_blocks"])
    got = a.take(owner=1, count=g["allocate"])
    assert len(got) == len(set(got)) == g["allocate"]
    assert a.available == g["free_after_allocate"]
    a.give_back(1)
    assert a.available == g["free_after_deallocate"]
    assert a.held_by == {}


def test_allocator_is_lifo_and_raises_when_exhausted():
    g = _p2()["exhaustion"]
    a = FreeBlockStack(g["total_blocks"], stack=[3, 1, 0, 2])
    assert a.take(0) == [2]          # the top of the stack first
    a.give_back(0)
    assert a.take(5) == [2]          # the block just returned comes back first
    assert a.take(6, 2) == [0, 1]    # then the next ones down, top first
    a.give_back(6)
    a.give_back(5)
    assert a.stack == [3, 0, 1, 2]
    # one block per 16 tokens: 64 tokens fit in 4 blocks, the 65th does not
    held = 0
    for pos in range(g["tokens_before_error"]):
        if pos // g["block_size"] >= held:
            a.take(7)
            held += 1
    with pytest.raises(MemoryError):
        a.take(7)


def _slots_of(w, b, upto):
    bs = w.spec.block_size
    t = np.arange(upto)
    return w.block_tables[b].numpy()[t // bs].astype(np.int64) * bs + t % bs


def test_tiny_config_matches_its_statement():
    w = make_workload(config_spec(0))
    assert w.num_blocks == 32
    assert w.lens_steps[0].tolist() == [18, 34, 65, 101]
    assert w.pos_steps[0].tolist() == [17, 33, 64, 100]
    ids = [int(x) for b in range(4) for x in w.block_tables[b] if x >= 0]
    assert len(ids) == len(set(ids)) == 2 + 3 + 5 + 7  # ceil(L / 16) per sequence
    assert all(0 <= i < 32 for i in ids)
    assert w.scale == pytest.approx(0.125)
    assert w.k_cache.dtype == torch.float32 and tuple(w.k_cache.shape) == (32, 8, 16, 64)


def test_poison_marks_exactly_the_unheld_slots():
    w = make_workload(config_spec(0))
    nb, h, bs, d = w.k_cache.shape
    valid = np.zeros(nb * bs, bool)
    for b in range(4):
        valid[_slots_of(w, b, int(w.pos_steps[0, b]))] = True
    flat = w.k_cache.permute(0, 2, 1, 3).reshape(nb * bs, -1)
    assert torch.isnan(flat[torch.from_numpy(~valid)]).all()
    assert torch.isfinite(flat[torch.from_numpy(valid)]).all()


def test_uniform_lengths_and_pool_factor():
    w = make_workload(config_spec(1, num_seqs=16, num_q_heads=4, num_kv_heads=4))
    lens = w.lens_steps[0].numpy()
    assert lens.min() >= 512 and lens.max() <= 4096
    need = ((lens + 15) // 16).sum()
    assert w.num_blocks == int(np.ceil(1.2 * need))
    ids = w.block_tables.numpy()
    used = ids[ids >= 0]
    assert len(used) == len(set(used.tolist())) == need


def test_serving_mix_structure():
    spec = config_spec(4, num_seqs=64, num_q_heads=4, num_kv_heads=2, steps=32)
    w = make_workload(spec, poison=False)
    bs = 16
    pre = w.pos_steps[0].numpy()
    assert pre.min() >= 128 and pre.max() <= 2048
    assert w.steps == 32
    assert np.array_equal(w.lens_steps.numpy(), w.pos_steps.numpy() + 1)
    tables = w.block_tables.numpy()
    for g0 in range(0, 64, 16):
        members = range(g0, g0 + 16)
        for b in members:
            n_shared = min(16, pre[b] // bs)
            for c in members:
                m = min(n_shared, min(16, pre[c] // bs))
                assert np.array_equal(tables[b, :m], tables[c, :m])
    # occupancy at step 0
    assert w.unique_blocks / w.num_blocks == pytest.approx(0.7, abs=0.01)
    # every block a step appends into is private to its sequence
    for b in range(64):
        for s in range(32):
            blk = tables[b, w.pos_steps[s, b].item() // bs]
            sharers = [c for c in range(64) if c != b and blk in tables[c]]
            assert not sharers


def test_generator_is_deterministic():
    a = make_workload(config_spec(2, num_seqs=4, len_hi=1100))
    b = make_workload(config_spec(2, num_seqs=4, len_hi=1100))
    assert torch.equal(a.block_tables, b.block_tables)
    assert torch.equal(a.q_steps, b.q_steps)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
