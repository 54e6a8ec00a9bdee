"""Seeded synthetic workloads for paged decode attention.

This module produces inputs only: context lengths, block tables drawn from a
shuffled or fragmented block pool, a prefilled K/V pool, and the per-step new
tokens.  It holds none of the attention arithmetic and no slot arithmetic
(each side -- the CUDA library and the float64 oracle -- maps positions to
slots with its own code), so it can feed both without coupling them.

Workload recipes follow the five benchmark configurations of this project
(tiny fp32 / MHA fp16 / GQA bf16 / sliding-window bf16 / serving mix fp16).
The serving mix's fragmented pool hands out its free block ids last in, first
out, as the allocator of "Build a Paged KV Cache in Pure Python", Step 2 does
(``FreeBlockStack`` here).

Poisoning: every pool slot that no sequence's context covers holds NaN (and,
with ``poison_outside_window``, every slot before a sequence's window start
other than its attention sinks),
so a kernel that reads a slot it should not shows NaN in its output.  The slot
each step's append will write also starts as NaN.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

__all__ = [
    "FreeBlockStack", "WorkloadSpec", "Workload", "make_workload", "CONFIGS", "config_spec",
]


class FreeBlockStack:
    """The serving workload's pool bookkeeping: block ids not in use sit on a
    stack, and a request takes ids from its top (so the ids a sequence gave
    back are the first reused).

    The pages' allocator behaves the same way (a LIFO free list, an error once
    the pool cannot serve a request); this is only the part the serving mix
    needs to lay out a fragmented, partly occupied pool from a seed.  It never
    touches K/V data.
    """

    def __init__(self, num_blocks: int, stack: Optional[List[int]] = None):
        self.num_blocks = int(num_blocks)
        self.stack: List[int] = (list(range(self.num_blocks)) if stack is None
                                 else [int(x) for x in stack])
        self.held_by: dict = {}

    def take(self, owner: int, count: int = 1) -> List[int]:
        """Pop `count` ids for `owner`; MemoryError when fewer are left."""
        if count > len(self.stack):
            raise MemoryError(f"block pool exhausted: {count} requested, {len(self.stack)} of "
                              f"{self.num_blocks} left")
        ids = self.stack[len(self.stack) - count:][::-1]
        del self.stack[len(self.stack) - count:]
        self.held_by[owner] = self.held_by.get(owner, []) + ids
        return ids

    def give_back(self, owner: int) -> None:
        """Push every id `owner` holds back onto the stack, in the order taken."""
        self.stack.extend(self.held_by.pop(owner, []))

    @property
    def available(self) -> int:
        return len(self.stack)


@dataclass
class WorkloadSpec:
    name: str
    dtype: torch.dtype
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    # Lengths: either explicit, or drawn by `len_dist` in [len_lo, len_hi].
    # For single-step workloads the lengths are the decode lengths (the step's
    # appended token included); for multi-step ones they are the lengths before
    # the first step's append.
    lens: Optional[List[int]] = None
    len_dist: str = "uniform"  # "uniform" | "geometric"
    len_lo: int = 1
    len_hi: int = 1
    geom_mean: float = 512.0
    lens_are_pre_append: bool = False
    window: int = 0
    num_sinks: int = 0                # with a window: first positions kept (attention sinks)
    kv_fp8: bool = False              # pools of FP8 E4M3 codes + float32 row scales
    kv_int8: bool = False             # pools of int8 codes + float32 row scales
    steps: int = 1
    pool_factor: float = 1.2          # pool = ceil(factor * blocks needed), shuffled ids
    explicit_pool: Optional[int] = None
    occupancy: Optional[float] = None  # serving: fraction of the pool held at step 0
    prefix_group: int = 0             # serving: sequences per shared-prefix group
    prefix_tokens: int = 0            # serving: shared prefix length in tokens
    seed: int = 0


def config_spec(idx: int, **overrides) -> WorkloadSpec:
    """The five benchmark workloads (index 0..4) and FP8-pool (5, 6) and INT8-pool
    (7, 8) variants of the MHA and GQA ones, optionally resized for tests."""
    table = {
        0: dict(name="tiny_fp32", dtype=torch.float32, num_seqs=4, num_q_heads=8, num_kv_heads=8,
                head_dim=64, block_size=16, lens=[17, 33, 64, 100], lens_are_pre_append=True,
                explicit_pool=32, seed=0),
        1: dict(name="mha_fp16", dtype=torch.float16, num_seqs=64, num_q_heads=32, num_kv_heads=32,
                head_dim=128, block_size=16, len_lo=512, len_hi=4096, seed=1),
        2: dict(name="gqa_bf16", dtype=torch.bfloat16, num_seqs=256, num_q_heads=32,
                num_kv_heads=8, head_dim=128, block_size=32, len_lo=1024, len_hi=8192, seed=2),
        3: dict(name="sliding_bf16", dtype=torch.bfloat16, num_seqs=16, num_q_heads=32,
                num_kv_heads=8, head_dim=128, block_size=16, len_lo=16384, len_hi=32768,
                window=4096, seed=3),
        4: dict(name="serving_fp16", dtype=torch.float16, num_seqs=1024, num_q_heads=32,
                num_kv_heads=8, head_dim=128, block_size=16, len_dist="geometric", len_lo=128,
                len_hi=2048, geom_mean=512.0, lens_are_pre_append=True, steps=32,
                occupancy=0.7, prefix_group=16, prefix_tokens=256, seed=4),
    }
    # the MHA and GQA shapes over FP8 E4M3 pools (fp16 queries and new tokens)
    table[5] = dict(table[1], name="mha_fp8", kv_fp8=True, seed=5)
    table[6] = dict(table[2], name="gqa_fp8", dtype=torch.float16, kv_fp8=True, seed=6)
    # the same shapes over INT8 pools
    table[7] = dict(table[1], name="mha_int8", kv_int8=True, seed=7)
    table[8] = dict(table[2], name="gqa_int8", dtype=torch.float16, kv_int8=True, seed=8)
    base = dict(table[idx])
    base.update(overrides)
    return WorkloadSpec(**base)


CONFIGS = {config_spec(i).name: i for i in range(9)}


@dataclass
class Workload:
    spec: WorkloadSpec
    scale: float                 # float32-rounded 1/sqrt(head_dim)
    num_blocks: int
    block_tables: torch.Tensor   # [B, MB] int32; -1 where a sequence has no block
    lens_steps: torch.Tensor     # [S, B] int32 decode length at each step (append included)
    pos_steps: torch.Tensor      # [S, B] int64 position of each step's new token
    q_steps: torch.Tensor        # [S, B, Hq, D]
    k_steps: torch.Tensor        # [S, B, Hkv, D]
    v_steps: torch.Tensor        # [S, B, Hkv, D]
    k_cache: torch.Tensor        # [NB, Hkv, bs, D] (uint8 E4M3 codes for FP8 pools)
    v_cache: torch.Tensor        # [NB, Hkv, bs, D]
    k_scale: Optional[torch.Tensor] = None  # FP8 pools: [NB, Hkv, bs] float32 row scales
    v_scale: Optional[torch.Tensor] = None
    unique_blocks: int = 0       # distinct physical blocks referenced at step 0
    free_list_after: List[int] = field(default_factory=list)

    @property
    def steps(self) -> int:
        return self.lens_steps.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]


def _draw_lengths(spec: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    if spec.lens is not None:
        return np.asarray(spec.lens, dtype=np.int64)
    if spec.len_dist == "uniform":
        return rng.integers(spec.len_lo, spec.len_hi + 1, size=spec.num_seqs).astype(np.int64)
    if spec.len_dist == "geometric":
        # geometric on {1, 2, ...} with success probability 1/mean, then clipped
        raw = rng.geometric(1.0 / spec.geom_mean, size=spec.num_seqs)
        return np.clip(raw, spec.len_lo, spec.len_hi).astype(np.int64)
    raise ValueError(spec.len_dist)


def _fill_random(t: torch.Tensor, gen: torch.Generator, chunk_elems: int = 1 << 26) -> None:
    """t <- N(0, 1) drawn in fp32 and rounded to t's dtype, in chunks (bounded temporaries)."""
    flat = t.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=t.device, dtype=torch.float32)


def make_workload(spec: WorkloadSpec, device="cpu", poison: bool = True,
                  poison_outside_window: bool = False) -> Workload:
    """Build the seeded inputs of one workload on `device`.

    Host-side planning (lengths, block ids) uses numpy's PCG64 seeded with
    ``spec.seed``; tensor data uses a torch generator on ``device`` with the same
    seed.  The cache holds every sequence's tokens [0, L-1) of the first step;
    each step's append writes position ``pos_steps[s, b]``.
    """
    device = torch.device(device)
    rng = np.random.default_rng(spec.seed)
    B, Hq, Hkv, D, bs = (spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                         spec.block_size)
    if Hq % Hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    S = spec.steps
    lens0 = _draw_lengths(spec, rng)
    if len(lens0) != B:
        raise ValueError("lens must have num_seqs entries")
    if spec.lens_are_pre_append:
        pre = lens0                      # tokens already cached before step 0
    else:
        pre = np.maximum(lens0 - 1, 0)   # the first step appends token L-1
    # position of each step's new token and decode length after it
    pos = pre[None, :] + np.arange(S, dtype=np.int64)[:, None]          # [S, B]
    lens_steps = pos + 1
    final_len = lens_steps[-1]
    need_final = (final_len + bs - 1) // bs                             # blocks by the last step
    MB = int(need_final.max()) if B else 0
    block_tables = np.full((B, max(MB, 1)), -1, dtype=np.int64)

    if spec.occupancy is None:
        # Shuffled pool: ids from a random permutation, taken consecutively per sequence.
        total_need = int(need_final.sum())
        nb = spec.explicit_pool if spec.explicit_pool is not None else int(
            math.ceil(spec.pool_factor * total_need))
        if nb < total_need:
            raise ValueError("pool smaller than the blocks the workload needs")
        perm = rng.permutation(nb)
        cursor = 0
        for b in range(B):
            n = int(need_final[b])
            block_tables[b, :n] = perm[cursor:cursor + n]
            cursor += n
        unique = total_need
        free_after: List[int] = [int(x) for x in perm[cursor:]]
    else:
        # Serving mix: groups of `prefix_group` consecutive sequences share their
        # leading full blocks (identical block ids); the rest is private.  The
        # pool is sized so the step-0 blocks fill `occupancy` of it, at random
        # ids; the remaining ids form a shuffled free list popped LIFO.
        need0 = (pre + bs - 1) // bs
        shared_per_seq = np.zeros(B, dtype=np.int64)
        if spec.prefix_group > 0 and spec.prefix_tokens > 0:
            cap = spec.prefix_tokens // bs
            shared_per_seq = np.minimum(cap, pre // bs)
        groups = []
        for g0 in range(0, B, max(spec.prefix_group, 1) if spec.prefix_group else B):
            members = list(range(g0, min(B, g0 + (spec.prefix_group or B))))
            groups.append(members)
        n_shared = [int(shared_per_seq[m].max()) if m else 0 for m in groups]
        unique = int(sum(n_shared) + sum(int(need0[b] - shared_per_seq[b]) for b in range(B)))
        nb = int(math.ceil(unique / spec.occupancy))
        ids = rng.permutation(nb)
        occupied, free = ids[:unique], ids[unique:]
        cursor = 0
        for members, ns in zip(groups, n_shared):
            shared_ids = occupied[cursor:cursor + ns]
            cursor += ns
            for b in members:
                block_tables[b, :shared_per_seq[b]] = shared_ids[:shared_per_seq[b]]
        for b in range(B):
            n = int(need0[b] - shared_per_seq[b])
            block_tables[b, shared_per_seq[b]:need0[b]] = occupied[cursor:cursor + n]
            cursor += n
        alloc = FreeBlockStack(nb, stack=list(free))
        held = need0.copy()
        for s in range(S):                      # blocks the 32 steps need, in step order
            for b in range(B):
                while held[b] * bs <= pos[s, b]:
                    block_tables[b, held[b]] = alloc.take(b)[0]
                    held[b] += 1
        free_after = list(alloc.stack)

    # ---- tensors ---------------------------------------------------------
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    dt = spec.dtype
    k_scale = v_scale = None
    if spec.kv_fp8:
        # E4M3 codes of N(0, 1) * 64 (torch's float8 cast) and row scales around 1/64
        k_cache = torch.empty((nb, Hkv, bs, D), dtype=torch.uint8, device=device)
        v_cache = torch.empty((nb, Hkv, bs, D), dtype=torch.uint8, device=device)
        for c in (k_cache, v_cache):
            tmp = torch.empty(c.shape, dtype=torch.float32, device=device)
            _fill_random(tmp, gen)
            c.copy_((tmp * 64.0).to(torch.float8_e4m3fn).view(torch.uint8))
            del tmp
        k_scale = torch.rand((nb, Hkv, bs), generator=gen, device=device) * (1 / 64) + 1 / 128
        v_scale = torch.rand((nb, Hkv, bs), generator=gen, device=device) * (1 / 64) + 1 / 128
    elif spec.kv_int8:
        # int8 codes of N(0, 1) * 32 (rounded, clamped to +-127) and row scales around 1/64
        k_cache = torch.empty((nb, Hkv, bs, D), dtype=torch.int8, device=device)
        v_cache = torch.empty((nb, Hkv, bs, D), dtype=torch.int8, device=device)
        for c in (k_cache, v_cache):
            tmp = torch.empty(c.shape, dtype=torch.float32, device=device)
            _fill_random(tmp, gen)
            c.copy_((tmp * 32.0).round().clamp(-127, 127).to(torch.int8))
            del tmp
        k_scale = torch.rand((nb, Hkv, bs), generator=gen, device=device) * (1 / 64) + 1 / 128
        v_scale = torch.rand((nb, Hkv, bs), generator=gen, device=device) * (1 / 64) + 1 / 128
    else:
        k_cache = torch.empty((nb, Hkv, bs, D), dtype=dt, device=device)
        v_cache = torch.empty((nb, Hkv, bs, D), dtype=dt, device=device)
        _fill_random(k_cache, gen)
        _fill_random(v_cache, gen)
    q_steps = torch.empty((S, B, Hq, D), dtype=dt, device=device)
    k_steps = torch.empty((S, B, Hkv, D), dtype=dt, device=device)
    v_steps = torch.empty((S, B, Hkv, D), dtype=dt, device=device)
    for t in (q_steps, k_steps, v_steps):
        _fill_random(t, gen)

    if poison:
        # valid[slot] = some sequence holds a token there before step 0
        valid = np.zeros(nb * bs, dtype=bool)
        for b in range(B):
            lo = 0
            if poison_outside_window and spec.window > 0:
                lo = max(0, int(lens_steps[0, b]) - spec.window)
            keep = np.arange(0, min(lo, spec.num_sinks), dtype=np.int64)  # sink positions
            t = np.concatenate([keep, np.arange(lo, int(pre[b]), dtype=np.int64)])
            t = t[t < int(pre[b])]
            if t.size:
                valid[block_tables[b, t // bs] * bs + t % bs] = True
        bad = torch.from_numpy(np.nonzero(~valid)[0]).to(device)
        if bad.numel():
            blk, row = bad // bs, bad % bs
            if spec.kv_fp8 or spec.kv_int8:
                code = 0x7F if spec.kv_fp8 else -128  # E4M3 NaN / never-written int8 code
                k_cache[blk, :, row, :] = code
                v_cache[blk, :, row, :] = code
                k_scale[blk, :, row] = float("nan")
                v_scale[blk, :, row] = float("nan")
            else:
                k_cache[blk, :, row, :] = float("nan")
                v_cache[blk, :, row, :] = float("nan")

    return Workload(
        spec=spec,
        scale=float(np.float32(1.0 / math.sqrt(D))),
        num_blocks=nb,
        block_tables=torch.from_numpy(block_tables.astype(np.int32)).to(device),
        lens_steps=torch.from_numpy(lens_steps.astype(np.int32)).to(device),
        pos_steps=torch.from_numpy(pos.astype(np.int64)).to(device),
        q_steps=q_steps, k_steps=k_steps, v_steps=v_steps,
        k_cache=k_cache, v_cache=v_cache, k_scale=k_scale, v_scale=v_scale,
        unique_blocks=unique,
        free_list_after=free_after,
    )
