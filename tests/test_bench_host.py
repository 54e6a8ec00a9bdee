"""Host-side figures of bench.py: step bytes (touched and over distinct pool
rows) and the step-time percentiles, on tiny hand-built inputs."""
import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _w(tables, lens, window=0, hkv=2, d=64, bs=16, dtype=torch.float16, hq=4):
    spec = SimpleNamespace(dtype=dtype, kv_fp8=False, kv_int8=False, num_seqs=len(lens),
                           num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                           window=window)
    return SimpleNamespace(spec=spec, steps=1,
                           lens_steps=torch.tensor([lens], dtype=torch.int32),
                           block_tables=torch.tensor(tables, dtype=torch.int32))


def test_shared_prefix_rows_count_once():
    # both sequences read block 0 whole; then blocks 1 and 2 (4 rows each)
    sb = bench.step_bytes(_w([[0, 1], [0, 2]], [20, 20]))[0]
    row = 2 * 2 * 64 * 2          # K and V rows of 2 kv heads, D 64, fp16
    assert sb["kv"] == 40 * row
    assert sb["step_unique"] - sb["step"] == (24 - 40) * row


def test_windows_and_disjoint_tables():
    # window 10 over lengths 20 and 5: rows 10..19 of sequence 0, 0..4 of sequence 1
    sb = bench.step_bytes(_w([[3, 4], [5, 6]], [20, 5], window=10))[0]
    row = 2 * 2 * 64 * 2
    assert sb["kv"] == 15 * row
    assert sb["step_unique"] == sb["step"]     # nothing shared
    # the same physical block reached through two tables at different rows
    sb = bench.step_bytes(_w([[7, 0], [7, 0]], [3, 9]))[0]
    assert sb["kv"] == 12 * row and sb["step_unique"] - sb["step"] == (9 - 12) * row


def test_empty_contexts():
    sb = bench.step_bytes(_w([[0], [1]], [0, 0]))[0]
    assert sb["kv"] == 0 and sb["step_unique"] == sb["step"]


def test_percentiles():
    p = bench.percentiles_ms(list(range(1, 11)))
    assert p == pytest.approx({"p10": 1.9, "p50": 5.5, "p90": 9.1})
    assert bench.percentiles_ms([2.5]) == {"p10": 2.5, "p50": 2.5, "p90": 2.5}
