"""The oracle's pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a temporary copy of oracle/pkv_oracle.c (on the
CPU, never in the product), rebuilds it, and runs the oracle pin files
(tests/test_oracle*.py) against the copy: the pin suite has to fail.  The mistakes are the ones a careful
reader of the pages could still make: a wrong GQA head mapping, a flipped or
missing max-subtraction, an off-by-one window start, a wrong attention-sink
count or ignored sinks, swapped K and V, wrong row/block or head-major
indexing, a squared scale, wrong element decoding, a wrong slot, a wrong
append destination, the wrong query head, a non-zero empty context, and in the
FP8 cache a wrong exponent bias, ties broken to odd, a dropped sign, a wrong
quantisation constant, or an ignored row scale, in the INT8 cache a wrong
scale constant, truncation or ties away from zero instead of ties to even, or
codes read as unsigned, and in the prefill a query position off by one, a
missing causal limit or ignored attention sinks.
"""
import os
import shutil
import subprocess
import sys

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "gqa_head_mapping": ("const int32_t hk = h / G;", "const int32_t hk = h % p->num_kv_heads;"),
    "exp_sign": ("s[t] = exp(s[t] - m);", "s[t] = exp(m - s[t]);"),
    "no_max_subtraction": ("s[t] = exp(s[t] - m);", "s[t] = exp(s[t]);"),
    "window_off_by_one": ("int64_t lo = L - window;", "int64_t lo = L - window + 1;"),
    "sink_count_off_by_one": (
        "if (p->window > 0 && p->num_sinks > 0) n_sink = p->num_sinks < lo ? p->num_sinks : lo;",
        "if (p->window > 0 && p->num_sinks > 0) n_sink = p->num_sinks + 1 < lo ? p->num_sinks + 1 : lo;"),
    "sinks_ignored": ("if (!(t < n_sink || t >= lo)) continue;", "if (!(t >= lo)) continue;"),
    "k_v_swapped": ("V[i * D + d] = load_elem(p->v_cache", "V[i * D + d] = load_elem(p->k_cache"),
    "row_index": ("int64_t row = t % p->block_size;",
                  "int64_t row = (t / p->block_size) % p->block_size;"),
    "token_major_offset": (
        "int64_t prow = (physical * p->num_kv_heads + hk) * p->block_size + row;",
        "int64_t prow = (physical * p->block_size + row) * p->num_kv_heads + hk;"),
    "scale_squared": ("s[t] = scale * dot;", "s[t] = scale * scale * dot;"),
    "f16_exponent_bias": ("mag = ldexp((double)(1024 + frac), expo - 25);",
                          "mag = ldexp((double)(1024 + frac), expo - 24);"),
    "bf16_shift": ("uint32_t w = ((uint32_t)bits) << 16;", "uint32_t w = ((uint32_t)bits) << 15;"),
    "slot_offset": ("return physical * block_size + offset;",
                    "return physical * block_size + offset + 1;"),
    "append_destination": (
        "size_t dst_row = (((size_t)block * num_kv_heads + h) * block_size + row);",
        "size_t dst_row = (((size_t)row * num_kv_heads + h) * block_size + block);"),
    "query_head": (
        "q[d] = load_elem(p->q, ((int64_t)b * p->num_q_heads + h) * D + d, p->dtype);",
        "q[d] = load_elem(p->q, ((int64_t)b * p->num_q_heads + hk) * D + d, p->dtype);"),
    "e4m3_exponent_bias": ("else mag = ldexp((double)(8 + frac), expo - 10);",
                           "else mag = ldexp((double)(8 + frac), expo - 9);"),
    "e4m3_ties_to_odd": ("(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    "e4m3_sign_dropped": ("uint8_t sign = (x < 0.0f || (x == 0.0f && 1.0f / x < 0.0f)) ? 0x80 : 0x00;",
                          "uint8_t sign = 0x00;"),
    "fp8_scale_constant": ("volatile float num = 448.0f;", "volatile float num = 480.0f;"),
    "fp8_scale_ignored": ("double ks = (double)p->k_scale[prow], vs = (double)p->v_scale[prow];",
                          "double ks = 1.0, vs = (double)p->v_scale[prow];"),
    "int8_scale_constant": ("volatile float top = 127.0f;", "volatile float top = 128.0f;"),
    "int8_round_truncates": ("double r = nearbyint((double)prod);",
                             "double r = trunc((double)prod);"),
    "int8_ties_away_from_zero": ("double r = nearbyint((double)prod);",
                                 "double r = round((double)prod);"),
    "int8_codes_unsigned": ("kc = (double)((const int8_t*)p->k_cache)[base + d];",
                            "kc = (double)((const uint8_t*)p->k_cache)[base + d];"),
    "prefill_position_off_by_one": (
        "const int64_t p = context_lens[b] - n + (t - cu_q[b]); /* its position */",
        "const int64_t p = context_lens[b] - n + (t - cu_q[b]) + 1; /* its position */"),
    "prefill_not_causal": ("int32_t len = (int32_t)(p + 1);", "int32_t len = context_lens[b];"),
    "prefill_ignores_sinks": ("max_blocks, &len, window,\n                         num_sinks, scale};",
                              "max_blocks, &len, window,\n                         0, scale};"),
    "empty_context_not_zero": (
        "for (int32_t d = 0; d < D; ++d) out[d] = 0.0;\n  if (T <= 0) return;",
        "for (int32_t d = 0; d < D; ++d) out[d] = 0.0;\n  if (T <= 0) { out[0] = 1.0; return; }"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, oracle_lib):
    if shutil.which("gcc") is None:
        pytest.skip("gcc unavailable")
    original, mutated = MUTANTS[name]
    src = open(os.path.join(REPO, "oracle", "pkv_oracle.c")).read()
    assert src.count(original) == 1, f"mutation site for {name} not found exactly once"
    shutil.copytree(os.path.join(REPO, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    (tmp_path / "oracle" / "pkv_oracle.c").write_text(src.replace(original, mutated))
    shutil.copytree(os.path.join(REPO, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutants.py",
                                                  "test_gpu*", "test_zz*"))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle.py", "tests/test_oracle_fp8.py",
                        "tests/test_oracle_int8.py", "tests/test_oracle_prefill.py"],
                       cwd=tmp_path,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"pins did not catch '{name}':\n{r.stdout[-2000:]}"
