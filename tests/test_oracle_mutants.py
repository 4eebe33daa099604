"""Plant plausible mistakes in the oracle and check that the pins reject each one.

Every mutant is a copy of oracle/pf_oracle.c with one textual change (a dropped
term, a wrong index or sign, a transposed layout ...).  It is compiled with gcc
into a temporary directory and the whole pin suite (tests/test_oracle_pins.py)
is run against it in a child process; the mutant counts as caught when that run
fails (or crashes).  The unmodified source must pass the same run.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "gqa_interleaved_head_map": [("    return h / g;", "    return h % P->Hkv;")],
    "dropped_scale": [("s[t - t0] = P->scale * dot;", "s[t - t0] = dot;")],
    "score_sign": [("dot += bf16_to_f64(qv[c])", "dot -= bf16_to_f64(qv[c])")],
    "reversed_offset_in_block": [("int off = t % P->bs;", "int off = (P->bs - 1) - t % P->bs;")],
    "transposed_cache_layout": [("return (((size_t)p * Hkv + kh) * bs + off) * D + c;",
                                 "return (((size_t)p * bs + off) * Hkv + kh) * D + c;")],
    "missing_normalisation": [("double w = exp(s[t - t0] - m) / l;", "double w = exp(s[t - t0] - m);")],
    "min_instead_of_max": [("if (s[t] > m) m = s[t];", "if (s[t] < m || m == -INFINITY) m = s[t];")],
    "query_head_collapsed": [("P->q + ((size_t)i * P->Hq + h) * P->D",
                              "P->q + ((size_t)i * P->Hq + h / (P->Hq / P->Hkv)) * P->D")],
    "value_read_from_key_cache": [("bf16_to_f64(P->v_cache[", "bf16_to_f64(P->k_cache[")],
    "partition_drops_a_token": [("int t1 = t0 + partition_size < L ? t0 + partition_size : L;",
                                 "int t1 = t0 + partition_size <= L ? t0 + partition_size - 1 : L;")],
    "merge_drops_partition_sum": [("W += tmp_l[base + k] * exp(tmp_m[base + k] - M);",
                                   "W += exp(tmp_m[base + k] - M);"),
                                  ("double w = tmp_l[base + k] * exp(tmp_m[base + k] - M) / W;",
                                   "double w = exp(tmp_m[base + k] - M) / W;")],
    "merge_exponent_sign": [("exp(tmp_m[base + k] - M)", "exp(M - tmp_m[base + k])")],
    "append_wrong_offset": [("int off = (int)(s % block_size);", "int off = (int)(s / block_size % block_size);")],
    "append_token_head_swapped": [("size_t src = ((size_t)i * num_kv_heads + h) * head_dim + c;",
                                   "size_t src = ((size_t)h * num_kv_heads + i) * head_dim + c;")],
    "append_no_skip_of_minus_one": [("if (s == -1) continue;", "")],
    "copy_direction_swapped": [("int64_t src = block_mapping[2 * j], dst = block_mapping[2 * j + 1];",
                                "int64_t dst = block_mapping[2 * j], src = block_mapping[2 * j + 1];")],
    "multi_query_not_causal": [("int t1 = pos + 1;", "int t1 = context_lens[i];")],
    "multi_query_row_off_by_one": [("int pos = context_lens[i] - q_len + j;", "int pos = context_lens[i] - q_len + j - 1;")],
    "copy_skips_v": [("            v_cache[(size_t)dst * per_block + e] = v_cache[(size_t)src * per_block + e];\n", "")],
}


def _build(tmp_path, name, edits):
    with open(oracle.SOURCE) as f:
        text = f.read()
    for old, new in edits:
        assert old in text, f"{name}: pattern not found: {old}"
        text = text.replace(old, new)
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    return oracle.compile_oracle(str(src), out_dir=str(tmp_path), openmp=False)


def _pin_run(so_path):
    env = dict(os.environ, PF_ORACLE_SO=so_path)
    return subprocess.Popen([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                             os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                            cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)


def test_pins_reject_every_mutant(tmp_path):
    runs = {"unmodified": _pin_run(_build(tmp_path, "unmodified", []))}
    for name, edits in MUTANTS.items():
        runs[name] = _pin_run(_build(tmp_path, name, edits))
    results = {name: (p.wait(timeout=900), p.stdout.read().decode(errors="replace")) for name, p in runs.items()}
    rc, log = results.pop("unmodified")
    assert rc == 0, "pins fail on the unmodified oracle:\n" + log[-2000:]
    survivors = [name for name, (rc, _) in results.items() if rc == 0]
    assert not survivors, f"mutants not caught by any pin: {survivors}"
