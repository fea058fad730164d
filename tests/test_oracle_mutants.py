"""The oracle pins must catch plausible mistakes.

Each mutant below plants one bug in a copy of ``oracle/ccv_oracle.c`` (a
dropped term, a wrong sign, index or operand), builds it on the CPU, and runs
the pin suite ``test_oracle.py`` against it.  The suite has to fail for every
mutant; a mutant that survives means a part of the oracle is not pinned.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

from oracle import build as oracle_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text to find in the source, replacement); every occurrence is replaced.
MUTANTS = [
    ("taps_reversed", "weight[c * ws_dim + k * ws_w]", "weight[c * ws_dim + (W - 1 - k) * ws_w]"),
    ("bias_dropped", "float b = bias ? bf16_to_f32(bias[c]) : 0.0f;", "float b = 0.0f;"),
    ("silu_sign", "exp(-d)", "exp(d)"),
    ("rounding_ties_away", "u += 0x7fffu + keep_lsb;", "u += 0x8000u;"),
    ("prior_columns_reversed",
     "? conv_states[line * ss_line + c * ss_dim + j * ss_tok]",
     "? conv_states[line * ss_line + c * ss_dim + (W - 2 - j) * ss_tok]"),
    ("has_init_ignored",
     "int use_prior = conv_states && has_initial_state && has_initial_state[i];",
     "int use_prior = conv_states != 0;"),
    ("writeback_off_by_one", "= u_bits[L + j];", "= u_bits[L + j - 1];"),
    ("zero_length_rewrites_state", "if (L == 0) continue;", ""),
    ("pad_not_skipped_fwd", "if (line == pad_slot_id) continue;\n        int start",
     "int start"),
    ("decode_no_shift", "= u_bits[1 + j];", "= u_bits[j];"),
    ("decode_reads_x_wrong_token", "x[b * xs_b + c * xs_d + t * xs_t]",
     "x[b * xs_b + c * xs_d]"),
    ("paged_intra_boundary", "if (row >= query_start[t])", "if (row > query_start[t])"),
    ("paged_window_offset", "positions[t] - (W - 1) + iw", "positions[t] - W + iw"),
    ("paged_head_dropped", "head * cs_h +", "0 * cs_h +"),
    ("paged_block_offset", "(src % N) * cs_n", "((src + 1) % N) * cs_n"),
    ("paged_residual_row", "if (residual) acc = acc + bf16_to_f32(x[(int64_t)t * xs_t + c]);",
     "if (residual) acc = acc + bf16_to_f32(x[(int64_t)(t > 0 ? t - 1 : 0) * xs_t + c]);"),
    ("paged_insert_no_stream_offset", "(slot % N) * cs_n + off_s + c % ws] =",
     "(slot % N) * cs_n + c % ws] ="),
    ("paged_pad_not_masked", "int real = slot_mapping[t] >= 0;", "int real = 1;"),
    ("paged_block_not_clamped", "if (lblk > max_blocks - 1) lblk = max_blocks - 1;", ""),
    ("paged_pad_row_tap_zeroed", "v = bf16_to_f32(x[row * xs_t + c]);",
     "v = slot_mapping[row] >= 0 ? bf16_to_f32(x[row * xs_t + c]) : 0.0f;"),
    ("metadata_strict", "if (query_start_loc[j] <= t) owner = j;",
     "if (query_start_loc[j] < t) owner = j;"),
    ("spec_offset_is_count", "num_accepted_tokens[b] - 1 : 0", "num_accepted_tokens[b] : 0"),
    ("spec_window_lags", "uint16_t v = u_bits[t + 1 + j];", "uint16_t v = u_bits[t + j];"),
    ("spec_never_shifts", "const int shift = inter == NULL && out_state_idx == NULL;",
     "const int shift = 0;"),
    ("spec_output_column_shifted", "conv_state[o * ss_line + c * ss_dim + j * ss_tok] = v;",
     "conv_state[o * ss_line + c * ss_dim + (j + 1) * ss_tok] = v;"),
    ("update_bias_dropped", "float bc = bias ? bf16_to_f32(bias[c]) : 0.0f;", "float bc = 0.0f;"),
    ("silu_ignores_flag", "if (silu) acc = silu_f32(acc);", "acc = silu_f32(acc);"),
    ("metadata_pad_rows_take_last_request",
     "            seq_idx_out[t] = 0;\n            query_start_out[t] = 0;",
     "            seq_idx_out[t] = num_reqs - 1;\n            query_start_out[t] = 0;"),
    ("decode_pad_counted_as_error",
     "        if (line == pad_slot_id) continue;\n        if (line < 0 || line >= num_cache_lines) {",
     "        if (line < 0 || line >= num_cache_lines) {"),
    ("paged_taps_reversed", "weight[c * ws_c + iw * ws_w]", "weight[c * ws_c + (W - 1 - iw) * ws_w]"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_kill_mutant(tmp_path, name, old, new):
    src = open(oracle_build.SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c_file = tmp_path / f"{name}.c"
    c_file.write_text(mutated)
    lib = tmp_path / f"lib_{name}.so"
    oracle_build.compile_to(str(c_file), str(lib))
    env = dict(os.environ, CCV_ORACLE_LIB=str(lib), OMP_NUM_THREADS="1",
               MKL_NUM_THREADS="1")
    proc = subprocess.run(
        [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
         "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, f"mutant {name} survived the oracle pins"
