"""The pins reject plausible mistakes: each test plants one mistake in a copy of the oracle (on the
CPU), builds it, and checks that the named pin fails against it while the real oracle passes."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_prefill_pins as ppins
import test_oracle_varlen_pins as vpins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (id, text in oracle.c, planted replacement, pin that must fail).  Every planted mistake keeps all
# accesses inside the test's buffers.
MUTANTS = [
    ("taps_reversed", "const float prod = wj * fullf[t + j];", "const float prod = wj * fullf[t + W - 1 - j];",
     lambda: pins.test_p2_impulse_response()),
    ("bias_dropped",
     "                float acc = a->bias ? bits_to_float(get_bits(a->bias, bf, c), bf) : 0.0f;\n"
     "                for (int j = 0; j < W; ++j) {\n"
     "                    const float wj = bits_to_float(get_bits(a->weight, bf, (int64_t)c * W + j), bf);\n"
     "                    const float prod = wj * fullf[t + j];",
     "                float acc = 0.0f;\n"
     "                for (int j = 0; j < W; ++j) {\n"
     "                    const float wj = bits_to_float(get_bits(a->weight, bf, (int64_t)c * W + j), bf);\n"
     "                    const float prod = wj * fullf[t + j];",
     lambda: pins.test_p1_matches_float64_conv1d("f32", "dense", 4)),
    ("silu_sign", "acc / (1.0f + expf(-acc));\n            }\n\n            if (a->recompute)",
     "acc / (1.0f + expf(acc));\n            }\n\n            if (a->recompute)",
     lambda: pins.test_p1_matches_float64_conv1d("f32", "dense", 3)),
    ("eps_as_norm_floor", "1.0f / sqrtf(ss + a->l2_eps)", "1.0f / fmaxf(sqrtf(ss), a->l2_eps)",
     lambda: pins.test_p3_one_hot_taps_and_constant_group()),
    ("snapshot_off_by_one", "win_index(a, s, t, c, k), full[t + 1 + k])", "win_index(a, s, t, c, k), full[t + k])",
     lambda: pins.test_p4_sequential_equals_batched_in_T("dense", "f32")),
    ("state_write_lags", "put_bits(a->state, sbf, srow + k, full[Ts + k])", "put_bits(a->state, sbf, srow + k, full[Ts - 1 + k])",
     lambda: pins.test_p11_single_token_update()),
    ("offset_ignored", "full[k] = get_bits(a->state, sbf, srow + o + k);", "full[k] = get_bits(a->state, sbf, srow + k);",
     lambda: pins.test_p10_state_offset_equals_preshifted_state()),
    ("commit_wrong_snapshot", "const int t = acc - 1;", "const int t = acc < a->T ? acc : acc - 1;",
     lambda: pins.test_p9_commit_equals_shorter_verify("dedup")),
    ("v_normalised", "g + hd <= a->qk_channels", "g + hd <= dim",
     lambda: pins.test_p8_group_norms_and_v_passthrough()),
    ("bf16_truncates", "u += 0x7fffu + keep_lsb;", "(void)keep_lsb;",
     lambda: pins.test_bf16_rounding_matches_torch()),
    ("dedup_step_uses_ch", "int64_t step = a->dedup ? a->w_col : a->w_step;", "int64_t step = a->dedup ? 0 : a->w_step;",
     lambda: pins.test_p6_dedup_view_equals_dense(4)),
    ("history_row_shifted", "srow + t + k, full[t + 1 + k])", "srow + t + k, full[t + k])",
     lambda: pins.test_h1_history_row_equals_dedup_row(3)),
    ("history_row_last_window_only", "for (int t = 0; t < Ts; ++t)\n                    for (int k = 0; k < W - 1; ++k) put_bits(a->state",
     "for (int t = Ts - 1; t < Ts; ++t)\n                    for (int k = 0; k < W - 1; ++k) put_bits(a->state",
     lambda: pins.test_h2_history_chain_equals_verify_commit_chain()),
    ("recompute_wrong_snapshot", "put_bits(a->state, bf, srow + k, full[acc + k]);",
     "put_bits(a->state, bf, srow + k, full[acc - 1 + k]);",
     lambda: pins.test_r3_recompute_commit_closed_form()),
    ("recompute_verify_writes_state", "if (a->recompute) continue; /* outputs only",
     "if (a->recompute) { put_bits(a->state, bf, srow, full[Ts]); continue; } /* outputs only",
     lambda: pins.test_r1_recompute_verify_writes_outputs_only(3, "f32")),
    ("prefill_init_ignored", "full[k] = init ? get_bits(a->state, bf, srow + k) : 0u;",
     "full[k] = get_bits(a->state, bf, srow + k);", lambda: ppins.test_pf4_no_initial_state_is_a_zero_window()),
    ("prefill_state_lags", "put_bits(a->state, bf, srow + k, full[L + k]);",
     "put_bits(a->state, bf, srow + k, full[L > 0 ? L - 1 + k : k]);",
     lambda: ppins.test_pf3_split_prompt_equals_whole()),
    ("prefill_token_offset", "full[W - 1 + t] = get_bits(a->x, bf, (int64_t)(b + t) * a->x_tok + c);",
     "full[W - 1 + t] = get_bits(a->x, bf, (int64_t)(t) * a->x_tok + c);",
     lambda: ppins.test_pf5_packed_equals_separate_and_untouched()),
    ("mixed_snapshot_truncates", "return float_to_bits(bits_to_float(v, 0), 1);", "return v >> 16;",
     lambda: pins.test_m3_fp32_inputs_round_into_bf16_snapshots()),
    ("mixed_state_read_as_x_dtype", "full[k] = get_bits(a->state, sbf, srow + o + k);\n                fullf[k] = bits_to_float(full[k], sbf);",
     "full[k] = get_bits(a->state, sbf, srow + o + k);\n                fullf[k] = bits_to_float(full[k], bf);",
     lambda: pins.test_m4_mixed_matches_float64_conv1d("bf16", "f32")),
    ("tree_parent_ignored", "const int base = (a->parent[(int64_t)s * T + t] + 1) * R;", "const int base = t * R;",
     lambda: pins.test_tr2_tree_paths_equal_chain_verifies()),
    ("tree_window_not_shifted", "wbits[nb + k] = wbits[base + k + 1];", "wbits[nb + k] = wbits[base + k];",
     lambda: pins.test_tr1_chain_parents_equal_the_plain_verify(4, "bf16")),
    ("tree_state_one_token_short", "put_bits(a->state, sbf, srow + k, wbits[T * R + k]);",
     "put_bits(a->state, sbf, srow + k, wbits[(T - 1) * R + k]);",
     lambda: pins.test_tr1_chain_parents_equal_the_plain_verify(4, "f32")),
    ("varlen_state_uses_T", "put_bits(a->state, sbf, srow + k, full[Ts + k]);",
     "put_bits(a->state, sbf, srow + k, full[T + k]);",
     lambda: vpins.test_v1_packed_equals_separate_verifies("dense", "f32")),
    ("varlen_rows_shifted", "xrow = (int64_t)b * a->x_tok;", "xrow = (int64_t)(b > 0 ? b - 1 : 0) * a->x_tok;",
     lambda: vpins.test_v3_matches_float64_conv1d(4)),
    ("varlen_snapshots_past_Ts",
     "for (int t = 0; t < Ts; ++t)\n                for (int k = 0; k < W - 1; ++k) put_bits(a->window",
     "for (int t = 0; t < T; ++t)\n                for (int k = 0; k < W - 1; ++k) put_bits(a->window",
     lambda: vpins.test_v5_untouched_regions()),
    ("varlen_commit_accept_past_Ts", "(acc < 1 || acc > Ts)) st |= 4;", "(acc < 1 || acc > a->T)) st |= 4;",
     lambda: vpins.test_v6_bad_spans_flagged_and_untouched()),
    ("varlen_empty_commit_not_skipped", "if (Ts == 0) continue; /* no draft token was verified",
     "/* mutated */ /* no draft token was verified",
     lambda: vpins.test_v4_commit_equals_shorter_verify("dedup")),
    ("padded_row_written", "if (slot < 0 || st) continue;\n\n", "if (st) continue;\n        if (slot < 0) { if (a->out) put_bits(a->out, bf, (int64_t)s * a->out_seq, 0); continue; }\n\n",
     lambda: pins.test_p7_padded_rows_untouched()),
]


@pytest.mark.parametrize("mid,old,new,pin", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_rejects_planted_mistake(tmp_path, mid, old, new, pin):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {mid} not found"
    mut = src.replace(old, new, 1)
    c = tmp_path / f"{mid}.c"
    so = tmp_path / f"{mid}.so"
    c.write_text(mut)
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"],
                   check=True)
    pin()  # the real oracle passes this pin
    prev = oracle.swap_library(str(so))
    try:
        with pytest.raises(AssertionError):
            pin()
    finally:
        oracle.swap_library(prev)
