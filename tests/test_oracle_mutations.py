"""The oracle's pins must catch plausible mistakes (no GPU).

Each case copies kda_oracle.c to a temporary directory, plants one mistake by
a textual edit (a wrong decay order, a dropped beta, a transposed read-out, a
missed reset, a wrong tap index, an off-by-one in cu_seqlens ...), compiles
the copy with gcc and checks that at least one pin from the oracle tests
fails on it. The oracle itself is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

MUTATIONS = {
    # recurrence
    "decay_after_update": ("row[j] = row[j] * decay + bk * vt[j];",
                           "row[j] = (row[j] + bk * vt[j]) * decay;"),
    "beta_dropped": ("const double bk = bt * kt[i];", "const double bk = kt[i];"),
    "readout_uses_k": ("acc += S[i * Dv + j] * qt[i];", "acc += S[i * Dv + j] * kt[i];"),
    "decay_sign": ("const double decay = exp(gt[i]);", "const double decay = exp(-gt[i]);"),
    "decay_wrong_token": ("const double *gt = J->g + (p * H + h) * Dk;",
                          "const double *gt = J->g + ((p > 0 ? p - 1 : p) * H + h) * Dk;"),
    "no_reset_between_docs": ("while (e < T && (seg ? seg[b * T + e] : 1) == s)",
                              "while (e < T && (seg ? seg[b * T + e] : 1) != 0)"),
    # per-segment state
    "initial_state_ignored": ("if (J->init && r < J->n_state)", "if (0 && J->init && r < J->n_state)"),
    "state_rank_off_by_one": ("units[5 * n_units + 4] = rank;", "units[5 * n_units + 4] = rank + 1;"),
    # delta rule
    "delta_correction_dropped": ("W[j] = vt[j] - u;", "W[j] = vt[j];"),
    "delta_correction_sign": ("W[j] = vt[j] - u;", "W[j] = vt[j] + u;"),
    "delta_no_decay": ("                    row[j] *= ei;", "                    row[j] *= 1.0;"),
    "delta_decay_sign": ("const double ei = exp(gt[i]);", "const double ei = exp(-gt[i]);"),
    "delta_beta_in_correction": ("u += S[i * Dv + j] * kt[i];", "u += S[i * Dv + j] * bt * kt[i];"),
    "delta_state_transposed": ("u += S[i * Dv + j] * kt[i];", "u += S[j * Dv + i] * kt[i];"),
    "delta_beta_dropped": ("const double wk = bt * kt[i];", "const double wk = kt[i];"),
    # gradients
    "bwd_no_adjoint_decay": ("                A[i * Dv + j] *= exp(gt[i]);",
                             "                A[i * Dv + j] *= 1.0;"),
    "bwd_dg_current_state": ("sg += A[i * Dv + j] * Sp[i * Dv + j];",
                             "sg += A[i * Dv + j] * S[i * Dv + j];"),
    "bwd_dq_no_scale": ("dqt[i] = J->scale * sq;", "dqt[i] = sq;"),
    "bwd_dv_uses_q": ("ak += A[i * Dv + j] * kt[i];", "ak += A[i * Dv + j] * qt[i];"),
    "bwd_dbeta_dropped_k": ("db += kt[i] * av;", "db += av;"),
    # conv
    "conv_tap_forward": ("const int64_t s = t - j;", "const int64_t s = t - (K - 1 - j);"),
    "conv_no_mask": ("if (seg && seg[b * T + s] != seg[b * T + t])", "if (0)"),
    # cu_seqlens
    "cu_off_by_one": ("e = (i < max_segs) ? starts[i] : N;",
                      "e = (i < max_segs) ? starts[i - 1] : N;"),
    "cu_padding_starts": ("const int is_start = seg[p] != 0 && (is_row_start || seg[p] != seg[p - 1]);",
                          "const int is_start = (is_row_start || seg[p] != seg[p - 1]);"),
}


def _build_mutant(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib_{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(path),
                    "-o", str(so), "-lm"], check=True)
    return str(so)


def _pins_pass(monkeypatch, so_path) -> bool:
    """Run a representative subset of the pins against a mutant library."""
    lib = ctypes.CDLL(so_path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.oracle_cu_seqlens.argtypes = [vp, i64, i64, i32, ctypes.c_int, ctypes.c_int, vp,
                                      ctypes.POINTER(ctypes.c_int64)]
    lib.oracle_short_conv.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp]
    lib.oracle_kda_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                   ctypes.c_double, vp, ctypes.c_int]
    lib.oracle_kda_fwd_state.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                         ctypes.c_double, vp, vp, i64, vp, ctypes.c_int]
    lib.oracle_kda_fwd_delta.argtypes = lib.oracle_kda_fwd.argtypes
    lib.oracle_kda_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                   ctypes.c_double, vp, vp, vp, vp, vp, vp, ctypes.c_int]
    monkeypatch.setattr(oracle, "_lib", lib)
    import tests.test_oracle_cu_seqlens as tc
    import tests.test_oracle_conv as tv
    import tests.test_oracle_kda as tk
    import tests.test_oracle_bwd as tb
    import tests.test_oracle_state as ts
    import tests.test_oracle_delta as td
    golden = os.path.join(os.path.dirname(tc.__file__), "golden")
    checks = [
        lambda: tc.test_worked_examples(golden),
        lambda: tc.test_matches_cumulative_length_definition("tiny"),
        lambda: tc.test_bruteforce_two_rows(),
        lambda: tc.test_overflow_merges_into_last_slot(),
        lambda: tv.test_no_segments_equals_library_conv1d(4),
        lambda: tv.test_length_one_document_and_impulse(),
        lambda: tv.test_packed_equals_concatenated_documents(),
        lambda: tk.test_closed_form_bruteforce(),
        lambda: tk.test_hand_worked_three_tokens(),
        lambda: tk.test_zero_decay_is_causal_linear_attention(),
        lambda: tk.test_scalar_channel_is_first_order_filter(),
        lambda: tk.test_length_one_documents(),
        lambda: ts.test_closed_forms_bruteforce(),
        lambda: ts.test_chaining_identity(),
        lambda: ts.test_state_slots_beyond_n_state_and_ranks(),
        lambda: tb.test_finite_differences(),
        lambda: tb.test_autograd_of_closed_form(),
        lambda: td.test_unit_keys_read_back_their_values(),
        lambda: td.test_projector_form(),
        lambda: td.test_first_token_of_a_segment_is_the_additive_rule(),
        lambda: td.test_zero_beta_writes_nothing_and_linearity_in_v(),
        lambda: td.test_segments_are_independent(),
    ]
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


def test_unmodified_copy_passes(tmp_path, monkeypatch):
    so = tmp_path / "lib_clean.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", SRC, "-o",
                    str(so), "-lm"], check=True)
    assert _pins_pass(monkeypatch, str(so))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(tmp_path, monkeypatch, name):
    so = _build_mutant(tmp_path, name)
    assert not _pins_pass(monkeypatch, so), f"planted mistake '{name}' passed every pin"
