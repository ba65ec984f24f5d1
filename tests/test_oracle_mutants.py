"""The oracle's pins must be sensitive: plant plausible mistakes in a copy of the
oracle's C source (on the CPU), rebuild it, and check that the pins catch each one.
"""
import os
import subprocess
import tempfile
import types

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("gate_without_exp_A", "exp(-exp(A_h) * z)", "exp(-A_h * z)"),
    ("gate_sign", "g_min / (1.0 + exp(-exp(A_h) * z))", "g_min / (1.0 + exp(exp(A_h) * z))"),
    ("delta_sign", "u[j] = beta * ((v ? v[j] : 0.0) - acc);", "u[j] = beta * (acc - (v ? v[j] : 0.0));"),
    ("write_without_beta", "u[j] = beta * ((v ? v[j] : 0.0) - acc);", "u[j] = ((v ? v[j] : 0.0) - acc);"),
    ("transposed_read", "acc += S[c * w + j] * q[c];", "acc += S[(j % dk) * w + (c % w)] * q[c];"),
    ("decay_after_write",
     "    for (int c = 0; c < dk; ++c)\n        for (int j = 0; j < w; ++j)\n            S[c * w + j] *= alpha[c];\n    for (int j = 0; j < w; ++j) {",
     "    for (int j = 0; j < w; ++j) {"),
    ("chunk_exclusive_decay", "a[r * dk + i] = exp(G[r * dk + i]);",
     "a[r * dk + i] = exp(G[r * dk + i] - oracle_gate(c->g_min, c->A[h], c->z[((t0 + r) * H + h) * dk + i]));"),
    ("chunk_strict_mqk", "Mqk[r * C + s] = (s <= r) ? qk : 0.0;", "Mqk[r * C + s] = (s < r) ? qk : 0.0;"),
    ("chunk_restore_from_kdecay", "Kr[r * dk + i] = aC[i] * Ki[r * dk + i];", "Kr[r * dk + i] = aC[i] * Kd[r * dk + i];"),
    ("chunk_inverse_sign", "acc -= L[r * C + s] * INV[s * C + col];", "acc += L[r * C + s] * INV[s * C + col];"),
    ("pair_no_reset_of_M", "            memset(M, 0, sizeof(double) * (size_t)dk * dk);\n            if (init_state)",
     "            if (init_state)"),
    ("compose_swapped", "acc += M2[i * dk + r] * S1[r * dv + j];", "acc += M1[i * dk + r] * S2[r * dv + j];"),
    ("decode_replay_one_more", "for (int64_t j = 0; j < nacc; ++j) {", "for (int64_t j = 0; j <= nacc && j < W - 1; ++j) {"),
    ("decode_drafts_from_stale_state", "memcpy(Sd, S, sizeof(double) * (size_t)dk * dv);",
     "memcpy(Sd, c->state + (b * H + h) * (int64_t)dk * dv, sizeof(double) * (size_t)dk * dv);\n    for (int64_t i0 = 0; i0 < (int64_t)dk * dv; ++i0) Sd[i0] *= 0.5;"),
]

PIN_TESTS = [
    pins.test_gate_special_values_and_symmetry,
    pins.test_gate_bounds_match_pages,
    pins.test_beta_zero_is_pure_channel_decay,
    lambda: pins.test_recurrence_equals_dense_transition_products(5),
    lambda: pins.test_wy_and_ut_match_brute_force(7),
    lambda: pins.test_chunk_form_equals_recurrence(16),
    lambda: pins.test_segment_composition_equals_unsplit(False),
    lambda: pins.test_segment_composition_equals_unsplit(True),
    pins.test_composition_associative_not_commutative,
    pins.test_document_start_inside_segment_resets_pair,
    pins.test_delta_rule_recalls_orthonormal_keys,
    pins.test_decode_replay_equals_committed_stream,
]


def _build(src_text, out_dir, name):
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", so, c,
                           "-lpthread", "-lm"])
    return so


def _caught(so):
    with oracle.use_library(so):
        for t in PIN_TESTS:
            try:
                t()
            except (AssertionError, ValueError, FloatingPointError):
                return True
    return False


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} not found"
    with tempfile.TemporaryDirectory() as d:
        so = _build(src.replace(old, new, 1), d, name)
        assert _caught(so), f"no pin fails for planted mistake {name}"


def test_unmutated_copy_passes_all_pins():
    with tempfile.TemporaryDirectory() as d:
        so = _build(open(SRC).read(), d, "clean")
        assert not _caught(so)


# The fused decode step's convolution and output norm are numpy code in the
# oracle's package: the same check, with the mistakes planted in a copy of that
# module's source.
PY_MUTANTS = [
    ("conv_taps_reversed", "y = y + w[..., None, :, j] * s[..., j:j + n, :]",
     "y = y + w[..., None, :, CONV_WIDTH - 1 - j] * s[..., j:j + n, :]"),
    ("conv_without_history", "s = np.concatenate([hist, x], axis=-2)", "s = np.concatenate([0.0 * hist, x], axis=-2)"),
    ("conv_silu_dropped", "y = y / (1.0 + np.exp(-y))", "y = y"),
    ("conv_state_one_token_early", "cs[b, :, i] = full[:, n + 1:n + 4]", "cs[b, :, i] = full[:, n:n + 3]"),
    ("replay_from_window_inputs", "stream = np.concatenate([cx[b, :n], x[b]])",
     "stream = np.concatenate([x[b, 1:n + 1], x[b]])"),
    ("norm_sum_not_mean", "np.mean(o * o, axis=-1, keepdims=True)", "np.sum(o * o, axis=-1, keepdims=True)"),
    ("norm_over_heads", "np.mean(o * o, axis=-1, keepdims=True)", "np.mean(o * o, axis=-2, keepdims=True)"),
    ("eps_outside_root", "np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)",
     "(np.sqrt(np.mean(o * o, axis=-1, keepdims=True)) + eps)"),
    ("gate_without_sigmoid", "return o * r * w / (1.0 + np.exp(-gate))", "return o * r * w * gate"),
    ("norm_without_weight", "return o * r * w / (1.0 + np.exp(-gate))", "return o * r / (1.0 + np.exp(-gate))"),
    ("input_options_before_conv", "yq, yk, bb = input_prep(yq, yk, bb, qk_l2norm, beta_sigmoid, q_scale=q_scale)",
     "_, _, bb = input_prep(yq, yk, bb, qk_l2norm, beta_sigmoid, q_scale=q_scale)"),
    ("q_scale_inverted", "q = q / np.sqrt(q.shape[-1])", "q = q * np.sqrt(q.shape[-1])"),
    ("q_scale_on_k", "q = q / np.sqrt(q.shape[-1])", "k = k / np.sqrt(k.shape[-1])"),
    ("q_scale_before_norm", """    if qk_l2norm:
        q = q / np.sqrt(np.sum(q * q, axis=-1, keepdims=True) + eps)
        k = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + eps)
    if q_scale:
        q = q / np.sqrt(q.shape[-1])""", """    if q_scale:
        q = q / np.sqrt(q.shape[-1])
    if qk_l2norm:
        q = q / np.sqrt(np.sum(q * q, axis=-1, keepdims=True) + eps)
        k = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + eps)"""),
]

PY_PIN_TESTS = [
    pins.test_short_conv_equals_numpy_convolve,
    pins.test_short_conv_silu_closed_forms,
    pins.test_gated_output_norm_invariants,
    pins.test_fused_decode_with_unit_conv_is_plain_decode,
    pins.test_fused_decode_equals_convolved_committed_stream,
    pins.test_fused_decode_output_is_normalised_prenorm,
    pins.test_input_prep_q_scale_closed_forms,
]
PY_FUNCS = ("short_conv", "rms_norm_gated", "decode_step_fused", "input_prep")


def _py_caught(monkeypatch, src_text):
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = oracle.__file__
    exec(compile(src_text, oracle.__file__, "exec"), mod.__dict__)
    for f in PY_FUNCS:
        monkeypatch.setattr(oracle, f, getattr(mod, f))
    for t in PY_PIN_TESTS:
        try:
            t()
        except (AssertionError, ValueError, FloatingPointError):
            return True
    return False


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_fused_pins_catch_planted_mistake(monkeypatch, name, old, new):
    src = open(oracle.__file__).read()
    assert old in src, f"mutation anchor for {name} not found"
    assert _py_caught(monkeypatch, src.replace(old, new, 1)), f"no pin fails for planted mistake {name}"


def test_unmutated_python_copy_passes_fused_pins(monkeypatch):
    assert not _py_caught(monkeypatch, open(oracle.__file__).read())
