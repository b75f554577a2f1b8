"""The oracle's pins catch plausible mistakes (CPU).

Each case plants one mistake in a scratch copy of ``oracle/kda_oracle.c`` (a
wrong clamp, a flipped sign, a dropped term, q and k swapped, a non-strict
mask, ...), builds it into a temporary library, points the ``oracle`` module at
it, and runs the pins of ``test_oracle.py`` against it: at least one pin must
fail.  The unmodified copy, built the same way, must pass them all, so a
failure is the mistake's and not the harness's.  No mutation changes an index
range, so a mutated build cannot read or write out of bounds.
"""
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle as pins
import test_oracle_bwd as bwd_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, original text, planted text): each original occurs exactly once
MUTATIONS = [
    ("clamp on the wrong side",
     "return la < lower_bound ? lower_bound : la;", "return la > lower_bound ? lower_bound : la;"),
    ("softplus sign", "return pos + log1p(exp(-fabs(x)));", "return pos + log1p(exp(fabs(x)));"),
    ("A_log used without exp", "double la = -exp(A_log) * softplus(g + dt_bias);",
     "double la = -A_log * softplus(g + dt_bias);"),
    ("dt_bias dropped", "double la = -exp(A_log) * softplus(g + dt_bias);",
     "double la = -exp(A_log) * softplus(g);"),
    ("decay dropped", "for (int64_t j = 0; j < V; ++j) S[c * V + j] *= a[c];",
     "for (int64_t j = 0; j < V; ++j) S[c * V + j] *= 1.0;"),
    ("initial state ignored", "S[i] = P->h0.p ? src_get(P->h0, sbase + i) : 0.0;", "S[i] = 0.0;"),
    ("erase sign", "(src_get(P->v, v_row + j) - P->erase * r[j])",
     "(src_get(P->v, v_row + j) + P->erase * r[j])"),
    ("beta dropped", "r[j] = b * (src_get", "r[j] = 1.0 * (src_get"),
    ("q read as the erase key",
     "const double kc = src_get(P->k, qk_row + c);\n            for (int64_t j = 0; j < V; ++j) r[j]",
     "const double kc = src_get(P->q, qk_row + c);\n            for (int64_t j = 0; j < V; ++j) r[j]"),
    ("k read as the query", "const double qc = src_get(P->q, qk_row + c);",
     "const double qc = src_get(P->k, qk_row + c);"),
    ("scale dropped", "for (int64_t j = 0; j < V; ++j) o[j] *= P->scale;",
     "for (int64_t j = 0; j < V; ++j) o[j] *= 1.0;"),
    ("non-strict A mask", "Al[i * c + j] = (j < i) ?", "Al[i * c + j] = (j <= i) ?"),
    ("strict output mask", "Ql[i * c + j] = (j <= i) ? sqk : 0.0;",
     "Ql[i * c + j] = (j < i) ? sqk : 0.0;"),
    ("forward-substitution sign", "s -= Al[i * c + l] * Tl[l * c + j];",
     "s += Al[i * c + l] * Tl[l * c + j];"),
    ("W without the in-chunk decay", "* k[l * ldk + ch] * exp(Gl[l * K + ch]);",
     "* k[l * ldk + ch];"),
    ("chunk-end decay from the first token", "gam[ch] = exp(Gl[(c - 1) * K + ch]);",
     "gam[ch] = exp(Gl[ch]);"),
    ("l2norm without the square root", "const double inv = 1.0 / sqrt(ss + eps);",
     "const double inv = 1.0 / (ss + eps);"),
    ("l2norm over the first channel only", "for (int64_t c = 0; c < D; ++c) ss += row[c] * row[c];",
     "for (int64_t c = 0; c < 1; ++c) ss += row[c] * row[c];"),
    ("bwd: sign of the erase-key gradient", "dr[j] = -b * du[j];", "dr[j] = b * du[j];"),
    ("bwd: decay not carried back", "dS[c * V + j] *= alpha[c];", "dS[c * V + j] *= 1.0;"),
    ("bwd: clamp mask inverted", "const double dpre = pre[c] >= P->lower_bound ? dla : 0.0;",
     "const double dpre = pre[c] >= P->lower_bound ? 0.0 : dla;"),
    ("bwd: softplus derivative dropped", "const double dx = -a * dpre * sigmoid(xg[c]);",
     "const double dx = -a * dpre;"),
    ("bwd: dq from the state before the write", "s += Scur[c * V + j] * dov[j];",
     "s += St[c * V + j] * dov[j];"),
]

PINS = [
    ("gate vs torch softplus", pins.test_gate_matches_torch_softplus),
    ("gate special values", pins.test_gate_special_values),
    ("single-token closed form", pins.test_single_token_closed_form),
    ("brute force T=5", lambda m: pins.test_brute_force(m, 5)),
    ("exact rational", pins.test_exact_rational),
    ("beta = 0 pure decay", pins.test_beta_zero_is_pure_decay),
    ("state orientation", pins.test_state_orientation),
    ("orthonormal overwrite", pins.test_orthonormal_overwrite),
    ("strong decay", pins.test_strong_decay_forgets),
    ("linear-attention limits", pins.test_linear_attention_limits),
    ("chunked = recurrent C=7", lambda m: pins.test_chunked_equals_recurrent(m, 7)),
    ("chunked = recurrent C=64", lambda m: pins.test_chunked_equals_recurrent(m, 64)),
    ("state passing", pins.test_state_passing_equals_one_call),
    ("affine state map", pins.test_final_state_affine_in_initial_state),
    ("packed = separate", pins.test_packed_equals_separate),
    ("chunk-stage identities", pins.test_chunk_stage_identities),
    ("l2norm closed form", pins.test_l2norm_closed_form),
    ("l2norm scale-free rows", pins.test_l2norm_is_scale_free_per_row),
    ("l2norm vs brute force", pins.test_l2norm_matches_brute_force),
    ("bwd directional lb=-3", lambda m: bwd_pins.test_directional_derivatives(m, -3.0)),
    ("bwd directional lb=-0.6", lambda m: bwd_pins.test_directional_derivatives(m, -0.6)),
    ("bwd elementwise Jacobian", bwd_pins.test_jacobian_elementwise_tiny),
    ("bwd beta = 0 closed form", bwd_pins.test_beta_zero_closed_form),
    ("bwd all clamped", bwd_pins.test_all_clamped_gate_has_no_gradient),
]


def _load(tmp_path, monkeypatch, text, tag):
    d = tmp_path / tag
    d.mkdir()
    src = d / "kda_oracle.c"
    src.write_text(text)
    monkeypatch.setattr(oracle, "_SRC", str(src))
    monkeypatch.setattr(oracle, "_LIB_PATH", str(d / "libkda_oracle.so"))
    monkeypatch.setattr(oracle, "_lib", None)
    oracle.lib()  # builds the scratch copy
    return oracle


def _failing_pins(m):
    failed = []
    for name, pin in PINS:
        try:
            pin(m)
        except (AssertionError, ValueError):
            failed.append(name)
    return failed


pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")


def test_unmodified_copy_passes_every_pin(tmp_path, monkeypatch):
    with open(SRC) as f:
        text = f.read()
    assert _failing_pins(_load(tmp_path, monkeypatch, text, "orig")) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, monkeypatch, name, old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation target not unique: {old!r}"
    failed = _failing_pins(_load(tmp_path, monkeypatch, text.replace(old, new), "mut"))
    print(f"\n[mutation] {name}: caught by {failed}")
    assert failed, f"no pin catches: {name}"
