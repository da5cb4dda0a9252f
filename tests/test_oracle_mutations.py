"""Planted mistakes in the oracle fail its pins (CPU only).

Each case copies the oracle's C source, makes one plausible slip by a textual
substitution, compiles the copy with gcc and runs one pin against that library;
the pin must fail. The oracle source itself carries no hook for this.
"""
from __future__ import annotations

import importlib
import subprocess

import pytest

import oracle

CASES = [
    # name, fragment of the oracle, slip, pin module, pin, pin arguments
    ("gru-n-gate-without-r", "(double)r * ((double)gh[2] + bh[2])", "((double)gh[2] + bh[2])",
     "test_oracle_pins", "test_gru_matches_torch_grucell", ("f32", True)),
    ("gru-z-roles-swapped", "(1.0 - (double)z) * (double)n + (double)z * (double)s[i]",
     "(double)z * (double)n + (1.0 - (double)z) * (double)s[i]",
     "test_oracle_pins", "test_gru_matches_torch_grucell", ("f32", True)),
    ("tree-depth-offset", "c->q->base + (size_t)(j - 1) * m->V;",
     "c->q->base + (size_t)(j < m->D ? j : j - 1) * m->V;",
     "test_oracle_pins", "test_scores_match_torch_rescoring", ("bf16-bias-state0-T",)),
    ("tree-relu-for-silu", "c->h[t] = (float)(a * sigmoid64(a));",
     "c->h[t] = (float)(a > 0 ? a : 0);",
     "test_oracle_pins", "test_scores_match_torch_rescoring", ("tiny-config",)),
    ("tree-without-temperature", "(double)dl) / (double)c->Teff);", "(double)dl));",
     "test_oracle_pins", "test_temperature_half_equals_doubled_logits_and_w2", ()),
    ("heap-tie-break-reversed", "return a->seq < b->seq;", "return a->seq > b->seq;",
     "test_oracle_pins", "test_exact_ties_follow_push_order", ()),
    ("chain-depth-offset", "const float *base = q->base + (size_t)i * V;",
     "const float *base = q->base + (size_t)(i + 1 < m->D ? i + 1 : i) * V;",
     "test_oracle_chain", "test_zero_correction_greedy_is_base_argmax", ()),
    ("chain-relu-for-silu", "      h[t] = (float)(a * sigmoid64(a));",
     "      h[t] = (float)(a > 0 ? a : 0);",
     "test_oracle_chain", "test_greedy_chain_is_the_k1_full_vocabulary_tree", ("f32",)),
    ("chain-gru-fed-the-anchor", "      embed(m, t, x);", "      embed(m, q->anchor, x);",
     "test_oracle_chain", "test_greedy_chain_is_the_k1_full_vocabulary_tree", ("f32",)),
    ("chain-lp-without-logz", "lp[i] = (mx == -INFINITY) ? -INFINITY : (float)((double)xv[t] - (mx + log(Z)));",
     "lp[i] = (mx == -INFINITY) ? -INFINITY : (float)((double)xv[t] - mx);",
     "test_oracle_chain", "test_sampled_chain_lp_matches_tree_children", (0.6,)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_fails_a_pin(case, tmp_path, monkeypatch):
    name, before, after, module, func, args = case
    src = open(oracle._SRC).read()
    assert src.count(before) == 1, f"{name}: fragment not unique"
    c_file = tmp_path / "dt_oracle_slip.c"
    c_file.write_text(src.replace(before, after))
    so = tmp_path / "liboracle_slip.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so),
                           str(c_file), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.load(str(so)))
    pin = getattr(importlib.import_module(module), func)
    with pytest.raises(Exception):
        pin(*args)


def test_unmutated_oracle_passes_the_same_pins():
    """The control: the same pins pass on the oracle as built."""
    oracle.build()
    for _, _, _, module, func, args in CASES:
        getattr(importlib.import_module(module), func)(*args)
