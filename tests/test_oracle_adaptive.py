"""Pins of the oracle's cost-aware adaptive budget (CondAdaptive), CPU only.

* the incremental rule equals the argmax, over every prefix length n, of the
  throughput A(n) / C(n) evaluated in exact rational arithmetic from the same
  fp64 exponentials (lowest n on ties): the rule is "stop where throughput
  peaks", not an accident of its incremental form;
* limits: a negligible per-node cost keeps every node (saturation at the
  budget), a huge one keeps none;
* truncation keeps a valid tree: the first rows unchanged, the mask's ancestor
  closure intact, later rows empty.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import dt_workloads as W
import oracle


def trees(seed, N=40, batch=3):
    wl = W.custom_workload(V=500, d=16, d_s=16, r=8, D=6, M=8, k=3, N=N, batch=batch,
                           wdtype="f32", seed=seed, logits="zipf", zipf=(0.8, 1.6))
    return oracle.build_trees(wl)


def throughput_argmax(scores, tokens, c_fixed, c_node):
    best, arg = None, 0
    A, C = Fraction(1), Fraction(c_fixed)
    for n in range(0, len(scores)):
        if n > 0:
            if tokens[n] < 0:
                break
            A += Fraction(float(np.exp(np.float64(scores[n]))))
            C += Fraction(c_node)
        th = A / C
        if best is None or th > best:
            best, arg = th, n
    return arg


@pytest.mark.parametrize("c_node", [1 / 512, 1 / 64, 1 / 16, 1 / 4])
def test_rule_is_the_throughput_argmax(c_node):
    for seed in (111, 112):
        for t in trees(seed):
            n = oracle.adaptive_count(t["scores"], t["tokens"], 1.0, c_node)
            assert n == throughput_argmax(t["scores"], t["tokens"], 1.0, c_node)


def test_limits():
    for t in trees(113):
        n_nodes = int((t["tokens"] >= 0).sum()) - 1
        assert oracle.adaptive_count(t["scores"], t["tokens"], 1.0, 1e-30) == n_nodes
        assert oracle.adaptive_count(t["scores"], t["tokens"], 1.0, 1e30) == 0


def test_truncation_is_a_valid_tree():
    for t in trees(114):
        n = oracle.adaptive_count(t["scores"], t["tokens"], 1.0, 1 / 32)
        cut = oracle.truncate_tree(t, n)
        for key in ("tokens", "parents", "depths", "scores"):
            np.testing.assert_array_equal(cut[key][:n + 1], t[key][:n + 1])
        assert (cut["tokens"][n + 1:] == -1).all() and np.isneginf(cut["scores"][n + 1:]).all()
        np.testing.assert_array_equal(cut["mask"][:n + 1], t["mask"][:n + 1])
        assert not cut["mask"][n + 1:].any()
        assert not cut["mask"][:n + 1, n + 1:].any()   # no kept row sees a dropped one
