"""Pins of the oracle's Domino chain decoder (``orc_chain``), CPU only.

What fixes the chain independently of its own code:
* W2 = 0: the correction vanishes, so greedy tokens are numpy's argmax of each
  depth's base logits and lp is the full-vocabulary log-softmax there (the GRU
  then has no effect on the tokens);
* W2 = 0, T > 0: the sampled tokens are the inverse CDF of softmax(base / T) at
  the uniform draw (numpy's searchsorted on the cumulative sum), and a sweep of
  stratified draws hits every token in proportion to its probability;
* full model: with M = V, k = 1 and N = D the tree builder's best-first tree is
  a single chain, whose tokens and per-step score increments are the greedy
  chain's tokens and lp (the tree oracle is pinned by brute force elsewhere);
* full model, sampled: the lp of every chain token equals the tree oracle's
  full-vocabulary log-probability of that token below the same prefix, which
  that routine recomputes by replaying the GRU from the root;
* replay: forcing the chain along its own tokens changes nothing;
* degenerate inputs: an all -inf depth, NaN / +inf logits, bad temperatures.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
from scipy.special import log_softmax, softmax

import dt_workloads as W
import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def small(seed, wdtype="f32", V=300, D=5, T=0.0, **kw):
    kw = dict(dict(d=16, d_s=16, r=8, M=8, k=2, N=10, batch=2, logits="spiked", e_std=0.5), **kw)
    return W.custom_workload(V=V, D=D, wdtype=wdtype, seed=seed, temperature=T, **kw)


def test_zero_correction_greedy_is_base_argmax():
    wl = small(61, T=0.0)
    wl = dataclasses.replace(wl, W2=np.zeros_like(wl.W2))
    for b in range(wl.batch):
        o = oracle.chain(wl, b)
        assert o["status"] == 0
        base = wl.base_logits[b].astype(np.float64)
        np.testing.assert_array_equal(o["tokens"], np.argmax(base, axis=1))
        want_lp = log_softmax(base, axis=1)[np.arange(wl.D), o["tokens"]]
        np.testing.assert_allclose(o["lp"], want_lp, atol=2e-6, rtol=0)
        top2 = np.sort(base, axis=1)[:, -2:]
        np.testing.assert_allclose(o["margin"], top2[:, 1] - top2[:, 0], atol=1e-6, rtol=0)


@pytest.mark.parametrize("T", [0.5, 1.0, 1.7])
def test_zero_correction_sampled_is_inverse_cdf(T):
    wl = small(62, T=T, batch=3)
    wl = dataclasses.replace(wl, W2=np.zeros_like(wl.W2))
    u = W.chain_uniforms(wl.batch, wl.D, seed=62)
    for b in range(wl.batch):
        o = oracle.chain(wl, b, uniforms=u)
        assert o["status"] == 0
        x = (wl.base_logits[b].astype(np.float64) / T).astype(np.float32).astype(np.float64)
        for i in range(wl.D):
            c = np.cumsum(np.exp(x[i] - x[i].max()))
            tok = int(np.searchsorted(c, u[b, i] * c[-1], side="right"))
            assert o["tokens"][i] == tok
            assert abs(o["lp"][i] - log_softmax(x[i])[tok]) < 2e-6


def test_stratified_draws_follow_softmax():
    """Depth 1 depends on the anchor only: sweeping u over K strata must hit each
    token about K p_v times (inverse-CDF sampling puts the strata in order)."""
    V, T, K = 40, 0.8, 4000
    wl = small(63, V=V, D=1, T=T, M=4, k=1, N=1, batch=1)
    wl = dataclasses.replace(wl, W2=np.zeros_like(wl.W2))
    p = softmax(wl.base_logits[0, 0].astype(np.float64) / T)
    counts = np.zeros(V)
    for j in range(K):
        o = oracle.chain(wl, 0, uniforms=np.array([[(j + 0.5) / K]], np.float32))
        counts[o["tokens"][0]] += 1
    assert np.abs(counts - K * p).max() <= 1.5


@pytest.mark.parametrize("wdtype", ["f32", "bf16"])
def test_greedy_chain_is_the_k1_full_vocabulary_tree(wdtype):
    V, D = 256, 6
    wl = small(64, wdtype=wdtype, V=V, D=D, T=0.0, M=V, k=1, N=D, batch=2, d=24, d_s=24, r=16,
               logits="zipf", zipf=(0.9, 1.3))
    for b in range(wl.batch):
        tree = oracle.build_tree(wl, b)
        o = oracle.chain(wl, b)
        assert tree["status"] == 0 and o["status"] == 0
        np.testing.assert_array_equal(tree["parents"][1:], np.arange(D))
        np.testing.assert_array_equal(tree["tokens"][1:], o["tokens"])
        inc = np.diff(tree["scores"].astype(np.float64))
        np.testing.assert_allclose(inc, o["lp"], atol=1e-5, rtol=0)


@pytest.mark.parametrize("T", [0.6, 1.3])
def test_sampled_chain_lp_matches_tree_children(T):
    V, D = 200, 5
    wl = small(65, wdtype="bf16", V=V, D=D, T=T, M=V, k=3, N=10, batch=2, d=16, d_s=24, r=16,
               logits="zipf", zipf=(0.9, 1.3))
    u = W.chain_uniforms(wl.batch, D, seed=65)
    for b in range(wl.batch):
        o = oracle.chain(wl, b, uniforms=u)
        assert o["status"] == 0
        for i in range(D):
            _, _, all_lp, cand = oracle.children(wl, o["tokens"][:i], b)
            pos = int(np.nonzero(cand == o["tokens"][i])[0][0])
            assert abs(all_lp[pos] - o["lp"][i]) < 1e-6


def test_forced_replay():
    wl = small(66, T=0.9, batch=1)
    u = W.chain_uniforms(1, wl.D, seed=66)
    free = oracle.chain(wl, 0, uniforms=u)
    again = oracle.chain(wl, 0, uniforms=u, forced=free["tokens"])
    for key in ("decided", "tokens", "lp", "margin"):
        np.testing.assert_array_equal(again[key], free[key])
    other = (free["tokens"] + 1) % wl.V
    f = oracle.chain(wl, 0, uniforms=u, forced=other)
    np.testing.assert_array_equal(f["tokens"], other)
    assert f["decided"][0] == free["decided"][0]    # depth 1 depends on the anchor only


def test_degenerate_inputs():
    wl = small(67, T=0.0, batch=1)
    base = wl.base_logits.copy()
    base[0, 2, :] = -np.inf
    o = oracle.chain(dataclasses.replace(wl, base_logits=base), 0)
    assert o["status"] == 0 and o["decided"][2] == 0 and np.isneginf(o["lp"][2])
    assert np.isfinite(o["lp"][[0, 1, 3, 4]]).all()
    base[0, 1, 7] = np.nan
    assert oracle.chain(dataclasses.replace(wl, base_logits=base), 0)["status"] == oracle.ENONFINITE
    base = wl.base_logits.copy()
    base[0, 0, 3] = np.inf
    assert oracle.chain(dataclasses.replace(wl, base_logits=base), 0)["status"] == oracle.ENONFINITE
    for T in (-1.0, np.inf):
        wt = dataclasses.replace(wl, temperature=np.array([T], np.float32))
        assert oracle.chain(wt, 0)["status"] == oracle.EINVAL


def test_uniform_clamping():
    """u >= 1 takes the last token with mass, u < 0 and NaN read as 0."""
    wl = small(68, V=50, D=1, T=1.0, M=4, k=1, N=1, batch=1)
    wl = dataclasses.replace(wl, W2=np.zeros_like(wl.W2))
    p = softmax(wl.base_logits[0, 0].astype(np.float64))
    first = int(np.nonzero(p > 0)[0][0])
    last = int(np.nonzero(p > 0)[0][-1])
    for u, want in ((0.0, first), (-3.0, first), (np.nan, first), (1.0, last), (7.0, last)):
        o = oracle.chain(wl, 0, uniforms=np.array([[u]], np.float32))
        assert o["tokens"][0] == want, (u, o["tokens"][0], want)


def test_temperature_half_equals_doubled_logits_and_w2():
    """x = (L_base + W2 h) / T: T = 0.5 and T = 1 with L_base and W2 doubled give
    the same x exactly (scaling by 2 is exact), so the same chains bit for bit."""
    wl = small(69, T=0.5, batch=2)
    u = W.chain_uniforms(2, wl.D, seed=69)
    doubled = dataclasses.replace(wl, base_logits=wl.base_logits * 2, W2=wl.W2 * 2,
                                  temperature=np.ones(2, np.float32))
    for b in range(2):
        a, c = oracle.chain(wl, b, uniforms=u), oracle.chain(doubled, b, uniforms=u)
        for key in ("tokens", "lp", "margin"):
            np.testing.assert_array_equal(a[key], c[key])


def test_greedy_ties_take_the_lowest_id():
    wl = small(70, T=0.0, batch=1)
    wl = dataclasses.replace(wl, W2=np.zeros_like(wl.W2))
    base = wl.base_logits.copy()
    base[0, :, :] = -5.0
    base[0, :, [11, 40, 3]] = 2.0            # three tied maxima per depth
    o = oracle.chain(dataclasses.replace(wl, base_logits=base), 0)
    assert (o["tokens"] == 3).all() and (o["margin"] == 0).all()
