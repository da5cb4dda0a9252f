"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests needs a GPU. Each one is chosen so that a plausible slip in
the oracle (a dropped gate term, a wrong sign, a transposed W1 half, an off-by-one
depth, full-vocabulary normalisation, a wrong tie-break) fails at least one:

* top-M against numpy's lexsort (a textbook routine), with ties and signed zeros;
* the GRU cell against torch.nn.GRUCell (a library routine), hand-computed steps
  and closed-form special cases;
* whole trees against brute-force enumeration of the implicit candidate tree
  (sort-based, no heap);
* W2 = 0 against a separately written factorised (DDTree-style) builder;
* k = 1 against the greedy chain computed with torch;
* every node score against float64 torch re-scoring of its path;
* temperature and per-depth shift invariances, structural invariants, edge cases.
"""
from __future__ import annotations

import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import dt_workloads as W
import oracle
from _indep import (TorchScorer, ancestor_mask, enumerate_tree, top_n_tree, weights_f64,
                    gru_cell)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(**kw):
    base = dict(name="t", V=64, d=16, d_s=8, r=8, D=4, M=6, k=3, N=20, batch=1, wdtype="f32",
                seed=11, logits="spiked", e_std=0.5)
    base.update(kw)
    return W.custom_workload(**base)


# ------------------------------------------------------------------ top-M

@pytest.mark.parametrize("V,M,seed", [(1, 1, 0), (7, 3, 1), (64, 64, 2), (1000, 16, 3),
                                      (151936, 256, 4)])
def test_topm_matches_lexsort(V, M, seed):
    rng = np.random.default_rng(seed)
    row = rng.integers(-4, 5, size=V).astype(np.float32)     # many exact ties
    row[rng.integers(0, V, size=max(1, V // 10))] = -0.0      # signed zeros tie with +0
    row[rng.integers(0, V, size=max(1, V // 50))] = -np.inf
    ref = np.lexsort((np.arange(V), -row.astype(np.float64)))[:M]
    np.testing.assert_array_equal(oracle.topm(row, M), ref)


def test_topm_rejects_nan_and_posinf():
    row = np.zeros(10, np.float32)
    row[3] = np.nan
    with pytest.raises(ValueError):
        oracle.topm(row, 2)
    row[3] = np.inf
    with pytest.raises(ValueError):
        oracle.topm(row, 2)


# --------------------------------------------------------------- GRU cell

@pytest.mark.parametrize("wdtype,bias", [("f32", False), ("f32", True), ("bf16", True)])
def test_gru_matches_torch_grucell(wdtype, bias):
    rng = np.random.default_rng(5)
    d, d_s = 24, 12
    W_ih = rng.standard_normal((3 * d_s, d)).astype(np.float32) / 4
    W_hh = rng.standard_normal((3 * d_s, d_s)).astype(np.float32) / 3
    if wdtype == "bf16":
        W_ih, W_hh = W.f32_to_bf16_bits(W_ih), W.f32_to_bf16_bits(W_hh)
    b_ih = rng.standard_normal(3 * d_s).astype(np.float32) if bias else None
    b_hh = rng.standard_normal(3 * d_s).astype(np.float32) if bias else None
    x = rng.standard_normal(d).astype(np.float32)
    s = np.tanh(rng.standard_normal(d_s)).astype(np.float32)
    got = oracle.gru_step(W_ih, W_hh, x, s, b_ih, b_hh, wdtype=wdtype)
    dec = (lambda a: W.bf16_bits_to_f32(a)) if wdtype == "bf16" else (lambda a: a)
    Wt = dict(W_ih=torch.tensor(dec(W_ih), dtype=torch.float64),
              W_hh=torch.tensor(dec(W_hh), dtype=torch.float64),
              b_ih=None if b_ih is None else torch.tensor(b_ih, dtype=torch.float64),
              b_hh=None if b_hh is None else torch.tensor(b_hh, dtype=torch.float64))
    cell = gru_cell(Wt, d, d_s)
    with torch.no_grad():
        ref = cell(torch.tensor(x, dtype=torch.float64)[None],
                   torch.tensor(s, dtype=torch.float64)[None])[0].numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=2e-7)


def test_gru_hand_computed_2x2():
    g = json.load(open(os.path.join(GOLDEN, "gru_hand_2x2.json")))
    val = {"ln3": math.log(3.0), "4ln2": 4 * math.log(2.0), "2ln3": 2 * math.log(3.0)}
    gate = {"r": 0, "z": 1, "n": 2}
    W_ih = np.zeros((6, 2), np.float32)
    W_hh = np.zeros((6, 2), np.float32)
    for gname, unit, col, v in g["nonzero_W_ih"]:
        W_ih[gate[gname] * 2 + unit, col] = val[v]
    for gname, unit, col, v in g["nonzero_W_hh"]:
        W_hh[gate[gname] * 2 + unit, col] = val[v]
    got = oracle.gru_step(W_ih, W_hh, np.array(g["x"], np.float32), np.array(g["s"], np.float32))
    np.testing.assert_allclose(got, g["expected"], rtol=0, atol=1e-6)


def test_gru_closed_forms():
    rng = np.random.default_rng(6)
    d, d_s = 10, 7
    x = rng.standard_normal(d).astype(np.float32)
    s = rng.uniform(-1, 1, d_s).astype(np.float32)
    Z_ih, Z_hh = np.zeros((3 * d_s, d), np.float32), np.zeros((3 * d_s, d_s), np.float32)
    # all-zero weights and biases: r = z = 1/2, n = 0, so s' = s/2 exactly
    np.testing.assert_array_equal(oracle.gru_step(Z_ih, Z_hh, x, s), s * np.float32(0.5))
    # update gate saturated open (b_iz = +40): s' = s
    b = np.zeros(3 * d_s, np.float32)
    b[d_s:2 * d_s] = 40.0
    np.testing.assert_allclose(oracle.gru_step(Z_ih, Z_hh, x, s, b_ih=b), s, atol=1e-7)
    # only W_in nonzero: s' = tanh(W_in x)/2 + s/2
    W_ih = Z_ih.copy()
    W_ih[2 * d_s:] = rng.standard_normal((d_s, d)).astype(np.float32) / 3
    want = 0.5 * np.tanh(W_ih[2 * d_s:].astype(np.float64) @ x) + 0.5 * s
    np.testing.assert_allclose(oracle.gru_step(W_ih, Z_hh, x, s), want, atol=2e-7)
    # only W_hn nonzero: r = 1/2 scales the recurrent half of n
    W_hh = Z_hh.copy()
    W_hh[2 * d_s:] = rng.standard_normal((d_s, d_s)).astype(np.float32)
    want = 0.5 * np.tanh(0.5 * (W_hh[2 * d_s:].astype(np.float64) @ s)) + 0.5 * s
    np.testing.assert_allclose(oracle.gru_step(Z_ih, W_hh, x, s), want, atol=2e-7)


# ------------------------------------------------------ brute-force search

def brute_force(w, N, b=0):
    def kids(path):
        toks, lps, _, _ = oracle.children(w, list(path), b)
        return toks, lps
    enum = enumerate_tree(w.D, w.k, kids)
    t = top_n_tree(N, *enum)
    t["tokens"][0] = int(w.anchor[b])
    return t


def assert_same_tree(o, t, N, exact_scores=True):
    np.testing.assert_array_equal(o["tokens"], t["tokens"])
    np.testing.assert_array_equal(o["parents"], t["parents"])
    np.testing.assert_array_equal(o["depths"], t["depths"])
    if exact_scores:
        np.testing.assert_array_equal(o["scores"], t["scores"])
    else:
        fin = np.isfinite(t["scores"])
        np.testing.assert_array_equal(np.isfinite(o["scores"]), fin)
        np.testing.assert_allclose(o["scores"][fin], t["scores"][fin], atol=1e-5, rtol=0)
    assert o["n_nodes"] == t["n_nodes"]


@pytest.mark.parametrize("shape", [
    dict(M=4, k=2, D=3), dict(M=8, k=2, D=5), dict(M=8, k=3, D=4), dict(M=6, k=6, D=3),
    dict(M=5, k=1, D=4), dict(M=8, k=2, D=1),
])
def test_best_first_equals_brute_force(shape):
    w = tiny(**shape, N=1)
    full = sum(shape["k"] ** j for j in range(1, shape["D"] + 1))
    for N in sorted({0, 1, 2, 5, full // 2, full, full + 3}):
        w2 = dataclasses.replace(w, N=N)
        o = oracle.build_tree(w2)
        assert o["status"] == 0
        t = brute_force(w2, N)
        assert_same_tree(o, t, N)
        np.testing.assert_array_equal(o["mask"], ancestor_mask(o["parents"], o["n_nodes"], N))


def test_best_first_equals_brute_force_tiny_config():
    """The tiny configuration itself (V=1024, D=7, M=16, k=4, N=32)."""
    w = W.make_workload(0)
    o = oracle.build_tree(w)
    t = brute_force(w, w.N)
    assert_same_tree(o, t, w.N)


def test_ties_resolve_parent_first():
    """M = k = 1: every lp is exactly 0, so all scores tie; the canonical order is
    then push order, i.e. the chain in depth order."""
    w = tiny(M=1, k=1, D=5, N=8)
    o = oracle.build_tree(w)
    assert o["n_nodes"] == 6
    np.testing.assert_array_equal(o["parents"][:6], [-1, 0, 1, 2, 3, 4])
    np.testing.assert_array_equal(o["scores"][:6], np.zeros(6, np.float32))
    assert (o["tokens"][6:] == -1).all() and np.isneginf(o["scores"][6:]).all()
    assert_same_tree(o, brute_force(w, 8), 8)


# ---------------------------------------------------- W2 = 0: factorised tree

def factorised_tree(w, N, b=0):
    """DDTree-style builder on path-independent per-depth log-probabilities:
    lp_j = log_softmax over the top-M candidates of base_j / T (torch, float64,
    rounded to float32 like every stored value)."""
    T = float(w.temperature[b]) or 1.0
    per_depth = []
    for j in range(w.D):
        base = torch.tensor(w.base_logits[b, j], dtype=torch.float64)
        C = torch.sort(base, descending=True, stable=True).indices[:w.M]
        L = (base[C].to(torch.float32).to(torch.float64) / T).to(torch.float32)
        lp = torch.log_softmax(L.to(torch.float64), 0).to(torch.float32).numpy()
        order = np.lexsort((C.numpy(), -L.numpy().astype(np.float64)))[:w.k]
        per_depth.append((C.numpy()[order], lp[order]))
    enum = enumerate_tree(w.D, w.k, lambda path: per_depth[len(path)])
    t = top_n_tree(N, *enum)
    t["tokens"][0] = int(w.anchor[b])
    return t


@pytest.mark.parametrize("zero", ["W2", "W1"])
def test_zero_correction_is_factorised(zero):
    w = tiny(M=8, k=3, D=4, N=30, V=128, seed=21)
    w = dataclasses.replace(w, **{zero: np.zeros_like(getattr(w, zero))})
    o = oracle.build_tree(w)
    assert_same_tree(o, factorised_tree(w, w.N), w.N, exact_scores=False)
    # and the GRU state no longer matters
    w2 = dataclasses.replace(w, E=w.E * 3 + 1, W_hh=-w.W_hh,
                             state0=np.ones_like(w.state0))
    o2 = oracle.build_tree(w2)
    np.testing.assert_array_equal(o["tokens"], o2["tokens"])
    np.testing.assert_array_equal(o["parents"], o2["parents"])


def test_full_config_zero_w2_factorised_bf16():
    w = W.custom_workload(V=2000, d=64, d_s=32, r=16, D=6, M=12, k=3, N=40, batch=1,
                          wdtype="bf16", seed=7, logits="zipf", zipf=(1.1, 1.1))
    w = dataclasses.replace(w, W2=np.zeros_like(w.W2), temperature=np.array([0.5], np.float32))
    assert_same_tree(oracle.build_tree(w), factorised_tree(w, w.N), w.N, exact_scores=False)


# ------------------------------------------------------- k = 1: greedy chain

def test_k1_is_greedy_chain_torch():
    w = tiny(M=10, k=1, D=6, N=12, V=256, seed=31, d=32, d_s=16, r=8)
    o = oracle.build_tree(w)
    sc = TorchScorer(w)
    s, total, toks = sc.s_root, 0.0, []
    for j in range(1, w.D + 1):
        C, L = sc.logits(s, j)
        best = int(np.lexsort((C.numpy(), -L.numpy()))[0])
        toks.append(int(C[best]))
        total += float(torch.log_softmax(L, 0)[best])
        s = sc.step(s, C[best])
    assert o["n_nodes"] == w.D + 1
    np.testing.assert_array_equal(o["tokens"][1:w.D + 1], toks)
    np.testing.assert_array_equal(o["parents"][:w.D + 1], np.arange(-1, w.D))
    assert abs(float(o["scores"][w.D]) - total) < 1e-5


# ------------------------------------------- scores against float64 torch

@pytest.mark.parametrize("variant", ["tiny-config", "bf16-bias-state0-T"])
def test_scores_match_torch_rescoring(variant):
    if variant == "tiny-config":
        w = W.make_workload(0)
    else:
        w = W.custom_workload(V=3000, d=96, d_s=48, r=24, D=7, M=20, k=4, N=48, batch=1,
                              wdtype="bf16", seed=41, logits="zipf", zipf=(1.0, 1.0),
                              biases=True, state0_std=0.5, temperature=0.7)
    o = oracle.build_tree(w)
    sc = TorchScorer(w)
    # candidate sets
    np.testing.assert_array_equal(o["topm"], sc.cand.numpy())
    paths = {0: ()}
    for i in range(1, o["n_nodes"]):
        paths[i] = paths[int(o["parents"][i])] + (int(o["tokens"][i]),)
        total, _, in_tree = sc.path(paths[i])
        assert in_tree, f"node {i} is not among its parent's top-k children"
        assert abs(total - float(o["scores"][i])) < 1e-5, (i, total, o["scores"][i])
        # the path score the oracle reports for the same path agrees too
        s2, it = oracle.score_path(w, paths[i])
        assert it == 1 and s2 == o["scores"][i]


def test_lp_normalised_over_m_candidates():
    w = W.make_workload(0)
    for path in [(), tuple(oracle.build_tree(w)["tokens"][1:2])]:
        _, _, all_lp, cand = oracle.children(w, list(path))
        assert abs(np.exp(all_lp.astype(np.float64)).sum() - 1.0) < 1e-6
        sc = TorchScorer(w)
        s = sc.s_root if not path else sc.step(sc.s_root, path[0])
        C, L = sc.logits(s, len(path) + 1)
        np.testing.assert_array_equal(cand, C.numpy())
        np.testing.assert_allclose(all_lp, torch.log_softmax(L, 0).numpy(), atol=2e-6)


# ----------------------------------------------------------- invariances

def test_temperature_half_equals_doubled_logits_and_w2():
    w = W.make_workload(0)
    a = oracle.build_tree(dataclasses.replace(w, temperature=np.array([0.5], np.float32)))
    b = oracle.build_tree(dataclasses.replace(w, base_logits=w.base_logits * 2,
                                              W2=w.W2 * 2))
    for key in ("tokens", "parents", "depths", "scores", "mask"):
        np.testing.assert_array_equal(a[key], b[key])


def test_temperature_zero_reads_as_one():
    w = W.make_workload(0)
    a = oracle.build_tree(dataclasses.replace(w, temperature=np.array([0.0], np.float32)))
    b = oracle.build_tree(w)
    for key in ("tokens", "parents", "scores"):
        np.testing.assert_array_equal(a[key], b[key])


def test_depth_shift_leaves_tree_unchanged():
    w = W.make_workload(0)
    base = w.base_logits.copy()
    base[0, 2] += np.float32(3.0)
    a, b = oracle.build_tree(w), oracle.build_tree(dataclasses.replace(w, base_logits=base))
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    np.testing.assert_array_equal(a["parents"], b["parents"])
    np.testing.assert_allclose(a["scores"], b["scores"], atol=1e-5)


# ------------------------------------------------------- structural checks

def check_structure(w, o, b=0):
    n = o["n_nodes"]
    assert o["tokens"][0] == w.anchor[b] and o["parents"][0] == -1 and o["depths"][0] == 0
    assert o["scores"][0] == 0
    for i in range(1, n):
        p = o["parents"][i]
        assert 0 <= p < i
        assert o["depths"][i] == o["depths"][p] + 1 <= w.D
        assert o["tokens"][i] in set(o["topm"][o["depths"][i] - 1].tolist())
        assert o["scores"][i] <= o["scores"][i - 1]
        assert o["scores"][i] <= o["scores"][p]
    kids = {}
    for i in range(1, n):
        kids.setdefault(int(o["parents"][i]), []).append(i)
    for p, ch in kids.items():
        assert len(ch) <= w.k
    assert (o["tokens"][n:] == -1).all()
    np.testing.assert_array_equal(o["mask"], ancestor_mask(o["parents"], n, w.N))


def test_structure_tiny_and_bf16():
    check_structure(W.make_workload(0), oracle.build_tree(W.make_workload(0)))
    w = W.custom_workload(V=5000, d=64, d_s=32, r=16, D=15, M=32, k=8, N=64, batch=2,
                          wdtype="bf16", seed=9, logits="zipf", zipf=(0.8, 1.6))
    for b, o in enumerate(oracle.build_trees(w, threads=2)):
        assert o["status"] == 0
        check_structure(w, o, b)


# ------------------------------------------------------------ edge cases

def test_edge_cases():
    w = tiny()
    # N = 0: only the root
    o = oracle.build_tree(dataclasses.replace(w, N=0))
    assert o["n_nodes"] == 1 and o["tokens"][0] == w.anchor[0]
    # D = 1 with N beyond the k depth-1 nodes: exactly k nodes
    o = oracle.build_tree(dataclasses.replace(w, D=1, N=10, base_logits=w.base_logits[:, :1],
                                              H=w.H[:, :1]))
    assert o["n_nodes"] == 1 + w.k
    # M = V
    ws = tiny(V=8, M=8, k=3, D=3, N=15)
    assert_same_tree(oracle.build_tree(ws), brute_force(ws, 15), 15)
    # non-finite inputs
    bad = w.base_logits.copy()
    bad[0, 1, 5] = np.nan
    assert oracle.build_tree(dataclasses.replace(w, base_logits=bad))["status"] == oracle.ENONFINITE
    bad[0, 1, 5] = np.inf
    assert oracle.build_tree(dataclasses.replace(w, base_logits=bad))["status"] == oracle.ENONFINITE
    # -inf is a masked token, allowed
    bad[0, 1, 5] = -np.inf
    assert oracle.build_tree(dataclasses.replace(w, base_logits=bad))["status"] == 0
    # invalid arguments
    assert oracle.build_tree(dataclasses.replace(w, k=w.M + 1))["status"] == oracle.EINVAL
    assert oracle.build_tree(dataclasses.replace(
        w, temperature=np.array([-1.0], np.float32)))["status"] == oracle.EINVAL


def test_exact_ties_follow_push_order():
    """Flat base logits and W2 = 0: every candidate of a depth has the same lp, so
    all nodes of a depth tie exactly. The order must then be push order (parent
    position, child rank), which the sort-based brute force encodes."""
    w = tiny(M=3, k=3, D=3, N=30, V=16)
    w = dataclasses.replace(w, base_logits=np.zeros_like(w.base_logits), W2=np.zeros_like(w.W2))
    o = oracle.build_tree(w)
    assert_same_tree(o, brute_force(w, w.N), w.N)
    # breadth-first by construction: depth-1 nodes are ids 0,1,2 of depth 1 etc.
    np.testing.assert_array_equal(o["depths"][:13], [0] + [1] * 3 + [2] * 9)
    np.testing.assert_array_equal(o["tokens"][1:4], [0, 1, 2])
    np.testing.assert_array_equal(o["parents"][4:13], [1, 1, 1, 2, 2, 2, 3, 3, 3])


def test_expansion_count():
    """Every popped node is expanded except depth-D nodes and the N-th pop."""
    for w in (W.make_workload(0), tiny(M=5, k=2, D=3, N=9)):
        o = oracle.build_tree(w)
        n = o["n_nodes"]
        want = 1 + sum(1 for i in range(1, n) if o["depths"][i] < w.D and i < w.N)
        assert o["n_expanded"] == want
