"""Comparison of a GPU-built tree with the oracle's tree.

The bar (fixed by the build's contract):
* top-M candidate ids: bit-exact;
* tree topology (token paths, parent links): bit-exact, except where the two
  builds faced competing keys that differ by less than 1e-4 ("near tie") --
  such trees are counted and reported;
* node scores: within 1e-5 absolute.

Trees are compared as sets of token paths, so a swap of two near-equal pops
(which renumbers nodes) is recognised as such. Every node present in only one
of the two trees must descend from a "divergence root" u whose parent is common
and which is excused by the oracle itself: either u sits at its parent's top-k
boundary (its lp is within 1e-4 of the oracle's k-th best lp) or at the budget
boundary (its oracle path score is within 1e-4 of the smallest score kept).
"""
from __future__ import annotations

import numpy as np

import oracle

TOL_SCORE = 1e-5
TOL_TIE = 1e-4


def paths_of(tokens, parents):
    n = int((tokens >= 0).sum())
    paths = [()]
    for i in range(1, n):
        paths.append(paths[int(parents[i])] + (int(tokens[i]),))
    return paths


def check_structure(wl, b, g):
    """Validity of one GPU tree (any size; no oracle needed)."""
    tok, par, dep, sc = g["tokens"][b], g["parents"][b], g["depths"][b], g["scores"][b]
    n = int((tok >= 0).sum())
    assert (tok[:n] >= 0).all() and (tok[n:] == -1).all() and (par[n:] == -1).all()
    assert tok[0] == wl.anchor[b] and par[0] == -1 and dep[0] == 0 and sc[0] == 0
    assert np.isneginf(sc[n:]).all()
    topm = g["topm"][b]
    for i in range(1, n):
        p = int(par[i])
        assert 0 <= p < i
        assert dep[i] == dep[p] + 1 <= wl.D
        assert tok[i] in topm[dep[i] - 1]
        assert sc[i] <= sc[i - 1] and sc[i] <= sc[p]
    kids = np.bincount(par[1:n], minlength=n)
    assert kids.max(initial=0) <= wl.k
    if g.get("mask") is not None:
        m = g["mask"][b]
        want = np.zeros_like(m)
        for i in range(n):
            a = i
            while a >= 0:
                want[i, a] = 1
                a = int(par[a])
        np.testing.assert_array_equal(m, want)
    return n


def compare_tree(wl, b, g, ref):
    """'exact' or 'near-tie'; raises AssertionError otherwise. g: dict of batch
    arrays from the GPU; ref: oracle.build_tree(wl, b) output."""
    return compare_tree_err(wl, b, g, ref)[0]


def compare_tree_err(wl, b, g, ref):
    """compare_tree, plus the largest score difference over the nodes the two
    trees share (0 for a request that reports an error status)."""
    assert int(g["status"][b]) == ref["status"], (g["status"][b], ref["status"])
    if ref["status"] != 0:
        return "exact", 0.0
    np.testing.assert_array_equal(g["topm"][b], ref["topm"])
    check_structure(wl, b, g)
    gt, gp, gd, gs = (g[k][b] for k in ("tokens", "parents", "depths", "scores"))
    if (np.array_equal(gt, ref["tokens"]) and np.array_equal(gp, ref["parents"])
            and np.array_equal(gd, ref["depths"])):
        fin = np.isfinite(ref["scores"])
        assert np.array_equal(np.isfinite(gs), fin)
        err = np.abs(gs[fin].astype(np.float64) - ref["scores"][fin])
        assert err.max(initial=0) <= TOL_SCORE, f"score error {err.max()}"
        return "exact", float(err.max(initial=0))
    gpaths, opaths = paths_of(gt, gp), paths_of(ref["tokens"], ref["parents"])
    gmap = {p: float(gs[i]) for i, p in enumerate(gpaths)}
    omap = {p: float(ref["scores"][i]) for i, p in enumerate(opaths)}
    common_err = 0.0
    for p in gmap.keys() & omap.keys():
        assert abs(gmap[p] - omap[p]) <= TOL_SCORE, (p, gmap[p], omap[p])
        if np.isfinite(gmap[p]) and np.isfinite(omap[p]):
            common_err = max(common_err, abs(gmap[p] - omap[p]))
    boundary = min(min(gmap.values()), min(omap.values()))
    only = (gmap.keys() - omap.keys()) | (omap.keys() - gmap.keys())
    roots = {p for p in only if p[:-1] not in only}
    for u in roots:
        parent = u[:-1]
        toks, lps, all_lp, cand = oracle.children(wl, list(parent), b)
        lp_u = float(all_lp[list(cand).index(u[-1])])
        at_topk = abs(lp_u - float(lps[-1])) < TOL_TIE
        sc_u, _ = oracle.score_path(wl, list(u), b)
        at_budget = abs(sc_u - boundary) < TOL_TIE
        assert at_topk or at_budget, f"divergence at {u} is not a near tie"
    return "near-tie", common_err


def parity_summary(wl, g, refs):
    """Counts over the requests in `refs` ({b: oracle tree}): compared, exact,
    near-tie, the largest score error; raises on any tree outside the bar."""
    out = dict(compared=0, exact=0, near_tie=0, max_score_err=0.0)
    for b, ref in refs.items():
        kind, err = compare_tree_err(wl, b, g, ref)
        out["compared"] += 1
        out["exact" if kind == "exact" else "near_tie"] += 1
        out["max_score_err"] = max(out["max_score_err"], err)
    return out
