"""CondAdaptive budget (dt_adaptive_budget) against the oracle (needs a GB300).

Each side cuts its own tree: the GPU the GPU-built tree, the oracle the
oracle-built one (the trees agree, scores within 1e-5). The kept counts must be
equal unless the oracle's decision at the cut was within 1e-4 relative (a near
tie the score rounding may flip); the cut GPU tree must be the first rows of the
uncut one with the later rows emptied.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import dt_workloads as W
import oracle

pytestmark = pytest.mark.gpu

dt = pytest.importorskip("conditional_draft_tree_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conditional_draft_tree_gb300 import build
    build.build()
    oracle.build()


def margin(scores, n, c_fixed, c_node):
    """Relative gap of the oracle's decision about row n + 1 (the first row cut)."""
    A, C = 1.0, c_fixed
    for i in range(1, n + 1):
        A += float(np.exp(np.float64(scores[i])))
        C += c_node
    if n + 1 >= len(scores) or not np.isfinite(scores[n + 1]):
        return np.inf
    e = float(np.exp(np.float64(scores[n + 1])))
    return abs(e * C - A * c_node) / (A * c_node)


@pytest.mark.parametrize("cfg,reqs", [(0, [0]), (3, list(range(32)))])
@pytest.mark.parametrize("c_node", [1 / 1024, 1 / 64, 1 / 8])
def test_counts_and_cut(cfg, reqs, c_node):
    wl = W.make_workload(cfg)
    tb = dt.TreeBuilder.from_numpy(wl)
    out = tb.run(**tb.inputs_to_device(wl))
    torch.cuda.synchronize()
    full = {k: v.cpu().numpy() for k, v in out.items() if v is not None}
    counts = dt.adaptive_budget(out, wl.N, 1.0, c_node)
    torch.cuda.synchronize()
    got = counts.cpu().numpy()
    cut = {k: v.cpu().numpy() for k, v in out.items() if v is not None}
    for b in range(wl.batch):
        n = int(got[b])
        assert 0 <= n <= wl.N
        for key in ("tokens", "parents", "depths", "scores"):
            np.testing.assert_array_equal(cut[key][b, :n + 1], full[key][b, :n + 1])
        assert (cut["tokens"][b, n + 1:] == -1).all() and np.isneginf(cut["scores"][b, n + 1:]).all()
        np.testing.assert_array_equal(cut["mask"][b, :n + 1], full["mask"][b, :n + 1])
        assert not cut["mask"][b, n + 1:].any()
    for b, t in zip(reqs, oracle.build_trees(wl, reqs, threads=os.cpu_count() or 8)):
        want = oracle.adaptive_count(t["scores"], t["tokens"], 1.0, c_node)
        if got[b] != want:
            assert margin(t["scores"], min(want, got[b]), 1.0, c_node) < 1e-4, (b, got[b], want)


def test_invalid_costs_rejected():
    wl = W.make_workload(0)
    out = dt.alloc_outputs(dt.dims_of(wl.V, wl.d, wl.d_s, wl.r, wl.D, wl.M, wl.k, wl.N, 1), "cuda")
    for cf, cn in ((0.0, 1.0), (1.0, 0.0), (1.0, float("inf")), (float("nan"), 1.0)):
        with pytest.raises(dt.DtError):
            dt.adaptive_budget(out, wl.N, cf, cn)
