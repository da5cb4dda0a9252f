"""Failure detection on the GPU without a GPU fault (needs a GB300).

The search kernel's waits are all bounded. The test hook
DT_OPT_TEST_BARRIER_TIMEOUT makes the last block of the launch skip its first
grid-barrier arrival and limits every wait to 2 ms, so the other blocks' waits
run out: the launch must end by itself, report DT_ERR_TIMEOUT for every
request with empty rows, and leave the context usable for the next call.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import dt_workloads as W
import oracle
from _parity import compare_tree

pytestmark = pytest.mark.gpu

dt = pytest.importorskip("conditional_draft_tree_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conditional_draft_tree_gb300 import build
    build.build()
    oracle.build()


def _run(tb, wl):
    out = tb.run(**tb.inputs_to_device(wl))
    torch.cuda.synchronize()
    return {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items()}


@pytest.mark.parametrize("wdtype", ["f32", "bf16"])
def test_barrier_timeout_is_reported_and_context_survives(wdtype):
    wl = W.custom_workload(V=3000, d=64, d_s=32, r=24, D=7, M=20, k=4, N=48, batch=4,
                           wdtype=wdtype, seed=21, logits="zipf", zipf=(0.8, 1.6))
    bad = _run(dt.TreeBuilder.from_numpy(wl, flags=dt.OPT_TEST_BARRIER_TIMEOUT), wl)
    assert (bad["status"] == dt.ERR_TIMEOUT).all()
    assert (bad["tokens"] == -1).all() and (bad["parents"] == -1).all()
    assert np.isneginf(bad["scores"]).all() and not bad["mask"].any()
    # the same process and context build correct trees right after
    good = _run(dt.TreeBuilder.from_numpy(wl), wl)
    refs = oracle.build_trees(wl, list(range(wl.batch)), threads=4)
    for b in range(wl.batch):
        assert compare_tree(wl, b, good, refs[b]) in ("exact", "near-tie")


def test_kernel_launch_count():
    wl = W.custom_workload(V=3000, d=64, d_s=32, r=24, D=7, M=20, k=4, N=48, batch=4,
                           wdtype="bf16", seed=21, logits="zipf", zipf=(0.8, 1.6))
    tb = dt.TreeBuilder.from_numpy(wl)
    n = dt.kernel_launches(tb.dims, tb.w.wdtype, tb.opt)
    # top-M, projection (+ its split-K sum), one search wave for 4 requests
    assert n in (3, 4)
