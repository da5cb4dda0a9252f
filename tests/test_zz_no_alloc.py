"""The allocation-free top-M entry point (dt_select_topm_noalloc).

It is meant for callers that may not allocate device memory (a runtime whose
device memory is all pre-reserved for its own pool, a latency-critical loop
that cannot take cudaMalloc's implicit synchronisation, a plug-in inside a
framework that owns every allocation). Its scratch is a static device array
shared by every call, so these tests also check that a second call in a row,
which finds the first call's leftovers in that array, gives the same answer.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test. It passes alone and after the
other tests.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import dt_workloads as W
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conditional_draft_tree_gb300 import build
    build.build()
    import conditional_draft_tree_gb300 as dt
    return dt


def reference_topm(dt, wl):
    """top-M ids and status from the existing entry point, dt_build_trees."""
    tb = dt.TreeBuilder.from_numpy(wl)
    out = tb.run(**tb.inputs_to_device(wl))
    torch.cuda.synchronize()
    return out["topm"].cpu().numpy(), out["status"].cpu().numpy()


def oracle_topm(wl):
    """The oracle's top-M of every row (the pinned CPU selection)."""
    oracle.build()
    return np.stack([[oracle.topm(wl.base_logits[b, j], wl.M) for j in range(wl.D)]
                     for b in range(wl.batch)])


def noalloc_topm(dt, wl, calls=2):
    logits = torch.from_numpy(np.ascontiguousarray(wl.base_logits)).cuda()
    res = []
    for _ in range(calls):
        topm = torch.full((wl.batch, wl.D, wl.M), -7, dtype=torch.int32, device="cuda")
        status = torch.full((wl.batch,), -7, dtype=torch.int32, device="cuda")
        assert dt.select_topm_noalloc(logits, wl.M, topm, status) == dt.OK
        torch.cuda.synchronize()
        res.append((topm.cpu().numpy(), status.cpu().numpy()))
    return res


@pytest.mark.parametrize("shape", [
    dict(V=151936, d=16, d_s=8, r=8, D=15, M=64, k=8, N=16, batch=3, wdtype="bf16",
         logits="zipf", zipf=(0.8, 1.6), seed=31),
    dict(V=5001, d=16, d_s=8, r=8, D=7, M=256, k=4, N=8, batch=5, wdtype="f32",
         logits="spiked", seed=32),
])
def test_noalloc_matches_build_trees_twice(dt, shape):
    wl = W.custom_workload(**shape)
    ref_topm, ref_status = reference_topm(dt, wl)
    want = oracle_topm(wl)
    np.testing.assert_array_equal(ref_topm, want)
    for topm, status in noalloc_topm(dt, wl, calls=2):
        np.testing.assert_array_equal(topm, want)
        np.testing.assert_array_equal(status, ref_status)


def test_noalloc_segment_fallback_matches_oracle(dt):
    """A shape whose contiguous-range launch does not fit the static scratch
    (the row pieces' lists), so the call cuts the rows into fewer segments."""
    wl = W.custom_workload(V=4096, d=16, d_s=8, r=8, D=16, M=256, k=4, N=8, batch=128,
                           wdtype="f32", logits="zipf", zipf=(0.8, 1.6), seed=34)
    want = oracle_topm(wl)
    for topm, status in noalloc_topm(dt, wl, calls=2):
        assert (status == dt.OK).all()
        np.testing.assert_array_equal(topm, want)


def test_noalloc_allocates_no_device_memory(dt):
    """After a first call, further calls leave the device's free memory as it
    is (the inputs and outputs are allocated before the measurement)."""
    wl = W.custom_workload(V=151936, d=16, d_s=8, r=8, D=15, M=64, k=8, N=16, batch=4,
                           wdtype="bf16", logits="zipf", zipf=(0.8, 1.6), seed=35)
    logits = torch.from_numpy(np.ascontiguousarray(wl.base_logits)).cuda()
    topm = torch.empty((wl.batch, wl.D, wl.M), dtype=torch.int32, device="cuda")
    status = torch.empty((wl.batch,), dtype=torch.int32, device="cuda")
    assert dt.select_topm_noalloc(logits, wl.M, topm, status) == dt.OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        assert dt.select_topm_noalloc(logits, wl.M, topm, status) == dt.OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_flags_nonfinite_and_recovers(dt):
    wl = W.custom_workload(V=3000, d=16, d_s=8, r=8, D=4, M=16, k=4, N=8, batch=3, wdtype="f32",
                           logits="spiked", seed=33)
    bad = wl.base_logits.copy()
    bad[1, 2, 7] = np.nan
    (topm, status), = noalloc_topm(dt, dataclasses.replace(wl, base_logits=bad), calls=1)
    assert list(status) == [dt.OK, dt.ERR_NONFINITE, dt.OK]
    want = oracle_topm(wl)
    np.testing.assert_array_equal(topm[0], want[0])
    # the next call starts from clean tickets and flags
    (topm, status), = noalloc_topm(dt, wl, calls=1)
    assert list(status) == [dt.OK] * 3
    np.testing.assert_array_equal(topm, want)


def test_noalloc_rejects_shapes_beyond_the_static_scratch(dt):
    batch, D, V, M = 200, 64, 1024, 256         # 12800 rows x (4 M + 4) B ~ 13 MB > 8 MiB
    logits = torch.zeros((batch, D, V), dtype=torch.float32, device="cuda")
    topm = torch.empty((batch, D, M), dtype=torch.int32, device="cuda")
    status = torch.empty((batch,), dtype=torch.int32, device="cuda")
    assert dt.select_topm_noalloc(logits, M, topm, status) == dt.ERR_INVALID_ARG
