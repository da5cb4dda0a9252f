"""CUDA path against the CPU oracle, through the C ABI (needs a GB300).

Every request of every configuration is compared with the oracle, tree by
tree: the tiny configuration, small custom shapes, the Qwen3-shaped batch-1
configurations, all 32 requests of the Qwen3-8B batch-32 configuration (the
benchmark workload, in its launch configuration) and all 128 requests of the
stress configuration at both temperatures, plus 32 requests of its separate
T = 0 pass. The oracle runs on every host core. Near ties (competing keys
within 1e-4, where the two builds may order differently) are counted and
printed in pytest's terminal summary.
"""
from __future__ import annotations

import dataclasses
import functools

import numpy as np
import pytest
import torch

import os

import dt_workloads as W
import oracle
from _parity import check_structure, parity_summary
from _report import record

pytestmark = pytest.mark.gpu

dt = pytest.importorskip("conditional_draft_tree_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conditional_draft_tree_gb300 import build
    build.build()
    oracle.build()


@functools.lru_cache(maxsize=4)
def workload(cfg):
    return W.make_workload(cfg)


def run_gpu(wl, spec=0, builder=None, temperature=None):
    tb = builder or dt.TreeBuilder.from_numpy(wl, spec_width=spec)
    inp = tb.inputs_to_device(wl)
    if temperature is not None:
        inp["temperature"] = torch.as_tensor(temperature, dtype=torch.float32, device="cuda")
    out = tb.run(**inp)
    torch.cuda.synchronize()
    return {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items()}


def oracle_trees(wl, reqs, threads=None):
    threads = threads or os.cpu_count() or 8
    return dict(zip(reqs, oracle.build_trees(wl, reqs, threads=threads)))


def check_against_oracle(wl, g, reqs, max_near_ties=None, name=None):
    """Every tree in `reqs` within the bar (exact, or a near tie); the counts
    are recorded for the session summary. Returns ['exact' | 'near-tie']."""
    refs = oracle_trees(wl, reqs)
    summ = parity_summary(wl, g, refs)
    record(name or wl.name, summ)
    if max_near_ties is not None:
        assert summ["near_tie"] <= max_near_ties, summ
    return ["exact"] * summ["exact"] + ["near-tie"] * summ["near_tie"]


def topm_reference(row, M):
    # exact tie handling: take every element >= the M-th value, then lexsort
    vm = np.partition(row, row.size - M)[row.size - M]
    cand = np.nonzero(row >= vm)[0]
    order = np.lexsort((cand, -row[cand].astype(np.float64)))
    return cand[order][:M]


# --------------------------------------------------------------- tiny/custom

def test_tiny_config_exact():
    wl = workload(0)
    g = run_gpu(wl)
    assert check_against_oracle(wl, g, [0]) == ["exact"]


SHAPES = {
    "ragged-V-f32": dict(V=1001, d=32, d_s=16, r=16, D=5, M=12, k=3, N=40, batch=3, wdtype="f32",
                         seed=1, logits="spiked", e_std=0.3),
    "bf16-bias-state0-T": dict(V=3000, d=64, d_s=32, r=24, D=7, M=20, k=4, N=48, batch=4,
                               wdtype="bf16", seed=2, logits="zipf", zipf=(0.8, 1.6),
                               biases=True, state0_std=0.5, temperature=[0.5, 1.0, 0.0, 2.0]),
    "k-equals-M": dict(V=500, d=16, d_s=8, r=8, D=4, M=5, k=5, N=60, batch=2, wdtype="f32",
                       seed=3, logits="spiked", e_std=0.5),
    "k1-chain": dict(V=700, d=16, d_s=16, r=8, D=9, M=7, k=1, N=20, batch=2, wdtype="f32",
                     seed=4, logits="spiked", e_std=0.5),
    "M1": dict(V=300, d=16, d_s=8, r=8, D=6, M=1, k=1, N=4, batch=1, wdtype="f32", seed=5,
               logits="spiked", e_std=0.5),
    "D1": dict(V=900, d=16, d_s=8, r=8, D=1, M=32, k=8, N=30, batch=2, wdtype="f32", seed=6,
               logits="spiked", e_std=0.5),
    "N0": dict(V=900, d=16, d_s=8, r=8, D=3, M=8, k=2, N=0, batch=2, wdtype="f32", seed=7,
               logits="spiked", e_std=0.5),
    "N1": dict(V=900, d=16, d_s=8, r=8, D=3, M=8, k=2, N=1, batch=2, wdtype="f32", seed=8,
               logits="spiked", e_std=0.5),
    "M256-k32": dict(V=5000, d=32, d_s=24, r=16, D=4, M=256, k=32, N=200, batch=2,
                     wdtype="bf16", seed=9, logits="zipf", zipf=(1.0, 1.4)),
    "wide-M100": dict(V=20000, d=40, d_s=40, r=40, D=15, M=100, k=10, N=150, batch=5,
                      wdtype="bf16", seed=10, logits="zipf", zipf=(0.8, 1.6)),
    "big-ds": dict(V=2048, d=64, d_s=1280, r=64, D=4, M=16, k=4, N=24, batch=2, wdtype="bf16",
                   seed=11, logits="zipf", zipf=(1.0, 1.2)),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("spec", [1, 5])
def test_custom_shapes(name, spec):
    wl = W.custom_workload(name=name, **SHAPES[name])
    g = run_gpu(wl, spec=spec)
    check_against_oracle(wl, g, list(range(wl.batch)), max_near_ties=1,
                         name=f"{name} (spec width {spec})")


def test_flat_logits_exact_ties():
    """All candidates tie: the order must follow push order on the GPU too."""
    wl = W.custom_workload(V=64, d=16, d_s=8, r=8, D=3, M=3, k=3, N=30, batch=1, wdtype="f32",
                           seed=12, logits="spiked", e_std=0.5)
    wl = dataclasses.replace(wl, base_logits=np.zeros_like(wl.base_logits),
                             W2=np.zeros_like(wl.W2))
    for spec in (1, 4, 16):
        g = run_gpu(wl, spec=spec)
        assert check_against_oracle(wl, g, [0]) == ["exact"]


def test_status_codes():
    wl = W.custom_workload(V=400, d=16, d_s=8, r=8, D=3, M=8, k=2, N=10, batch=4, wdtype="f32",
                           seed=13, logits="spiked", e_std=0.5,
                           temperature=[1.0, -1.0, 1.0, 1.0])
    base = wl.base_logits.copy()
    base[2, 1, 17] = np.nan
    base[3, 0, 5] = np.inf
    wl = dataclasses.replace(wl, base_logits=base)
    g = run_gpu(wl)
    assert list(g["status"]) == [dt.OK, dt.ERR_BAD_TEMPERATURE, dt.ERR_NONFINITE,
                                 dt.ERR_NONFINITE]
    for b in (1, 2, 3):
        assert (g["tokens"][b] == -1).all() and not g["mask"][b].any()
    check_against_oracle(wl, g, [0])


def test_neg_inf_logits_are_masked_tokens():
    wl = W.custom_workload(V=400, d=16, d_s=8, r=8, D=3, M=8, k=2, N=10, batch=1, wdtype="f32",
                           seed=14, logits="spiked", e_std=0.5)
    base = wl.base_logits.copy()
    base[0, :, :395] = -np.inf        # only 5 finite tokens per depth, M = 8
    wl = dataclasses.replace(wl, base_logits=base)
    g = run_gpu(wl)
    check_against_oracle(wl, g, [0])


# ------------------------------------------------------------ Qwen3 shapes

def test_config1_qwen3_4b_b1():
    wl = workload(1)
    g = run_gpu(wl)
    check_against_oracle(wl, g, [0], max_near_ties=1)


def test_config2_qwen3_8b_b1():
    wl = workload(2)
    g = run_gpu(wl)
    check_against_oracle(wl, g, [0], max_near_ties=1)


def test_config3_qwen3_8b_b32_every_request():
    wl = workload(3)
    g = run_gpu(wl)
    for b in range(wl.batch):
        assert g["status"][b] == 0
        check_structure(wl, b, g)
        for j in range(wl.D):
            np.testing.assert_array_equal(g["topm"][b, j],
                                          topm_reference(wl.base_logits[b, j], wl.M))
    check_against_oracle(wl, g, list(range(wl.batch)), max_near_ties=3,
                         name="qwen3-8b-b32 (every request)")


def test_config3_spec_width_invariance_and_determinism():
    wl = workload(3)
    tb1 = dt.TreeBuilder.from_numpy(wl, spec_width=1)
    ref = run_gpu(wl, builder=tb1)
    for spec in (2, 8, 16):
        g = run_gpu(wl, spec=spec)
        for key in ("tokens", "parents", "depths", "scores", "mask", "topm", "status"):
            np.testing.assert_array_equal(g[key], ref[key], err_msg=f"{key} spec={spec}")
    again = run_gpu(wl, builder=tb1)
    for key in ("tokens", "parents", "depths", "scores", "mask"):
        np.testing.assert_array_equal(again[key], ref[key])


def test_config4_stress_every_request():
    wl = workload(4)
    g = run_gpu(wl)
    for b in range(wl.batch):
        assert g["status"][b] == 0
        check_structure(wl, b, g)
    for b in (0, 63, 127):
        for j in range(wl.D):
            np.testing.assert_array_equal(g["topm"][b, j],
                                          topm_reference(wl.base_logits[b, j], wl.M))
    # T cycles 0.5 / 1.0 over the requests
    check_against_oracle(wl, g, list(range(wl.batch)), max_near_ties=12,
                         name="stress-b128 (every request, T 0.5 / 1.0)")
    # the separate T = 0 pass: read as T = 1 (greedy ordering)
    g0 = run_gpu(wl, temperature=np.zeros(wl.batch, np.float32))
    wl0 = dataclasses.replace(wl, temperature=np.zeros(wl.batch, np.float32))
    for b in range(wl.batch):
        assert g0["status"][b] == 0
        check_structure(wl0, b, g0)
    check_against_oracle(wl0, g0, list(range(0, wl.batch, 4)), max_near_ties=3,
                         name="stress-b128 T = 0 pass (32 requests)")


def test_host_io_variant_matches_device():
    wl = W.custom_workload(V=3000, d=64, d_s=32, r=24, D=7, M=20, k=4, N=48, batch=3,
                           wdtype="bf16", seed=15, logits="zipf", zipf=(0.8, 1.6))
    tb = dt.TreeBuilder.from_numpy(wl)
    dev = run_gpu(wl, builder=tb)
    host_ws = torch.empty(dt.host_workspace_bytes(tb.dims, tb.opt), dtype=torch.uint8,
                          device="cuda")
    pin = lambda a, t: torch.from_numpy(np.ascontiguousarray(a, dtype=t)).pin_memory()
    base = pin(wl.base_logits, np.float32)
    # page-locked logits are mapped: read in place by default, copied with the flag
    assert dt.mapped_host_pointer(base) is not None
    paged = torch.from_numpy(np.ascontiguousarray(wl.base_logits, dtype=np.float32))
    for logits, flags in ((base, 0), (base, dt.OPT_STAGE_HOST_LOGITS), (paged, 0)):
        out = dt.alloc_outputs(tb.dims, "cpu", pin=True)
        dt.build_trees_host(tb.dims, tb.w, tb.prepared, logits,
                            pin(wl.H, np.float32), pin(wl.state0, np.float32),
                            pin(wl.anchor, np.int32), pin(wl.temperature, np.float32), host_ws,
                            out, dt.options(flags=flags))
        torch.cuda.synchronize()
        for key in ("tokens", "parents", "depths", "scores", "mask", "topm", "status"):
            np.testing.assert_array_equal(out[key].numpy(), dev[key])


def test_mapped_host_pointer():
    pinned = torch.zeros(1 << 20, dtype=torch.float32).pin_memory()
    p = dt.mapped_host_pointer(pinned)
    assert p is not None
    lib = dt.lib()
    # an extent past the registration, pageable memory and device memory are not mapped
    assert lib.dt_mapped_host_pointer(pinned.data_ptr(), 1 << 40) is None
    assert dt.mapped_host_pointer(torch.zeros(1 << 20, dtype=torch.float32)) is None
    assert dt.mapped_host_pointer(torch.zeros(1 << 20, dtype=torch.float32, device="cuda")) is None
    # a sub-range of the registration is mapped at the matching offset
    assert lib.dt_mapped_host_pointer(pinned.data_ptr() + 4096, 4096) == p + 4096


# --------------------------------------------- more requests than one wave

def test_batch_beyond_one_wave():
    """300 requests: the search runs as two waves of launches (at most one block
    per SM and request per wave); requests of both waves against the oracle."""
    wl = W.custom_workload(V=3000, d=64, d_s=32, r=24, D=7, M=20, k=4, N=48, batch=300,
                           wdtype="bf16", seed=31, logits="zipf", zipf=(0.8, 1.6))
    tb = dt.TreeBuilder.from_numpy(wl)
    assert dt.kernel_launches(tb.dims, tb.w.wdtype, tb.opt) >= 5   # >= 2 search waves
    g = run_gpu(wl, builder=tb)
    for b in range(wl.batch):
        assert g["status"][b] == 0
        check_structure(wl, b, g)
    check_against_oracle(wl, g, list(range(wl.batch)), max_near_ties=2,
                         name="two search waves (300 requests)")
