"""Marginal-score trees (DT_OPT_MARGINAL) against the oracle (needs a GB300).

The marginal builder is the conditional builder with the correction removed
("Riassunto Tecnico: DominoTree", Risultati Sperimentali: the conditionality
ablation, a DDTree-style builder), so its reference is the oracle run with
W2 = 0; the oracle's W2 = 0 trees are themselves pinned against a separately
written factorised builder in the oracle tests. Two more checks come from the
GPU side: the conditional search kernel with W2 = 0 computes the same L values
(base + 0, divided by T), so its trees must equal the marginal kernel's bit for
bit; and the marginal mode reads no weight, GRU state or backbone state, so
those pointers are passed as NULL.
"""
from __future__ import annotations

import os

import dataclasses
import functools

import numpy as np
import pytest
import torch

import dt_workloads as W
import oracle
from _parity import check_structure, compare_tree

pytestmark = pytest.mark.gpu

dt = pytest.importorskip("conditional_draft_tree_gb300")

KEYS = ("tokens", "parents", "depths", "scores", "mask", "topm", "status")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conditional_draft_tree_gb300 import build
    build.build()
    oracle.build()


def zero_w2(wl):
    return dataclasses.replace(wl, W2=np.zeros_like(wl.W2))


@functools.lru_cache(maxsize=2)
def workload_w2zero(cfg):
    return zero_w2(W.make_workload(cfg))


def to_dev(a, t):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=t)).cuda()


def run_marginal(wl, temperature=None, mask=True):
    mb = dt.MarginalTreeBuilder.from_workload(wl)
    T = wl.temperature if temperature is None else temperature
    out = dt.alloc_outputs(mb.dims, "cuda", mask=mask)
    mb.run(to_dev(wl.base_logits, np.float32), to_dev(wl.anchor, np.int32),
           to_dev(T, np.float32), out=out)
    torch.cuda.synchronize()
    return {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items()}


def run_conditional(wl, spec=0):
    tb = dt.TreeBuilder.from_numpy(wl, spec_width=spec)
    out = tb.run(**tb.inputs_to_device(wl))
    torch.cuda.synchronize()
    return {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items()}


def check_against_oracle(wl, g, reqs, max_near_ties=None):
    refs = oracle.build_trees(wl, reqs, threads=os.cpu_count() or 8)
    kinds = [compare_tree(wl, b, g, ref) for b, ref in zip(reqs, refs)]
    if max_near_ties is not None:
        assert kinds.count("near-tie") <= max_near_ties
    return kinds


SHAPES = {
    "ragged-V": dict(V=1001, d=32, d_s=16, r=16, D=5, M=12, k=3, N=40, batch=3, wdtype="f32",
                     seed=41, logits="spiked", e_std=0.3),
    "zipf-T": dict(V=3000, d=64, d_s=32, r=24, D=7, M=20, k=4, N=48, batch=4, wdtype="bf16",
                   seed=42, logits="zipf", zipf=(0.8, 1.6), temperature=[0.5, 1.0, 0.0, 2.0]),
    "k-equals-M": dict(V=500, d=16, d_s=8, r=8, D=4, M=5, k=5, N=60, batch=2, wdtype="f32",
                       seed=43, logits="spiked", e_std=0.5),
    "k1-chain": dict(V=700, d=16, d_s=16, r=8, D=9, M=7, k=1, N=20, batch=2, wdtype="f32",
                     seed=44, logits="spiked", e_std=0.5),
    "M1": dict(V=300, d=16, d_s=8, r=8, D=6, M=1, k=1, N=4, batch=1, wdtype="f32", seed=45,
               logits="spiked", e_std=0.5),
    "D1": dict(V=900, d=16, d_s=8, r=8, D=1, M=32, k=8, N=30, batch=2, wdtype="f32", seed=46,
               logits="spiked", e_std=0.5),
    "N0": dict(V=900, d=16, d_s=8, r=8, D=3, M=8, k=2, N=0, batch=2, wdtype="f32", seed=47,
               logits="spiked", e_std=0.5),
    "N1": dict(V=900, d=16, d_s=8, r=8, D=3, M=8, k=2, N=1, batch=2, wdtype="f32", seed=48,
               logits="spiked", e_std=0.5),
    "M64-depth-loop": dict(V=8000, d=16, d_s=8, r=8, D=20, M=64, k=6, N=300, batch=3,
                           wdtype="f32", seed=49, logits="zipf", zipf=(0.9, 1.5)),
    "M100": dict(V=20000, d=16, d_s=8, r=8, D=15, M=100, k=10, N=150, batch=5, wdtype="bf16",
                 seed=50, logits="zipf", zipf=(0.8, 1.6)),
    # every limit of the build at once: D 64, M 256, k 32, N 1024
    "max-sizes": dict(V=4096, d=16, d_s=8, r=8, D=64, M=256, k=32, N=1024, batch=2,
                      wdtype="f32", seed=51, logits="zipf", zipf=(0.7, 1.3)),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_custom_shapes(name):
    wl = zero_w2(W.custom_workload(name=name, **SHAPES[name]))
    g = run_marginal(wl)
    check_against_oracle(wl, g, list(range(wl.batch)), max_near_ties=1)


@pytest.mark.parametrize("name", ["ragged-V", "zipf-T", "k1-chain", "M100", "D1"])
def test_equals_conditional_kernel_with_zero_w2(name):
    """Same L values on both GPU paths, so the same trees bit for bit."""
    wl = zero_w2(W.custom_workload(name=name, **SHAPES[name]))
    g = run_marginal(wl)
    for spec in (1, 8):
        c = run_conditional(wl, spec)
        for key in KEYS:
            np.testing.assert_array_equal(g[key], c[key], err_msg=f"{key} spec={spec}")


def test_tiny_config():
    wl = workload_w2zero(0)
    g = run_marginal(wl)
    assert check_against_oracle(wl, g, [0]) == ["exact"]


def test_flat_logits_exact_ties():
    """Every candidate ties: the pops follow push order."""
    wl = W.custom_workload(V=64, d=16, d_s=8, r=8, D=3, M=3, k=3, N=30, batch=1, wdtype="f32",
                           seed=52, logits="spiked", e_std=0.5)
    wl = dataclasses.replace(zero_w2(wl), base_logits=np.zeros_like(wl.base_logits))
    g = run_marginal(wl)
    assert check_against_oracle(wl, g, [0]) == ["exact"]


def test_status_codes_and_masked_tokens():
    wl = zero_w2(W.custom_workload(V=400, d=16, d_s=8, r=8, D=3, M=8, k=2, N=10, batch=5,
                                   wdtype="f32", seed=53, logits="spiked", e_std=0.5,
                                   temperature=[1.0, -1.0, 1.0, 1.0, 0.0]))
    base = wl.base_logits.copy()
    base[2, 1, 17] = np.nan
    base[3, 0, 5] = np.inf
    base[0, :, :395] = -np.inf       # request 0: 5 finite tokens per depth, M = 8
    wl = dataclasses.replace(wl, base_logits=base)
    g = run_marginal(wl)
    assert list(g["status"]) == [dt.OK, dt.ERR_BAD_TEMPERATURE, dt.ERR_NONFINITE,
                                 dt.ERR_NONFINITE, dt.OK]
    for b in (1, 2, 3):
        assert (g["tokens"][b] == -1).all() and not g["mask"][b].any()
        assert (g["parents"][b] == -1).all() and np.isneginf(g["scores"][b]).all()
    check_against_oracle(wl, g, [0, 4])     # masked tokens; T = 0 read as T = 1


def test_without_mask_output():
    wl = zero_w2(W.custom_workload(name="M100", **SHAPES["M100"]))
    full, nomask = run_marginal(wl), run_marginal(wl, mask=False)
    assert nomask["mask"] is None
    for key in ("tokens", "parents", "depths", "scores", "topm", "status"):
        np.testing.assert_array_equal(nomask[key], full[key])


def test_kernel_launches():
    wl = W.custom_workload(name="M100", **SHAPES["M100"])
    mb = dt.MarginalTreeBuilder.from_workload(wl)
    assert dt.kernel_launches(mb.dims, dt.F32, mb.opt) == 2


def test_host_io_variant_matches_device():
    wl = zero_w2(W.custom_workload(name="zipf-T", **SHAPES["zipf-T"]))
    dev = run_marginal(wl)
    mb = dt.MarginalTreeBuilder.from_workload(wl)
    host_ws = torch.empty(dt.host_workspace_bytes(mb.dims, mb.opt), dtype=torch.uint8,
                          device="cuda")
    pin = lambda a, t: torch.from_numpy(np.ascontiguousarray(a, dtype=t)).pin_memory()
    out = dt.alloc_outputs(mb.dims, "cpu", pin=True)
    dt.build_trees_host(mb.dims, None, None, pin(wl.base_logits, np.float32), None, None,
                        pin(wl.anchor, np.int32), pin(wl.temperature, np.float32), host_ws,
                        out, mb.opt)
    torch.cuda.synchronize()
    for key in KEYS:
        np.testing.assert_array_equal(out[key].numpy(), dev[key])


# ------------------------------------------------------------ Qwen3 shapes

def test_config2_qwen3_8b_b1():
    wl = workload_w2zero(2)
    g = run_marginal(wl)
    check_against_oracle(wl, g, [0], max_near_ties=1)


def test_config3_qwen3_8b_b32():
    """Batch 32 at the benchmark's shapes: every request against the conditional
    kernel with W2 = 0 (bit for bit) and for validity; sampled ones against the
    oracle."""
    wl = workload_w2zero(3)
    g = run_marginal(wl)
    c = run_conditional(wl)
    for key in KEYS:
        np.testing.assert_array_equal(g[key], c[key], err_msg=key)
    for b in range(wl.batch):
        assert g["status"][b] == 0
        check_structure(wl, b, g)
    check_against_oracle(wl, g, list(range(wl.batch)), max_near_ties=2)
