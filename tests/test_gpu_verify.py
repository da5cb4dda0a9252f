"""Verify-side consumption (dt_tree_positions, dt_tree_attention) against the
oracle (needs a GB300).

Positions are integers: bit-exact. Attention: bf16 inputs are exact in both,
the GPU accumulates in fp32 (head dimension up to 256 products, softmax sums
over at most P + n1 keys in chunks of 64) and the oracle in fp64; the outputs
are convex combinations of N(0, 1) values, so an absolute 2e-4 (with 2e-4
relative) leaves about an order of magnitude above the fp32 error. The kernel
keeps a per-row reference maximum that moves only when a chunk's maximum
exceeds it by more than 8 (then the accumulated output is rescaled);
`test_rescaled_accumulator` drives that path with keys whose norms grow or
shrink from chunk to chunk.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import dt_workloads as W
import oracle

pytestmark = pytest.mark.gpu

dt = pytest.importorskip("conditional_draft_tree_gb300")

ATOL = RTOL = 2e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conditional_draft_tree_gb300 import build
    build.build()
    oracle.build()


def gpu_trees(N, batch, seed):
    wl = W.custom_workload(V=400, d=16, d_s=16, r=8, D=6, M=6, k=3, N=N, batch=batch,
                           wdtype="f32", seed=seed, logits="spiked", e_std=0.5)
    tb = dt.TreeBuilder.from_numpy(wl)
    out = tb.run(**tb.inputs_to_device(wl))
    torch.cuda.synchronize()
    return out


def run_attention(q, k, v, mask, plen):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    out = dt.tree_attention(t(q), t(k), t(v), mask, torch.from_numpy(plen).cuda())
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check(q, k, v, mask_np, plen, got, pairs=None):
    f = W.bf16_bits_to_f32
    dh = q.shape[-1]
    B, H = q.shape[:2]
    group = H // k.shape[1]
    pairs = pairs or [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        ref = oracle.tree_attention(f(q[b:b + 1, h:h + 1]), f(k[b:b + 1, h // group:h // group + 1]),
                                    f(v[b:b + 1, h // group:h // group + 1]), mask_np[b:b + 1],
                                    plen[b:b + 1], dh ** -0.5)
        np.testing.assert_allclose(got[b, h], ref[0, 0], atol=ATOL, rtol=RTOL, err_msg=f"{b},{h}")


@pytest.mark.parametrize("N,batch", [(12, 3), (64, 2), (100, 2)])
def test_positions_bit_exact(N, batch):
    out = gpu_trees(N, batch, 91 + N)
    plen = np.array([7, 0, 300][:batch], np.int32)
    pos = dt.tree_positions(out["depths"], torch.from_numpy(plen).cuda())
    torch.cuda.synchronize()
    want = oracle.tree_positions(out["depths"].cpu().numpy(), plen)
    np.testing.assert_array_equal(pos.cpu().numpy(), want)


CASES = {
    "dh64-ragged-prefix": dict(N=12, batch=3, H=4, Hkv=2, P=5, dh=64),
    "dh128-two-row-tiles": dict(N=100, batch=2, H=4, Hkv=1, P=30, dh=128),
    "dh128-n65": dict(N=64, batch=2, H=8, Hkv=2, P=100, dh=128),
    "dh256": dict(N=20, batch=2, H=2, Hkv=1, P=40, dh=256),
    "no-prefix": dict(N=30, batch=2, H=2, Hkv=2, P=0, dh=64),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_attention_against_oracle(name):
    c = CASES[name]
    out = gpu_trees(c["N"], c["batch"], 101)
    n1 = c["N"] + 1
    q, k, v, plen = W.verify_inputs(c["batch"], c["H"], c["Hkv"], n1, c["P"], c["dh"], seed=102)
    got = run_attention(q, k, v, out["mask"], plen)
    check(q, k, v, out["mask"].cpu().numpy(), plen, got)


def test_rows_that_see_nothing_are_zero():
    n1, P = 17, 8
    q, k, v, _ = W.verify_inputs(2, 2, 1, n1, P, 64, seed=103)
    mask = np.zeros((2, n1, n1), np.uint8)
    mask[1] = np.eye(n1, dtype=np.uint8)
    plen = np.zeros(2, np.int32)
    got = run_attention(q, k, v, torch.from_numpy(mask).cuda(), plen)
    assert (got[0] == 0).all()
    np.testing.assert_allclose(got[1], np.repeat(W.bf16_bits_to_f32(v[1, :, P:]), 2, axis=0),
                               atol=1e-6)


def test_qwen3_8b_verification_shape_sampled():
    """Batch 32 trees of the Qwen3-8B workload (N = 64), 32 query heads over 8
    key/value heads, dh = 128, prefix cache padded to 1024 with lengths in
    [512, 1024]; every head of three requests (all key/value heads and every
    row tile of the stacked query heads) against the oracle, all finite."""
    wl = W.make_workload(3)
    tb = dt.TreeBuilder.from_numpy(wl)
    out = tb.run(**tb.inputs_to_device(wl))
    torch.cuda.synchronize()
    q, k, v, plen = W.verify_inputs(32, 32, 8, 65, 1024, 128, seed=3, min_prefix=512)
    got = run_attention(q, k, v, out["mask"], plen)
    assert np.isfinite(got).all()
    check(q, k, v, out["mask"].cpu().numpy(), plen, got,
          pairs=[(b, h) for b in (0, 5, 31) for h in range(32)])


@pytest.mark.parametrize("profile", ["rising", "falling", "alternating"])
def test_rescaled_accumulator(profile):
    """Key norms set per 64-key chunk so that the scores' maximum jumps by about
    10 from one chunk to the next (rising: every chunk moves the reference
    maximum and rescales the accumulated output; falling: none does after the
    first; alternating: every other one), prefix of 256 keys fully visible plus
    the tree rows under a GPU-built mask; against the fp64 oracle."""
    out = gpu_trees(64, 2, 131)
    n1, P, dh, H, Hkv = 65, 256, 128, 4, 2
    q, _, v, _ = W.verify_inputs(2, H, Hkv, n1, P, dh, seed=132)
    plen = np.full(2, P, np.int32)
    rng = np.random.default_rng(133)
    L = P + n1
    chunk = np.arange(L) // 64
    nch = int(chunk.max()) + 1
    order = {"rising": np.arange(nch), "falling": np.arange(nch)[::-1],
             "alternating": np.where(np.arange(nch) % 2 == 0, np.arange(nch), 0)}[profile]
    gain = (4.0 + 4.0 * order[chunk]).astype(np.float32)   # scores ~ N(0, gain^2)
    k = W.f32_to_bf16_bits(rng.standard_normal((2, Hkv, L, dh), dtype=np.float32)
                           * gain[None, None, :, None])
    got = run_attention(q, k, v, out["mask"], plen)
    assert np.isfinite(got).all()
    check(q, k, v, out["mask"].cpu().numpy(), plen, got)
