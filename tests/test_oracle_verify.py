"""Pins of the oracle's verify-side functions (tree positions, tree attention), CPU only.

* tree attention against torch's scaled_dot_product_attention in float64 with a
  boolean mask built from the prefix length and the ancestor mask, including
  grouped key/value heads (a library routine, not a restatement);
* closed forms: equal value rows give that row; a row that sees only itself
  gives its own value; scale 0 gives the plain mean of the visible values; a
  row that sees nothing gives 0;
* positions on real trees: the root at the prefix length, every node one past
  its parent, empty rows -1.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import dt_workloads as W
import oracle


def tree_inputs(seed, B=2, H=4, Hkv=2, dh=16, N=12, P=5, ragged=True):
    wl = W.custom_workload(V=300, d=16, d_s=16, r=8, D=4, M=6, k=3, N=N, batch=B, wdtype="f32",
                           seed=seed, logits="spiked", e_std=0.5)
    trees = oracle.build_trees(wl)
    mask = np.stack([t["mask"] for t in trees])
    depths = np.stack([t["depths"] for t in trees])
    rng = np.random.default_rng(seed)
    N1 = N + 1
    q = rng.standard_normal((B, H, N1, dh))
    k = rng.standard_normal((B, Hkv, P + N1, dh))
    v = rng.standard_normal((B, Hkv, P + N1, dh))
    plen = rng.integers(0, P + 1, B) if ragged else np.full(B, P)
    return q, k, v, mask, depths, plen


def visible(mask, plen, P):
    B, N1, _ = mask.shape
    vis = np.zeros((B, N1, P + N1), bool)
    for b in range(B):
        vis[b, :, :plen[b]] = True
        vis[b, :, P:] = mask[b].astype(bool)
    return vis


@pytest.mark.parametrize("seed", [81, 82, 83])
def test_tree_attention_matches_torch_sdpa(seed):
    q, k, v, mask, _, plen = tree_inputs(seed)
    B, H, N1, dh = q.shape
    Hkv, P = k.shape[1], k.shape[2] - N1
    scale = 1.0 / np.sqrt(dh)
    got = oracle.tree_attention(q, k, v, mask, plen, scale)
    vis = visible(mask, plen, P)
    rep = H // Hkv
    kt = torch.from_numpy(k).repeat_interleave(rep, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(rep, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), kt, vt, attn_mask=torch.from_numpy(vis)[:, None], scale=scale).numpy()
    has = vis.any(-1)                               # rows with at least one visible key
    for b in range(B):
        np.testing.assert_allclose(got[b][:, has[b]], ref[b][:, has[b]], atol=1e-12, rtol=1e-10)
        assert (got[b][:, ~has[b]] == 0).all()


def test_tree_attention_closed_forms():
    q, k, v, mask, _, plen = tree_inputs(84, ragged=False)
    B, H, N1, dh = q.shape
    P = k.shape[2] - N1
    c = np.linspace(-1, 1, dh)
    v_eq = np.broadcast_to(c, v.shape).copy()
    out = oracle.tree_attention(q, k, v_eq, mask, plen, 0.3)
    np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), atol=1e-12)
    eye = np.broadcast_to(np.eye(N1, dtype=np.uint8), mask.shape)
    out = oracle.tree_attention(q, k, v, eye, np.zeros(B, int), 0.3)
    np.testing.assert_allclose(out, np.repeat(v[:, :, P:], H // k.shape[1], axis=1), atol=1e-12)
    out = oracle.tree_attention(q, k, v, mask, plen, 0.0)
    vis = visible(mask, plen, P)
    for b in range(B):
        for h in range(H):
            vh = v[b, h // (H // k.shape[1])]
            for i in range(N1):
                np.testing.assert_allclose(out[b, h, i], vh[vis[b, i]].mean(axis=0), atol=1e-12)
    none = np.zeros_like(mask)
    assert (oracle.tree_attention(q, k, v, none, np.zeros(B, int), 0.3) == 0).all()


def test_tree_positions_follow_the_tree():
    _, _, _, mask, depths, plen = tree_inputs(85, N=30)
    pos = oracle.tree_positions(depths, plen)
    for b in range(depths.shape[0]):
        tree = oracle.build_trees(W.custom_workload(V=300, d=16, d_s=16, r=8, D=4, M=6, k=3, N=30,
                                                    batch=depths.shape[0], wdtype="f32", seed=85,
                                                    logits="spiked", e_std=0.5))[b]
        assert pos[b, 0] == plen[b]
        for i in range(1, depths.shape[1]):
            if depths[b, i] < 0:
                assert pos[b, i] == -1
            else:
                assert pos[b, i] == pos[b, tree["parents"][i]] + 1
