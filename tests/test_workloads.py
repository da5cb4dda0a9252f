"""The seeded input generator: reproducible, tensor streams independent, and
the shapes and value ranges every other test relies on. CPU only."""
from __future__ import annotations

import numpy as np

import dt_workloads as W

SMALL = dict(V=700, d=16, d_s=16, r=8, D=5, M=7, k=2, N=20, batch=3, wdtype="bf16",
             logits="zipf", zipf=(0.8, 1.6))


def test_same_seed_same_bytes():
    a = W.custom_workload(seed=5, **SMALL)
    b = W.custom_workload(seed=5, **SMALL)
    for key in ("base_logits", "H", "state0", "anchor", "E", "W_ih", "W_hh", "W1", "W2"):
        np.testing.assert_array_equal(getattr(a, key), getattr(b, key))
    np.testing.assert_array_equal(W.chain_uniforms(3, 5, 5), W.chain_uniforms(3, 5, 5))
    for x, y in zip(W.verify_inputs(2, 4, 2, 9, 6, 64, 5), W.verify_inputs(2, 4, 2, 9, 6, 64, 5)):
        np.testing.assert_array_equal(x, y)


def test_streams_are_independent():
    """Each tensor draws from its own child stream: changing one tensor's shape
    (here the rank r, which sizes W1 and W2) leaves the others' values alone."""
    a = W.custom_workload(seed=6, **SMALL)
    b = W.custom_workload(seed=6, **dict(SMALL, r=16))
    for key in ("base_logits", "H", "state0", "anchor", "E", "W_ih", "W_hh"):
        np.testing.assert_array_equal(getattr(a, key), getattr(b, key))


def test_shapes_and_ranges():
    wl = W.custom_workload(seed=7, **SMALL)
    assert wl.base_logits.shape == (3, 5, 700) and wl.base_logits.dtype == np.float32
    assert wl.H.shape == (3, 5, 16) and wl.state0.shape == (3, 16)
    assert wl.W2.shape == (700, 8) and wl.W2.dtype == np.uint16          # bf16 bits
    assert ((wl.anchor >= 0) & (wl.anchor < 700)).all()
    assert np.isfinite(wl.base_logits).all()
    u = W.chain_uniforms(4, 6, 7)
    assert u.shape == (4, 6) and u.dtype == np.float32 and (u >= 0).all() and (u < 1).all()
    q, k, v, plen = W.verify_inputs(2, 4, 2, 9, 6, 64, 7, min_prefix=3)
    assert q.shape == (2, 4, 9, 64) and k.shape == v.shape == (2, 2, 15, 64)
    assert q.dtype == np.uint16 and ((plen >= 3) & (plen <= 6)).all()


def test_bf16_rounding_is_round_to_nearest_even():
    import torch
    x = np.random.default_rng(8).standard_normal(10000).astype(np.float32)
    x = np.concatenate([x, np.float32([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(W.f32_to_bf16_bits(x), want)
    np.testing.assert_array_equal(W.bf16_bits_to_f32(want),
                                  torch.from_numpy(want.view(np.int16)).view(torch.bfloat16)
                                  .float().numpy())
