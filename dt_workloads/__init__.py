"""Seeded synthetic workloads for the conditional draft-tree builder.

This module only draws random inputs. It holds none of the builder's arithmetic:
no top-M, no GRU, no correction, no softmax, no search. Both the CUDA path and
the CPU oracle consume the exact bytes produced here.

Shapes follow the draft block of the Domino drafter ("Domino: decoupling causal
modelling from autoregressive drafting", reproduction section: block size 16,
GRU state 1024, correction rank 256) and the Qwen3-4B / Qwen3-8B vocabulary and
hidden sizes. The evaluation suites the pages use (math, code and chat
benchmarks) are not available; the Zipf-shaped base logits below stand in for
the mix of sharp and flat per-position marginals those suites produce.

Reading of the distribution notation (stated once, used everywhere):
  * "N(0, s)" for logits, H, E of the tiny case and the logit noise: s is the
    standard deviation;
  * "N(0, 1/fan_in)" for weights: 1/fan_in is the variance (LeCun init), with
    fan_in = d for W_ih and E, d_s for W_hh, d + d_s for W1, r for W2.

Every tensor gets its own child of ``np.random.SeedSequence(seed)`` so that the
shape of one tensor never changes the values of another.
"""
from __future__ import annotations

import dataclasses
import numpy as np

__all__ = ["Workload", "CONFIGS", "make_workload", "custom_workload", "f32_to_bf16_bits",
           "bf16_bits_to_f32", "chain_uniforms", "verify_inputs"]

# Index of each tensor's child seed. Fixed forever: changing it changes every input.
_SEED_SLOTS = {
    "base": 0, "spikes": 1, "H": 2, "E": 3, "W_ih": 4, "W_hh": 5, "W1": 6, "W2": 7,
    "anchor": 8, "zipf_s": 9, "state0": 10, "b_ih": 11, "b_hh": 12, "chain_u": 13,
    "verify": 14,
}
_N_SLOTS = 16


@dataclasses.dataclass
class Workload:
    """One batch of builder inputs, host-resident, C-contiguous."""
    name: str
    V: int
    d: int
    d_s: int
    r: int
    D: int
    M: int
    k: int
    N: int
    batch: int
    wdtype: str                 # "f32" or "bf16"
    base_logits: np.ndarray     # [batch][D][V] float32
    H: np.ndarray               # [batch][D][d] float32
    state0: np.ndarray          # [batch][d_s] float32
    anchor: np.ndarray          # [batch] int32
    temperature: np.ndarray     # [batch] float32
    E: np.ndarray               # [V][d]          uint16 (bf16 bits) or float32
    W_ih: np.ndarray            # [3 d_s][d]
    W_hh: np.ndarray            # [3 d_s][d_s]
    W1: np.ndarray              # [r][d + d_s]
    W2: np.ndarray              # [V][r]
    b_ih: np.ndarray | None = None   # [3 d_s] float32 or None
    b_hh: np.ndarray | None = None   # [3 d_s] float32 or None

    @property
    def dims(self) -> dict:
        return dict(V=self.V, d=self.d, d_s=self.d_s, r=self.r, D=self.D, M=self.M,
                    k=self.k, N=self.N, batch=self.batch)

    def request(self, b: int) -> "Workload":
        """A batch-1 view of request ``b`` (weights shared, not copied)."""
        return dataclasses.replace(
            self, name=f"{self.name}[{b}]", batch=1,
            base_logits=self.base_logits[b:b + 1], H=self.H[b:b + 1],
            state0=self.state0[b:b + 1], anchor=self.anchor[b:b + 1],
            temperature=self.temperature[b:b + 1])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rngs(seed: int):
    kids = np.random.SeedSequence(seed).spawn(_N_SLOTS)
    return {name: np.random.default_rng(kids[i]) for name, i in _SEED_SLOTS.items()}


def _normal(rng, shape, std, chunk_rows=8192):
    """float32 N(0, std^2), generated in row chunks to bound peak memory."""
    out = np.empty(shape, dtype=np.float32)
    flat = out.reshape(shape[0], -1) if len(shape) > 1 else out.reshape(-1, 1)
    for i in range(0, flat.shape[0], chunk_rows):
        blk = rng.standard_normal(flat[i:i + chunk_rows].shape, dtype=np.float32)
        blk *= np.float32(std)
        flat[i:i + chunk_rows] = blk
    return out


def _weight(rng, shape, var, wdtype):
    w = _normal(rng, shape, float(np.sqrt(var)))
    return w if wdtype == "f32" else f32_to_bf16_bits(w)


def _zipf_logits(rng, batch, D, V, exponents, noise_std):
    """logit(token) = 12 - s_b * ln(rank) + N(0, noise_std), rank over a fresh
    seeded permutation of the vocabulary for every (request, depth) row."""
    out = np.empty((batch, D, V), dtype=np.float32)
    lnrank = np.log(np.arange(1, V + 1, dtype=np.float64))
    for b in range(batch):
        s = float(exponents[b])
        for j in range(D):
            perm = rng.permutation(V)
            row = np.empty(V, dtype=np.float64)
            row[perm] = 12.0 - s * lnrank
            row += noise_std * rng.standard_normal(V)
            out[b, j] = row.astype(np.float32)
    return out


# name -> generator arguments. Index i is the i-th configuration of the build.
CONFIGS = {
    0: dict(name="tiny", V=1024, d=64, d_s=32, r=32, D=7, M=16, k=4, N=32, batch=1,
            wdtype="f32", seed=0, logits="spiked"),
    1: dict(name="qwen3-4b-b1", V=151936, d=2560, d_s=1024, r=256, D=15, M=64, k=8, N=64,
            batch=1, wdtype="bf16", seed=1, logits="zipf", zipf=(1.1, 1.1)),
    2: dict(name="qwen3-8b-b1", V=151936, d=4096, d_s=1024, r=256, D=15, M=128, k=8, N=128,
            batch=1, wdtype="bf16", seed=2, logits="zipf", zipf=(1.1, 1.1)),
    3: dict(name="qwen3-8b-b32", V=151936, d=4096, d_s=1024, r=256, D=15, M=64, k=8, N=64,
            batch=32, wdtype="bf16", seed=3, logits="zipf", zipf=(0.8, 1.6)),
    4: dict(name="stress-b128", V=151936, d=4096, d_s=1024, r=256, D=15, M=256, k=16, N=256,
            batch=128, wdtype="bf16", seed=4, logits="zipf", zipf=(0.8, 1.6),
            temperature="cycle"),
}


def custom_workload(*, name="custom", V, d, d_s, r, D, M, k, N, batch, wdtype="f32", seed=0,
                    logits="spiked", zipf=(1.1, 1.1), temperature=None, e_std=None,
                    state0_std=0.0, biases=False) -> Workload:
    """Generate a workload of arbitrary shape with the recipe above.

    logits="spiked": N(0, 2) per row plus three distinct seeded ids raised by +6.
    logits="zipf":   Zipf ranks over a seeded permutation, exponent U[zipf] per
                     request, plus N(0, 0.5) noise.
    e_std:           std of E; None means variance 1/d (bf16 configs), the tiny
                     case passes 0.02.
    temperature:     None (all 1.0), "cycle" (0.5, 1.0, 0.5, ...), a float, or an array.
    """
    g = _rngs(seed)
    if logits == "spiked":
        base = _normal(g["base"], (batch, D, V), 2.0)
        for b in range(batch):
            for j in range(D):
                ids = g["spikes"].choice(V, size=min(3, V), replace=False)
                base[b, j, ids] += np.float32(6.0)
    elif logits == "zipf":
        s = g["zipf_s"].uniform(zipf[0], zipf[1], size=batch) if zipf[0] != zipf[1] \
            else np.full(batch, zipf[0])
        base = _zipf_logits(g["base"], batch, D, V, s, 0.5)
    else:
        raise ValueError(logits)
    H = _normal(g["H"], (batch, D, d), 1.0)
    state0 = (_normal(g["state0"], (batch, d_s), state0_std) if state0_std
              else np.zeros((batch, d_s), dtype=np.float32))
    anchor = g["anchor"].integers(0, V, size=batch).astype(np.int32)
    if temperature is None:
        T = np.ones(batch, dtype=np.float32)
    elif isinstance(temperature, str) and temperature == "cycle":
        T = np.array([0.5 if b % 2 == 0 else 1.0 for b in range(batch)], dtype=np.float32)
    else:
        T = np.broadcast_to(np.asarray(temperature, dtype=np.float32), (batch,)).copy()
    e_std = (1.0 / np.sqrt(d)) if e_std is None else e_std
    E = _normal(g["E"], (V, d), e_std)
    E = E if wdtype == "f32" else f32_to_bf16_bits(E)
    W_ih = _weight(g["W_ih"], (3 * d_s, d), 1.0 / d, wdtype)
    W_hh = _weight(g["W_hh"], (3 * d_s, d_s), 1.0 / d_s, wdtype)
    W1 = _weight(g["W1"], (r, d + d_s), 1.0 / (d + d_s), wdtype)
    W2 = _weight(g["W2"], (V, r), 1.0 / r, wdtype)
    b_ih = b_hh = None
    if biases:
        b_ih = _normal(g["b_ih"], (3 * d_s,), 0.1)
        b_hh = _normal(g["b_hh"], (3 * d_s,), 0.1)
    return Workload(name=name, V=V, d=d, d_s=d_s, r=r, D=D, M=M, k=k, N=N, batch=batch,
                    wdtype=wdtype, base_logits=base, H=H, state0=state0, anchor=anchor,
                    temperature=T, E=E, W_ih=W_ih, W_hh=W_hh, W1=W1, W2=W2,
                    b_ih=b_ih, b_hh=b_hh)


def make_workload(cfg: int, batch: int | None = None) -> Workload:
    """The workload of configuration ``cfg`` (0..4). ``batch`` truncates the batch
    (the first requests are identical to the full batch's first requests only for
    the per-request tensors drawn row by row; use ``Workload.request`` to sample
    requests of the full batch)."""
    c = dict(CONFIGS[cfg])
    if batch is not None:
        c["batch"] = batch
    kw = {k: v for k, v in c.items() if k not in ("logits", "zipf", "temperature")}
    return custom_workload(logits=c["logits"], zipf=c.get("zipf", (1.1, 1.1)),
                           temperature=c.get("temperature"),
                           e_std=0.02 if cfg == 0 else None, **kw)


def chain_uniforms(batch: int, D: int, seed: int = 0) -> np.ndarray:
    """Uniform draws in [0, 1), float32 [batch][D]: the random numbers of the
    sampled (T > 0) chain decoder, one per draft position, passed to both the
    CUDA path and the oracle as an input. Drawn from the ``seed``'s own child
    stream, so they never change another tensor of the same seed."""
    kid = np.random.SeedSequence(seed).spawn(_N_SLOTS)[_SEED_SLOTS["chain_u"]]
    return np.random.default_rng(kid).random((batch, D), dtype=np.float32)


def verify_inputs(batch: int, H: int, Hkv: int, n1: int, P: int, dh: int, seed: int = 0,
                  min_prefix: int = 0):
    """Synthetic per-layer tensors of the target model for tree verification:
    q [batch][H][n1][dh], k and v [batch][Hkv][P + n1][dh] as bf16 bits
    (uint16, N(0, 1) values rounded to bf16), and prefix lengths [batch] int32
    uniform in [min_prefix, P] (the cache is padded to P keys). The target model
    itself is not available; these stand in for its projections."""
    kid = np.random.SeedSequence(seed).spawn(_N_SLOTS)[_SEED_SLOTS["verify"]]
    rng = np.random.default_rng(kid)
    q = f32_to_bf16_bits(rng.standard_normal((batch, H, n1, dh), dtype=np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((batch, Hkv, P + n1, dh), dtype=np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((batch, Hkv, P + n1, dh), dtype=np.float32))
    plen = rng.integers(min_prefix, P + 1, batch).astype(np.int32)
    return q, k, v, plen
