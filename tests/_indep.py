"""Independent checks of the oracle built from library routines and brute force.

Nothing here calls the oracle's arithmetic except where a test says so
explicitly (the brute-force search reuses the oracle's per-node scoring, so
that it pins only the best-first search).

* ``torch_path``: scores a token path with torch in float64 -- nn.GRUCell for
  the GRU, matmul + F.silu for the correction, torch.log_softmax for the
  normalisation, a stable descending torch.sort for the candidate sets.
* ``canonical_order``: sort-based replacement of the best-first heap: nodes by
  score descending; equal scores by (parent position, child rank), resolved
  group by group.
* ``enumerate_tree``: the whole implicit candidate tree (every node has the k
  best children among its depth's top-M candidates, depth <= D).
"""
from __future__ import annotations

import numpy as np
import torch

from dt_workloads import bf16_bits_to_f32


def weights_f64(w):
    def dec(a):
        if a is None:
            return None
        a = bf16_bits_to_f32(a) if w.wdtype == "bf16" else np.asarray(a, dtype=np.float32)
        return torch.from_numpy(np.asarray(a, dtype=np.float64))
    return dict(E=dec(w.E), W_ih=dec(w.W_ih), W_hh=dec(w.W_hh), W1=dec(w.W1), W2=dec(w.W2),
                b_ih=None if w.b_ih is None else torch.from_numpy(w.b_ih.astype(np.float64)),
                b_hh=None if w.b_hh is None else torch.from_numpy(w.b_hh.astype(np.float64)))


def gru_cell(W, d, d_s):
    cell = torch.nn.GRUCell(d, d_s, bias=True, dtype=torch.float64)
    with torch.no_grad():
        cell.weight_ih.copy_(W["W_ih"])
        cell.weight_hh.copy_(W["W_hh"])
        cell.bias_ih.copy_(W["b_ih"] if W["b_ih"] is not None else torch.zeros(3 * d_s,
                                                                              dtype=torch.float64))
        cell.bias_hh.copy_(W["b_hh"] if W["b_hh"] is not None else torch.zeros(3 * d_s,
                                                                              dtype=torch.float64))
    return cell


class TorchScorer:
    """float64 library-routine scoring of paths below request b's anchor."""

    def __init__(self, w, b=0):
        self.w, self.b = w, b
        self.W = weights_f64(w)
        self.cell = gru_cell(self.W, w.d, w.d_s)
        base = torch.from_numpy(np.asarray(w.base_logits[b], dtype=np.float64))
        self.base = base
        # candidate sets: stable descending sort keeps equal values in id order
        self.cand = torch.sort(base, dim=1, descending=True, stable=True).indices[:, :w.M]
        H = torch.from_numpy(np.asarray(w.H[b], dtype=np.float64))
        self.U = H @ self.W["W1"][:, :w.d].T                          # [D][r]
        T = float(w.temperature[b])
        self.T = 1.0 if T == 0.0 else T
        s0 = torch.from_numpy(np.asarray(w.state0[b], dtype=np.float64))
        with torch.no_grad():
            self.s_root = self.cell(self.W["E"][int(w.anchor[b])][None], s0[None])[0]

    def step(self, s, tok):
        with torch.no_grad():
            return self.cell(self.W["E"][int(tok)][None], s[None])[0]

    def logits(self, s, j):
        """corrected, temperature-scaled logits of the candidates of depth j (1-based)."""
        w = self.w
        h = torch.nn.functional.silu(self.U[j - 1] + self.W["W1"][:, w.d:] @ s)
        C = self.cand[j - 1]
        return C, (self.base[j - 1][C] + self.W["W2"][C] @ h) / self.T

    def path(self, path):
        """(score, lp per step, in_tree) of a token path."""
        s = self.s_root
        total, lps, in_tree = 0.0, [], True
        for j, tok in enumerate(path, start=1):
            C, L = self.logits(s, j)
            lp = torch.log_softmax(L, dim=0)
            pos = (C == int(tok)).nonzero()
            assert pos.numel() == 1, "token not among the depth's top-M"
            pos = int(pos[0, 0])
            order = np.lexsort((C.numpy(), -L.numpy()))
            if pos not in set(order[:self.w.k].tolist()):
                in_tree = False
            total += float(lp[pos])
            lps.append(float(lp[pos]))
            s = self.step(s, tok)
        return total, lps, in_tree


def canonical_order(scores, parents, ranks):
    """Positions of nodes under (score desc, parent position asc, rank asc).

    ``scores``/``parents``/``ranks`` index node ids; node 0 is the root (parent -1).
    Equal scores are resolved group by group: a node is ready once its parent
    has a position; among ready nodes the smallest (parent position, rank) goes
    first. Returns the node ids in canonical order (root first)."""
    ids = list(range(1, len(scores)))
    ids.sort(key=lambda n: -float(scores[n]))
    pos = {0: 0}
    order = [0]
    i = 0
    while i < len(ids):
        jend = i
        while jend < len(ids) and float(scores[ids[jend]]) == float(scores[ids[i]]):
            jend += 1
        remaining = set(ids[i:jend])
        while remaining:
            ready = [n for n in remaining if parents[n] in pos]
            n = min(ready, key=lambda q: (pos[parents[q]], ranks[q]))
            pos[n] = len(order)
            order.append(n)
            remaining.remove(n)
        i = jend
    return order


def enumerate_tree(D, k, children_fn):
    """All nodes of the implicit tree. children_fn(path) -> (tokens[k], lp[k]) in
    rank order. Returns lists (paths, scores(float32), parents, ranks, depths)."""
    paths, scores, parents, ranks, depths = [()], [np.float32(0.0)], [-1], [0], [0]
    frontier = [0]
    while frontier:
        nxt = []
        for n in frontier:
            if depths[n] >= D:
                continue
            toks, lps = children_fn(paths[n])
            for rnk in range(k):
                paths.append(paths[n] + (int(toks[rnk]),))
                scores.append(np.float32(scores[n] + np.float32(lps[rnk])))
                parents.append(n)
                ranks.append(rnk)
                depths.append(depths[n] + 1)
                nxt.append(len(paths) - 1)
        frontier = nxt
    return paths, scores, parents, ranks, depths


def top_n_tree(N, paths, scores, parents, ranks, depths):
    """First N+1 nodes (root included) in canonical order, as output arrays."""
    order = canonical_order(scores, parents, ranks)[:N + 1]
    pos = {n: i for i, n in enumerate(order)}
    tok = np.full(N + 1, -1, np.int32)
    par = np.full(N + 1, -1, np.int32)
    dep = np.full(N + 1, -1, np.int32)
    sc = np.full(N + 1, -np.inf, np.float32)
    for i, n in enumerate(order):
        tok[i] = paths[n][-1] if paths[n] else -2   # root token is filled by the caller
        par[i] = pos[parents[n]] if parents[n] >= 0 else -1
        dep[i] = depths[n]
        sc[i] = scores[n]
    return dict(tokens=tok, parents=par, depths=dep, scores=sc, n_nodes=len(order),
                paths=[paths[n] for n in order])


def ancestor_mask(parents, n_nodes, N):
    m = np.zeros((N + 1, N + 1), np.uint8)
    for i in range(n_nodes):
        a = i
        while a >= 0:
            m[i, a] = 1
            a = int(parents[a])
    return m
