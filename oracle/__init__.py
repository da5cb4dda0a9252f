"""ctypes front end of the plain-C CPU oracle (``dt_oracle.c``).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this module. The product
package never imports it and shares no code with it.

``build()`` compiles ``dt_oracle.c`` with gcc into ``liboracle.so`` next to it
(rebuilt when the source is newer). Threads: every C call releases the GIL, so
``build_trees(..., threads=n)`` runs requests concurrently.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dt_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ENONFINITE, ENOMEM = 0, -1, -4, -6


class _Model(C.Structure):
    _fields_ = [("V", C.c_int), ("d", C.c_int), ("d_s", C.c_int), ("r", C.c_int),
                ("D", C.c_int), ("M", C.c_int), ("k", C.c_int), ("N", C.c_int),
                ("wdtype", C.c_int),
                ("E", C.c_void_p), ("W_ih", C.c_void_p), ("W_hh", C.c_void_p),
                ("b_ih", C.c_void_p), ("b_hh", C.c_void_p), ("W1", C.c_void_p),
                ("W2", C.c_void_p)]


class _Request(C.Structure):
    _fields_ = [("base", C.c_void_p), ("H", C.c_void_p), ("state0", C.c_void_p),
                ("anchor", C.c_int32), ("temperature", C.c_float)]


class _Tree(C.Structure):
    _fields_ = [("tokens", C.c_void_p), ("parents", C.c_void_p), ("depths", C.c_void_p),
                ("scores", C.c_void_p), ("mask", C.c_void_p), ("topm", C.c_void_p),
                ("n_nodes", C.c_int32), ("n_expanded", C.c_int32)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, no target-specific flags)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                                   "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def load(path: str):
    """A ctypes handle on an oracle build at ``path`` with the argument types
    set (``lib()`` loads the default build; the mutation tests load others)."""
    L = C.CDLL(path)
    L.orc_topm.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p]
    L.orc_gru_step.argtypes = [C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    L.orc_gru_step.restype = None
    L.orc_build_tree.argtypes = [C.POINTER(_Model), C.POINTER(_Request), C.POINTER(_Tree)]
    L.orc_children.argtypes = [C.POINTER(_Model), C.POINTER(_Request), C.c_void_p, C.c_int,
                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    L.orc_score_path.argtypes = [C.POINTER(_Model), C.POINTER(_Request), C.c_void_p, C.c_int,
                                 C.c_void_p, C.c_void_p]
    L.orc_chain.argtypes = [C.POINTER(_Model), C.POINTER(_Request), C.c_void_p, C.c_void_p,
                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load(_LIB)
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _model(w, dims=None) -> tuple[_Model, list]:
    keep = []

    def c(a, dt=None):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dt) if dt else np.ascontiguousarray(a)
        keep.append(a)
        return a.ctypes.data

    m = _Model(w.V, w.d, w.d_s, w.r, w.D, w.M, w.k, w.N, 1 if w.wdtype == "bf16" else 0,
               c(w.E), c(w.W_ih), c(w.W_hh), c(w.b_ih, np.float32), c(w.b_hh, np.float32),
               c(w.W1), c(w.W2))
    return m, keep


def _request(w, b, keep):
    base = np.ascontiguousarray(w.base_logits[b], dtype=np.float32)
    H = np.ascontiguousarray(w.H[b], dtype=np.float32)
    s0 = np.ascontiguousarray(w.state0[b], dtype=np.float32)
    keep += [base, H, s0]
    return _Request(base.ctypes.data, H.ctypes.data, s0.ctypes.data, int(w.anchor[b]),
                    float(w.temperature[b]))


def topm(row: np.ndarray, M: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.float32)
    out = np.empty(M, dtype=np.int32)
    rc = lib().orc_topm(row.ctypes.data, row.size, M, out.ctypes.data)
    if rc:
        raise ValueError(f"orc_topm failed: {rc}")
    return out


def gru_step(W_ih, W_hh, x, s, b_ih=None, b_hh=None, wdtype="f32") -> np.ndarray:
    """One GRU cell step. Weights as float32 arrays, or uint16 bf16 bits with wdtype='bf16'."""
    dt = np.uint16 if wdtype == "bf16" else np.float32
    W_ih = np.ascontiguousarray(W_ih, dtype=dt)
    W_hh = np.ascontiguousarray(W_hh, dtype=dt)
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    d_s = s.size
    d = x.size
    assert W_ih.shape == (3 * d_s, d) and W_hh.shape == (3 * d_s, d_s)
    bi = None if b_ih is None else np.ascontiguousarray(b_ih, dtype=np.float32)
    bh = None if b_hh is None else np.ascontiguousarray(b_hh, dtype=np.float32)
    out = np.empty(d_s, dtype=np.float32)
    lib().orc_gru_step(d, d_s, 1 if wdtype == "bf16" else 0, W_ih.ctypes.data, W_hh.ctypes.data,
                       _ptr(bi), _ptr(bh), x.ctypes.data, s.ctypes.data, out.ctypes.data)
    return out


def build_tree(w, b: int = 0, *, mask: bool = True, topm_out: bool = True) -> dict:
    """Build request ``b`` of workload ``w``. Returns numpy arrays and the status."""
    m, keep = _model(w)
    q = _request(w, b, keep)
    N1 = w.N + 1
    out = dict(tokens=np.empty(N1, np.int32), parents=np.empty(N1, np.int32),
               depths=np.empty(N1, np.int32), scores=np.empty(N1, np.float32))
    if mask:
        out["mask"] = np.empty((N1, N1), np.uint8)
    if topm_out:
        out["topm"] = np.empty((w.D, w.M), np.int32)
    t = _Tree(out["tokens"].ctypes.data, out["parents"].ctypes.data, out["depths"].ctypes.data,
              out["scores"].ctypes.data, _ptr(out.get("mask")), _ptr(out.get("topm")), 0, 0)
    rc = lib().orc_build_tree(C.byref(m), C.byref(q), C.byref(t))
    out["status"] = rc
    out["n_nodes"] = t.n_nodes
    out["n_expanded"] = t.n_expanded
    return out


def build_trees(w, requests=None, *, threads: int | None = None, mask: bool = True,
                topm_out: bool = True) -> list[dict]:
    """Build several requests of ``w`` (all by default), ``threads`` at a time."""
    reqs = list(range(w.batch)) if requests is None else list(requests)
    lib()
    threads = threads or 1
    if threads == 1 or len(reqs) == 1:
        return [build_tree(w, b, mask=mask, topm_out=topm_out) for b in reqs]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda b: build_tree(w, b, mask=mask, topm_out=topm_out), reqs))


def children(w, path, b: int = 0):
    """(top-k tokens, their lp, lp of all M candidates, the candidate ids) of the
    node reached by ``path`` from request ``b``'s root."""
    m, keep = _model(w)
    q = _request(w, b, keep)
    p = np.ascontiguousarray(np.asarray(path, dtype=np.int32))
    toks = np.empty(w.k, np.int32)
    lps = np.empty(w.k, np.float32)
    all_lp = np.empty(w.M, np.float32)
    cand = np.empty(w.M, np.int32)
    rc = lib().orc_children(C.byref(m), C.byref(q), p.ctypes.data if p.size else None, int(p.size),
                            toks.ctypes.data, lps.ctypes.data, all_lp.ctypes.data,
                            cand.ctypes.data)
    if rc:
        raise ValueError(f"orc_children failed: {rc}")
    return toks, lps, all_lp, cand


def score_path(w, path, b: int = 0):
    """(score, in_tree) of a token path below request ``b``'s anchor."""
    m, keep = _model(w)
    q = _request(w, b, keep)
    p = np.ascontiguousarray(np.asarray(path, dtype=np.int32))
    sc = np.empty(1, np.float32)
    it = np.empty(1, np.int32)
    rc = lib().orc_score_path(C.byref(m), C.byref(q), p.ctypes.data if p.size else None,
                              int(p.size), sc.ctypes.data, it.ctypes.data)
    if rc:
        raise ValueError(f"orc_score_path failed: {rc}")
    return float(sc[0]), int(it[0])


def chain(w, b: int = 0, uniforms=None, forced=None) -> dict:
    """Domino chain decoding of request ``b`` (``orc_chain``): D draft tokens,
    greedy at T = 0, else drawn by inverse CDF at ``uniforms[b]`` ([batch][D]
    array, or None for zeros). ``forced`` ([D] tokens) replays the chain along
    given tokens. Returns decided, tokens, lp, margin and the status."""
    m, keep = _model(w)
    q = _request(w, b, keep)
    u = None
    if uniforms is not None:
        u = np.ascontiguousarray(np.asarray(uniforms)[b], dtype=np.float32)
    f = None if forced is None else np.ascontiguousarray(np.asarray(forced), dtype=np.int32)
    out = dict(decided=np.full(w.D, -1, np.int32), tokens=np.full(w.D, -1, np.int32),
               lp=np.full(w.D, np.nan, np.float32), margin=np.full(w.D, np.nan, np.float32))
    rc = lib().orc_chain(C.byref(m), C.byref(q), _ptr(u), _ptr(f), out["decided"].ctypes.data,
                         out["tokens"].ctypes.data, out["lp"].ctypes.data,
                         out["margin"].ctypes.data)
    out["status"] = rc
    return out


def chains(w, requests=None, uniforms=None, forced=None, *, threads: int | None = None):
    """``chain`` for several requests (all by default), ``threads`` at a time;
    ``forced`` is then [batch][D]."""
    reqs = list(range(w.batch)) if requests is None else list(requests)
    lib()
    run = lambda b: chain(w, b, uniforms, None if forced is None else np.asarray(forced)[b])
    if (threads or 1) == 1 or len(reqs) == 1:
        return [run(b) for b in reqs]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(run, reqs))


# ------------------------------------------------ verify-side consumption
# "Riassunto Tecnico: DominoTree", Componenti Core 5: the target model checks
# every drafted node in one forward pass with tree attention, each node seeing
# the verified prefix and its own ancestors (the ancestor mask of the tree).

def tree_positions(depths: np.ndarray, prefix_len: np.ndarray) -> np.ndarray:
    """Position ids of the tree rows. The prefix cache holds the prefix_len[b]
    tokens before the anchor (positions 0 .. prefix_len - 1); the anchor is
    tree row 0 at position prefix_len and a node at depth j sits j places
    after it: prefix_len[b] + depth. Empty rows (depth -1) get -1."""
    depths = np.asarray(depths)
    out = np.full(depths.shape, -1, dtype=np.int32)
    for b in range(depths.shape[0]):
        for i in range(depths.shape[1]):
            if depths[b, i] >= 0:
                out[b, i] = int(prefix_len[b]) + int(depths[b, i])
    return out


def tree_attention(q, k, v, mask, prefix_len, scale) -> np.ndarray:
    """Attention of the tree rows, in fp64, written from the definition.

    q [batch][H][N1][dh], k and v [batch][Hkv][P + N1][dh] (the first P keys
    are the prefix cache, key P + t is tree row t), mask [batch][N1][N1] (row i
    may see tree row t iff mask[i][t]), prefix_len [batch] (prefix keys
    p < prefix_len[b] are visible to every row; the rest are padding). Query
    head h reads key/value head h // (H / Hkv). For row i of head h:
        s_j = scale * q_i . k_j   over the visible keys j
        out_i = sum_j softmax(s)_j v_j,   0 when no key is visible.
    Returns float64 [batch][H][N1][dh]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N1, dh = q.shape
    Hkv, L = k.shape[1], k.shape[2]
    P = L - N1
    group = H // Hkv
    out = np.zeros((B, H, N1, dh))
    for b in range(B):
        for h in range(H):
            kh, vh = k[b, h // group], v[b, h // group]
            for i in range(N1):
                vis = [j for j in range(int(prefix_len[b]))] + \
                      [P + t for t in range(N1) if mask[b, i, t]]
                if not vis:
                    continue
                s = np.array([scale * np.dot(q[b, h, i], kh[j]) for j in vis])
                w = np.exp(s - s.max())
                w /= w.sum()
                out[b, h, i] = sum(w[n] * vh[j] for n, j in enumerate(vis))
    return out


# ------------------------------------------------- CondAdaptive budget
# "Riassunto Tecnico: DominoTree", Componenti Core 4: a cost-aware adaptive
# budget (CaDDTree's rule: stop growing the tree when the throughput gain
# fades) tried on the conditional tree, found to saturate at the maximum budget.

def adaptive_count(scores: np.ndarray, tokens: np.ndarray, c_fixed: float, c_node: float) -> int:
    """Nodes kept by the cost-aware rule on one tree (rows in pop order, row 0
    the root). Expected accepted length A(n) = 1 + sum_{i<=n} exp(score_i) (the
    drafter's path probabilities), round cost C(n) = c_fixed + c_node n;
    node n is kept while A(n) / C(n) > A(n - 1) / C(n - 1), i.e. while
    exp(score_n) C(n - 1) > A(n - 1) c_node, all in fp64, in pop order; growth
    stops at the first node that fails or at the first empty row."""
    A, C, n_keep = 1.0, float(c_fixed), 0
    for n in range(1, len(scores)):
        if tokens[n] < 0:
            break
        e = float(np.exp(np.float64(scores[n])))
        if e * C > A * float(c_node):
            A += e
            C += float(c_node)
            n_keep = n
        else:
            break
    return n_keep


def truncate_tree(tree: dict, n_keep: int) -> dict:
    """The tree cut to its first n_keep + 1 rows (a prefix of the pop order is
    a subtree: every ancestor of a row has a lower index); later rows empty."""
    out = {k: np.array(v, copy=True) for k, v in tree.items() if isinstance(v, np.ndarray)}
    for key, fill in (("tokens", -1), ("parents", -1), ("depths", -1), ("scores", -np.inf)):
        out[key][n_keep + 1:] = fill
    if "mask" in out:
        out["mask"][n_keep + 1:] = 0
    return out
