"""Top-M selection on the GPU against the oracle, on rows built to stress it.

The kernel streams each row once against a threshold that it raises as it goes
(the M-th largest value seen so far), and selects exactly by a radix select
over (value, id) keys. Rows are chosen so that every branch of that scheme
runs: ascending ramps (every tile beats the threshold, compaction after
compaction), descending ramps, values from a handful of levels (long runs of
exact ties, so ids decide), flat rows, rows of mostly -inf (fewer finite values
than M), signed zeros, extreme magnitudes and the Zipf-like logits of the
benchmark workload; M from 1 to 256; V a multiple of 4 (range launch) and
ragged (segment launch with scalar heads and tails). Both entry points that
run the top-M are checked: dt_build_trees (its top-M output, marginal mode so
that no weights are needed) and dt_select_topm_noalloc.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

dt = pytest.importorskip("conditional_draft_tree_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conditional_draft_tree_gb300 import build
    build.build()
    oracle.build()


KINDS = ("normal", "ascending", "descending", "levels", "flat", "mostly_neginf", "zeros",
         "extremes", "zipf")


def make_row(kind: str, V: int, M: int, rng) -> np.ndarray:
    if kind == "normal":
        return rng.standard_normal(V).astype(np.float32)
    if kind == "ascending":
        return np.linspace(-3.0, 3.0, V, dtype=np.float32)
    if kind == "descending":
        return np.linspace(3.0, -3.0, V, dtype=np.float32)
    if kind == "levels":
        return (np.rint(rng.standard_normal(V) * 2.0) / 2.0).astype(np.float32)
    if kind == "flat":
        return np.full(V, 0.25, dtype=np.float32)
    if kind == "mostly_neginf":
        row = np.full(V, -np.inf, dtype=np.float32)
        idx = rng.choice(V, size=max(1, M // 2), replace=False)
        row[idx] = rng.standard_normal(idx.size).astype(np.float32)
        return row
    if kind == "zeros":
        row = np.where(rng.random(V) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
        row[rng.choice(V, size=3, replace=False)] = -1.0
        return row
    if kind == "extremes":
        row = rng.standard_normal(V) * 3e38
        return np.clip(row, -3.4e38, 3.4e38).astype(np.float32)
    if kind == "zipf":
        rank = rng.permutation(V).astype(np.float64) + 1.0
        return (12.0 - 1.1 * np.log(rank) + rng.normal(0, 0.5, V)).astype(np.float32)
    raise ValueError(kind)


def logits_for(V: int, M: int, D: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = [make_row(KINDS[j % len(KINDS)], V, M, rng) for j in range(D)]
    return np.stack(rows)[None].copy()   # [1][D][V]


def expected(logits: np.ndarray, M: int) -> np.ndarray:
    return np.stack([[oracle.topm(logits[b, j], M) for j in range(logits.shape[1])]
                     for b in range(logits.shape[0])])


def topm_build_trees(logits: np.ndarray, M: int) -> tuple[np.ndarray, np.ndarray]:
    batch, D, V = logits.shape
    dims = dt.dims_of(V, 8, 8, 8, D, M, 1, 4, batch)
    mb = dt.MarginalTreeBuilder(dims)
    out = mb.run(torch.from_numpy(logits).cuda(),
                 torch.zeros(batch, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    return out["topm"].cpu().numpy(), out["status"].cpu().numpy()


def topm_noalloc(logits: np.ndarray, M: int) -> tuple[np.ndarray, np.ndarray]:
    batch, D, V = logits.shape
    topm = torch.full((batch, D, M), -7, dtype=torch.int32, device="cuda")
    status = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    rc = dt.select_topm_noalloc(torch.from_numpy(logits).cuda(), M, topm, status)
    assert rc == dt.OK, dt.status_string(rc)
    torch.cuda.synchronize()
    return topm.cpu().numpy(), status.cpu().numpy()


@pytest.mark.parametrize("V,M", [(151936, 64), (151936, 256), (151936, 1), (151936, 129),
                                 (20000, 100), (5001, 7), (4099, 256), (1001, 64), (300, 256)])
@pytest.mark.parametrize("entry", ["build_trees", "noalloc"])
def test_topm_stress_rows(V, M, entry):
    if M > V:
        pytest.skip("M > V")
    logits = logits_for(V, M, len(KINDS), seed=V * 7 + M)
    want = expected(logits, M)
    got, status = (topm_build_trees if entry == "build_trees" else topm_noalloc)(logits, M)
    assert list(status) == [dt.OK]
    for j in range(logits.shape[1]):
        np.testing.assert_array_equal(got[0, j], want[0, j], err_msg=f"row {j} ({KINDS[j]})")


def test_topm_many_rows_range_launch():
    """Many rows of a multiple-of-4 width, so that blocks' ranges straddle rows
    and most rows are merged from pieces of two or three blocks."""
    rng = np.random.default_rng(5)
    batch, D, V, M = 7, 13, 40000, 64
    logits = np.stack([[make_row(KINDS[(b * D + j) % len(KINDS)], V, M, rng) for j in range(D)]
                       for b in range(batch)])
    want = expected(logits, M)
    for fn in (topm_build_trees, topm_noalloc):
        got, status = fn(logits, M)
        assert (status == dt.OK).all()
        np.testing.assert_array_equal(got, want)
