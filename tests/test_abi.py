"""The C-ABI library builds, loads and exports every symbol include/dt.h declares.

CPU only: no call here launches device work. Argument validation happens before
any device access, so invalid shapes are rejected without a GPU.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dt():
    from conditional_draft_tree_gb300 import build
    build.build()
    import conditional_draft_tree_gb300 as dt
    return dt


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(dt_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_expected_entry_points(dt):
    assert declared_functions() == sorted(dt.EXPORTS)


def test_library_exports_every_declared_symbol(dt):
    lib = C.CDLL(dt.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_only_calls(dt):
    assert dt.abi_version() == 1
    assert dt.status_string(dt.OK) == "ok"
    assert "NaN" in dt.status_string(dt.ERR_NONFINITE)
    dims = dt.dims_of(V=151936, d=4096, d_s=1024, r=256, D=15, M=64, k=8, N=64, batch=32)
    assert dt.prepared_bytes(dims) == 4 * 151936 * 3 * 1024


@pytest.mark.parametrize("bad", [dict(k=9, M=8), dict(M=300), dict(d=12), dict(d_s=0),
                                 dict(r=7), dict(D=0), dict(N=-1), dict(batch=0), dict(M=2000, V=1000)])
def test_invalid_dims_rejected_before_device_work(dt, bad):
    base = dict(V=1024, d=64, d_s=32, r=32, D=7, M=16, k=4, N=32, batch=1)
    base.update(bad)
    dims = dt.dims_of(**base)
    assert dt.prepared_bytes(dims) == 0
    w = dt.DtWeights(16, 16, 16, None, None, 16, 16, 0)
    out = dt.DtTreeOut(16, 16, 16, 16, None, None, 16)
    rc = dt.lib().dt_build_trees(C.byref(dims), C.byref(w), 256, 256, 256, 256, 256, None, 256,
                                 1 << 20, C.byref(out), None, None)
    assert rc == dt.ERR_INVALID_ARG


def test_null_and_misaligned_pointers_rejected(dt):
    dims = dt.dims_of(V=1024, d=64, d_s=32, r=32, D=7, M=16, k=4, N=32, batch=1)
    out = dt.DtTreeOut(16, 16, 16, 16, None, None, 16)
    w_null = dt.DtWeights(None, 16, 16, None, None, 16, 16, 0)
    assert dt.lib().dt_build_trees(C.byref(dims), C.byref(w_null), 256, 256, 256, 256, 256, None,
                                   256, 1 << 20, C.byref(out), None, None) == dt.ERR_INVALID_ARG
    w_mis = dt.DtWeights(18, 16, 16, None, None, 16, 16, 0)
    assert dt.lib().dt_build_trees(C.byref(dims), C.byref(w_mis), 256, 256, 256, 256, 256, None,
                                   256, 1 << 20, C.byref(out), None, None) == dt.ERR_INVALID_ARG
    w = dt.DtWeights(16, 16, 16, None, None, 16, 16, 0)
    assert dt.lib().dt_build_trees(C.byref(dims), C.byref(w), 256, 256, 256, 256, 256, None,
                                   255, 1 << 20, C.byref(out), None, None) == dt.ERR_INVALID_ARG


def test_package_refuses_to_run_without_library(dt, monkeypatch, tmp_path):
    monkeypatch.setattr(dt, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(dt, "_lib", None)
    with pytest.raises(dt.DtError):
        dt.lib()


def _no_gpu():
    import torch
    return not torch.cuda.is_available()


@pytest.mark.skipif(not _no_gpu(), reason="passes unusable pointers; host-only check")
def test_marginal_mode_reads_no_weights(dt):
    """DT_OPT_MARGINAL reads no weights, prepared table, H or state0: NULL passes
    the argument checks (the call then stops at the device query on a host
    without a GPU); without the flag the same call is an invalid argument."""
    dims = dt.dims_of(V=1024, d=64, d_s=32, r=32, D=7, M=16, k=4, N=32, batch=1)
    out = dt.DtTreeOut(16, 16, 16, 16, None, None, 16)
    opt = dt.options(0, flags=dt.OPT_MARGINAL)
    call = lambda o: dt.lib().dt_build_trees(C.byref(dims), None, None, 256, None, None, 256, None,
                                             256, 1 << 20, C.byref(out), o, None)
    assert call(None) == dt.ERR_INVALID_ARG
    assert call(C.byref(opt)) in (dt.ERR_CUDA, dt.ERR_UNSUPPORTED)


def test_chain_entry_points_validate_before_device_work(dt):
    L = dt.lib()
    dims = dt.dims_of(V=151936, d=4096, d_s=1024, r=256, D=15, M=64, k=8, N=64, batch=32)
    # tiles of 128 rows x 64-wide K chunks, 16 KB each: [W_hh; W1_S] (3328 rows, K 1024)
    # and W2 (151936 rows, K 256)
    assert dt.chain_prepared_bytes(dims) == (26 * 16 + 1187 * 4) * 16384
    bad = dt.dims_of(V=1024, d=64, d_s=32, r=7, D=7, M=16, k=4, N=32, batch=1)
    assert dt.chain_prepared_bytes(bad) == 0
    w32 = dt.DtWeights(16, 16, 16, None, None, 16, 16, 0)
    w16 = dt.DtWeights(16, 16, 16, None, None, 16, 16, 1)
    assert L.dt_prepare_chain(C.byref(dims), C.byref(w32), 256, 1 << 30, None) == \
        dt.ERR_UNSUPPORTED
    assert L.dt_prepare_chain(C.byref(dims), C.byref(w16), 256, 16, None) == dt.ERR_INVALID_ARG
    # prepared, chain_prepared, base, H, state0, anchor, temperature, uniforms, workspace,
    # workspace_bytes, tokens, logprobs, status, stream
    args = [256, 256, 256, 256, 256, 256, None, None, 256, 1 << 30, 256, 256, 256, None]
    assert len(args) == len(L.dt_decode_chains.argtypes) - 2

    def decode(w, **over):
        a = list(args)
        for i, v in over.items():
            a[int(i[1:])] = v
        return L.dt_decode_chains(C.byref(dims), C.byref(w), *a)
    assert decode(w32) == dt.ERR_UNSUPPORTED              # f32 weights
    assert decode(w16, a2=None) == dt.ERR_INVALID_ARG      # no base logits
    assert decode(w16, a10=None) == dt.ERR_INVALID_ARG     # no token output
    assert decode(w16, a8=255) == dt.ERR_INVALID_ARG       # misaligned workspace
    assert decode(w16, a3=258) == dt.ERR_INVALID_ARG       # H not 16-byte aligned


def test_verify_and_adaptive_entry_points_validate_before_device_work(dt):
    L = dt.lib()
    # dt_tree_positions: sizes and pointers
    assert L.dt_tree_positions(None, 256, 1, 65, 256, None) == dt.ERR_INVALID_ARG
    assert L.dt_tree_positions(256, 256, 0, 65, 256, None) == dt.ERR_INVALID_ARG
    assert L.dt_tree_positions(256, 256, 1, 2000, 256, None) == dt.ERR_INVALID_ARG
    # dt_tree_attention: q k v mask prefix_len batch H Hkv n1 P dh scale out stream
    ok = [256, 256, 256, 256, 256, 2, 32, 8, 65, 1024, 128, 0.088, 256, None]
    for i, bad in ((6, 30), (7, 0), (10, 96), (8, 0), (9, -1), (11, float("inf")), (0, 258),
                   (12, 260), (3, None)):
        a = list(ok)
        a[i] = bad
        assert L.dt_tree_attention(*a) == dt.ERR_INVALID_ARG, (i, bad)
    # dt_adaptive_budget: costs and sizes
    out = dt.DtTreeOut(256, 256, 256, 256, None, None, 256)
    for batch, N, cf, cn in ((1, 64, 0.0, 1.0), (1, 64, 1.0, -1.0), (1, 64, float("nan"), 1.0),
                             (0, 64, 1.0, 1.0), (1, 5000, 1.0, 1.0)):
        assert L.dt_adaptive_budget(C.byref(out), batch, N, cf, cn, 256, None) == \
            dt.ERR_INVALID_ARG
