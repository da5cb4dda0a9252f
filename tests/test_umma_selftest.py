"""The library's tcgen05 building blocks (dt_umma.cuh) on a single-CTA GEMM.

Compiles tests/cuda/umma_selftest.cu (test-only) against the product header,
runs D = A (sum_s B_s)^T on the tensor cores and compares with float64. The
three-term case is the bf16 split the search uses for its fp32 GRU states.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np
import pytest
import torch

import dt_workloads as W

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    src = os.path.join(HERE, "cuda", "umma_selftest.cu")
    out_dir = os.path.join(HERE, "cuda", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libumma_selftest.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-o", so, src])
    L = C.CDLL(so)
    L.umma_selftest.argtypes = [C.c_void_p] * 3 + [C.c_int] * 3 + [C.c_void_p]
    return L


def split3(x):
    """fp32 -> three bf16 terms whose sum reproduces x to ~24 bits."""
    hi = W.bf16_bits_to_f32(W.f32_to_bf16_bits(x))
    r1 = (x - hi).astype(np.float32)
    mid = W.bf16_bits_to_f32(W.f32_to_bf16_bits(r1))
    lo = (r1 - mid).astype(np.float32)
    return [W.f32_to_bf16_bits(t) for t in (hi, mid, lo)]


@pytest.mark.parametrize("N,K,nsplit", [(16, 16, 1), (64, 64, 1), (256, 128, 1), (128, 64, 3),
                                        (48, 208, 3)])
def test_umma_gemm(lib, N, K, nsplit):
    rng = np.random.default_rng(N * 1000 + K)
    A = W.f32_to_bf16_bits(rng.standard_normal((128, K)).astype(np.float32))
    if nsplit == 1:
        Bs = [W.f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))]
        Bf = W.bf16_bits_to_f32(Bs[0]).astype(np.float64)
    else:
        x = np.tanh(rng.standard_normal((N, K))).astype(np.float32)
        Bs = split3(x)
        Bf = x.astype(np.float64)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(np.stack(Bs).view(np.int16)).cuda()
    dD = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    st = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    assert lib.umma_selftest(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), N, K, nsplit,
                             st.data_ptr()) == 0
    assert int(st.item()) == 0
    ref = W.bf16_bits_to_f32(A).astype(np.float64) @ Bf.T
    got = dD.cpu().numpy()
    err = np.abs(got - ref).max() / max(1.0, np.abs(ref).max())
    assert err < 2e-6, err
