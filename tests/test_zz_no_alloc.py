"""The allocation-free entry point, gwa_qmv_affine_noalloc.

It serves callers that cannot allocate device memory (a plug-in whose host
framework owns all device memory, a serving loop that must not make
allocation calls).  The test calls it through the C ABI and checks it
against gwa_qmv_affine with a caller-provided workspace, on two calls in a
row with different inputs (the built-in scratch keeps the previous call's
contents, which must not leak into the next result).  This file sorts last so
a run that stops at the first failure has run every other test before it.
"""
import ctypes

import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from helpers import bf16_to_f64, dev_bf16, dev_qweight

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def lib():
    gwa.build()
    return gwa.load()


def call_noalloc(lib, x, w, y):
    M = x.numel() // w.K
    rc = lib.gwa_qmv_affine_noalloc(
        x.data_ptr(), M, w.c(), y.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    return rc


@pytest.mark.parametrize("M,N,K", [(64, 384, 512), (300, 256, 1024),
                                   (4, 384, 512)])
def test_noalloc_matches_workspace_entry_point_twice(lib, M, N, K):
    w = dev_qweight(synth.qweight(2100 + N, N, K, 4))
    for call in range(2):                 # two calls in a row, new inputs
        x = dev_bf16(synth.activations(2200 + 10 * M + call, M, K))
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(lib, x, w, y) == gwa.GWA_OK, gwa.last_error()
        ref = gwa.qmv_affine(x, w, workspace=gwa.make_workspace(M, K))
        torch.cuda.synchronize()
        ok, err, worst = oracle.within_tolerance(bf16_to_f64(y),
                                                 bf16_to_f64(ref), TOL)
        assert ok, f"call {call}: max |err| {err:.3g}, worst {worst:.3g}"


def test_noalloc_rejects_problems_larger_than_its_scratch(lib):
    K = 4096
    M = gwa.GWA_NOALLOC_SCRATCH_BYTES // (2 * K) + 64  # more than the scratch
    w = dev_qweight(synth.qweight(2300, 16, K, 4))
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((M, 16), dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(lib, x, w, y) == gwa.GWA_ERR_WORKSPACE
    assert "scratch" in gwa.last_error()
    torch.cuda.synchronize()
