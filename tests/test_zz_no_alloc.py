"""The allocation-free entry point, gwa_qmv_affine_noalloc.

Who needs it: code that may not allocate device memory on this path.  A
plug-in running inside a host framework that owns every device allocation
has no allocator of its own to call, and a serving loop cannot afford an
allocation call in the middle of a request, because that call can
synchronize the device or fail when memory is short.  Neither kind of caller
can hand the tensor-core path (more than 8 tokens) a workspace, so this entry
point runs in a scratch buffer that the library keeps in device memory.

What is checked, through the C ABI: on two calls in a row with new inputs
(the scratch keeps the previous call's contents, which must not leak into
the next result) the output equals, bit for bit, gwa_qmv_affine's with a
caller-provided workspace, and it matches the oracle within the output bar;
no pipeline wait ran out (gwa_pipeline_status, which also covers the status
word in the scratch); a problem exactly at the scratch's size limit runs,
and one token more is refused without enqueuing anything.

This file sorts last, so a run that stops at the first failure has run every
other test first; it also passes when run alone in a fresh process.
"""
import numpy as np
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


def largest_fitting_M(K):
    M = 9
    while gwa.workspace_bytes(M + 1, K) <= gwa.GWA_NOALLOC_SCRATCH_BYTES:
        M += 1
    return M


@pytest.mark.parametrize("M,N,K,bits", [(64, 384, 512, 4), (300, 256, 1024, 4),
                                        (33, 128, 2048, 8), (4, 384, 512, 4)])
def test_noalloc_matches_workspace_entry_point_twice(lib, M, N, K, bits):
    hw = synth.qweight(2100 + N + bits, N, K, bits)
    w = dev_qweight(hw)
    gwa.pipeline_status(reset=True)
    for call in range(2):                 # two calls in a row, new inputs
        hx = synth.activations(2200 + 10 * M + call, M, K)
        x = dev_bf16(hx)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(lib, x, w, y) == gwa.GWA_OK, gwa.last_error()
        ref = gwa.qmv_affine(x, w, workspace=gwa.make_workspace(M, K))
        torch.cuda.synchronize()
        assert torch.equal(y, ref), f"call {call}: differs from gwa_qmv_affine"
        rows = list(range(0, N, 5)) + [N - 1]
        want = oracle.qmv(hx, hw.wq, hw.scales, hw.biases, N, K, bits, rows=rows)
        ok, err, worst = oracle.within_tolerance(bf16_to_f64(y)[:, rows], want,
                                                 TOL)
        assert ok, f"call {call}: max |err| {err:.3g}, worst {worst:.3g}"
    assert gwa.pipeline_status(reset=True) == 0


def test_noalloc_at_its_size_limit(lib):
    # a down projection's input width: the largest M that fits runs, one
    # more token is refused before anything is enqueued
    K, N = 13824, 16
    M = largest_fitting_M(K)
    assert gwa.workspace_bytes(M, K) <= gwa.GWA_NOALLOC_SCRATCH_BYTES
    hw = synth.qweight(2400, N, K, 4)
    w = dev_qweight(hw)
    hx = synth.activations(2401, M, K)
    x = dev_bf16(hx)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(lib, x, w, y) == gwa.GWA_OK, gwa.last_error()
    torch.cuda.synchronize()
    toks = [0, 1, M // 2, M - 1]
    want = oracle.qmv(hx[toks], hw.wq, hw.scales, hw.biases, N, K, 4)
    ok, err, worst = oracle.within_tolerance(bf16_to_f64(y)[toks], want, TOL)
    assert ok, f"max |err| {err:.3g}, worst {worst:.3g}"

    x2 = torch.zeros((M + 1, K), dtype=torch.bfloat16, device="cuda")
    y2 = torch.full((M + 1, N), 7.0, dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(lib, x2, w, y2) == gwa.GWA_ERR_WORKSPACE
    assert "scratch" in gwa.last_error()
    torch.cuda.synchronize()
    assert bool((y2 == 7.0).all())       # nothing ran
    assert gwa.pipeline_status(reset=True) == 0
