"""The kernels' bounded pipeline waits, made to run out on purpose.

Every wait on a shared-memory pipeline barrier in the decode and tensor-core
kernels gives up after a time limit (2 s) instead of spinning forever, so a
broken pipeline costs one failed call, not a hung GPU.  Here a test kernel
waits on a barrier that nothing completes, with a short limit, through both
forms of the wait; the test checks that each wait reports failure after
about the limit, that the GPU is still usable (a projection afterwards
matches the oracle), and that the production timeout counters saw nothing.
"""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from helpers import bf16_to_f64, dev_bf16, dev_qweight

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()


@pytest.mark.parametrize("limit_us", [2000, 20000])
def test_wait_gives_up_after_its_limit(limit_us):
    gwa.pipeline_status(reset=True)
    out = gwa.debug_bounded_wait(limit_us)
    torch.cuda.synchronize()
    gave_up_plain, waited_plain, gave_up_sleep, waited_sleep = out.cpu().tolist()
    assert gave_up_plain == 1 and gave_up_sleep == 1
    for waited in (waited_plain, waited_sleep):
        # at least the limit; well under the production limit of 2 s
        assert limit_us <= waited < limit_us + 500000, waited
    # the context is still usable and the production counters are untouched
    w = synth.qweight(2500, 256, 1024, 4)
    x = synth.activations(2501, 1, 1024)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w))
    torch.cuda.synchronize()
    ok, err, worst = oracle.within_tolerance(
        bf16_to_f64(y), oracle.qmv(x, w.wq, w.scales, w.biases, 256, 1024, 4),
        1e-2)
    assert ok, f"max |err| {err:.3g}"
    assert gwa.pipeline_status(reset=True) == 0


def test_wait_limit_is_checked_on_the_host():
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    lib = gwa.load()
    assert lib.gwa_debug_bounded_wait(0, out.data_ptr(), None) == gwa.GWA_ERR_INVALID_ARG
    assert lib.gwa_debug_bounded_wait(3000000, out.data_ptr(), None) == gwa.GWA_ERR_INVALID_ARG
    assert lib.gwa_debug_bounded_wait(1000, None, None) == gwa.GWA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [0, 0, 0, 0]
