"""GPU parity of the fused QKV projection with the rotary embedding of Q and
K ("The Cathedral Doubled Itself", "The kernel that worked and the kernel
that won't"; textbook rotate-half RoPE, see the oracle) against the oracle.

One token runs the projection and the rotation in one kernel (rotated in
the epilogue); other token counts run the projection and a rotation kernel.
Both must match the oracle within |err| <= 1e-2 * max(1, |ref|); at one
token V is the plain fused-sections output, bit for bit.
"""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from helpers import dev_bf16, dev_qweight

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()
    assert torch.cuda.is_available()


def run_case(M, q_size, kv_size, K, d, bits, base, positions, bias=False,
             seed=0):
    N = q_size + 2 * kv_size
    w = synth.qweight(9000 + seed, N, K, bits)
    x = synth.activations(9100 + seed, M, K)
    rng = np.random.default_rng(seed)
    biases = None
    if bias:
        biases = [synth.bf16_bits(rng.normal(0, 0.5, size=s).astype(np.float32))
                  for s in (q_size, kv_size, kv_size)]
    pos = np.asarray(positions, dtype=np.int32)
    dw = dev_qweight(w)
    got = gwa.qmv_qkv_rope(
        dev_bf16(x), dw, q_size, kv_size, d, base,
        torch.from_numpy(pos).cuda(),
        out_bias=[dev_bf16(b) for b in biases] if bias else None)
    plain = gwa.qmv_fused_sections(
        dev_bf16(x), dw, [q_size, kv_size, kv_size],
        out_bias=[dev_bf16(b) for b in biases] if bias else None)
    torch.cuda.synchronize()
    ref = oracle.qkv_rope(x, w.wq, w.scales, w.biases, q_size, kv_size, K,
                          bits, d, base, pos, out_bias=biases)
    for name, g, r in zip("QKV", got, ref):
        ok, max_err, worst = oracle.within_tolerance(
            g.float().cpu().numpy().astype(np.float64), r, TOL)
        assert ok, f"{name}: max |err| {max_err:.3g}, worst {worst:.3g}"
    if M == 1:
        # the one-token kernel's V is the plain one-token projection
        assert torch.equal(got[2], plain[2]), "V differs from the plain projection"
    return got, plain


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("pos", [0, 1, 4095, 32767, 131071])
def test_one_token_rotates_in_the_epilogue(bits, pos):
    # the decode shape: Q 5120 + K 1024 + V 1024 over K = 5120, heads of 128
    run_case(1, 5120, 1024, 5120, 128, bits, 1e6, [pos], seed=pos % 7)


@pytest.mark.parametrize("d", [64, 80, 128])
def test_head_widths_and_bias(d):
    run_case(1, 8 * d, 2 * d, 1024, d, 4, 1e4, [77], bias=True, seed=d)


def test_tiny_qkv():
    # the tiny fused-QKV workload: 512 -> Q 512 + K 128 + V 128, heads of 64
    run_case(1, 512, 128, 512, 64, 4, 1e4, [5], seed=1)


@pytest.mark.parametrize("M", [2, 4, 8])
def test_decode_batches_rotate_after_the_projection(M):
    run_case(M, 2048, 512, 2048, 128, 4, 1e6, list(range(100, 100 + M)),
             seed=M)


@pytest.mark.parametrize("M", [9, 16, 64])
def test_prefill_rotates_after_the_projection(M):
    pos = np.arange(M) * 37 + 1000
    run_case(M, 2048, 512, 1024, 128, 4, 1e6, pos, bias=True, seed=M)


def test_positions_per_token_are_used():
    got, plain = run_case(2, 256, 128, 512, 64, 4, 1e4, [0, 900], seed=3)
    # position 0 is the identity: token 0's Q equals the plain projection
    assert torch.equal(got[0][0], plain[0][0])
    assert not torch.equal(got[0][1], plain[0][1])


@pytest.mark.parametrize("M,d,bits", [(33, 64, 4), (300, 128, 4), (40, 128, 8),
                                      (24, 256, 4)])
def test_prefill_head_widths(M, d, bits):
    # heads dividing 128 rotate in the tensor-core epilogue (300 tokens:
    # 256-token tiles); heads of 256 take the staged kernels
    pos = np.arange(M) * 13 + 7
    run_case(M, 1024, 256, 512, d, bits, 1e4, pos, seed=M + d)
