"""GPU parity of the code widths and group sizes outside the tuned kernels
(u2, u3, u6, and groups of 32 and 128 at every width), which run on the
general-format decode kernel (one token of u4 / u8 in groups of 32 or 128:
on the one-token chunk kernel), against the oracle (same packed format: a
row's words are one little-endian bit stream, code k at bits [b*k, +b),
lowest bits first, so u3 and u6 codes straddle words; one bf16 scale and
bias per group; "saragossa", "Quantization formats").

Bars as for the tuned formats: unpacked codes and dequantized values bit
for bit; outputs within |err| <= 1e-2 * max(1, |ref|).
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
FORMATS = [(2, 32), (2, 64), (2, 128), (4, 32), (4, 128), (8, 32), (8, 128),
           (3, 32), (3, 64), (3, 128), (6, 32), (6, 64), (6, 128)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()
    assert torch.cuda.is_available()


def close(got, ref, what=""):
    ok, max_err, worst = oracle.within_tolerance(
        got.float().cpu().numpy().astype(np.float64), ref, TOL)
    assert ok, f"{what}: max |err| {max_err:.3g}, worst {worst:.3g}"


@pytest.mark.parametrize("bits,group", FORMATS)
def test_unpack_and_dequant_bit_exact(bits, group):
    N, K = 37, 512
    w = synth.qweight(3 + bits + group, N, K, bits, group)
    dw = dev_qweight(w)
    codes = gwa.debug_unpack(dw).cpu().numpy()
    assert np.array_equal(codes, oracle.unpack(w.wq, N, K, bits))
    wf = gwa.debug_dequant(dw).cpu().numpy().astype(np.float64)
    ref = oracle.dequant(w.wq, w.scales, w.biases, N, K, bits, group)
    assert np.array_equal(wf, ref.astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("bits,group", FORMATS)
@pytest.mark.parametrize("M", [1, 3, 8, 11])
def test_plain_projection(bits, group, M):
    N, K = 300, 1024
    w = synth.qweight(100 + bits + group, N, K, bits, group)
    x = synth.activations(200 + M, M, K)
    ws = gwa.make_workspace(M, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w), workspace=ws)
    torch.cuda.synchronize()
    close(y, oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits, group),
          f"u{bits} g{group} M={M}")


@pytest.mark.parametrize("bits,group", [(2, 32), (4, 128), (8, 32), (3, 64),
                                        (6, 64)])
def test_sections_gate_up_and_rope(bits, group):
    K, M = 512, 2
    rng = np.random.default_rng(bits + group)
    # sections with bias
    sizes = [256, 64, 64]
    w = synth.qweight(300 + group, sum(sizes), K, bits, group)
    x = synth.activations(301, M, K)
    bias = [synth.bf16_bits(rng.normal(0, 0.5, size=s).astype(np.float32))
            for s in sizes]
    dw = dev_qweight(w)
    outs = gwa.qmv_fused_sections(dev_bf16(x), dw, sizes,
                                  out_bias=[dev_bf16(b) for b in bias])
    refs = oracle.fused_sections(x, w.wq, w.scales, w.biases, sizes, K, bits,
                                 group=group, out_bias=bias)
    for o, r in zip(outs, refs):
        close(o, r, "sections")
    # gate+up SwiGLU
    g = synth.qweight(302 + group, 2 * 160, K, bits, group)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(g))
    close(h, oracle.gate_up_silu(x, g.wq, g.scales, g.biases, 2 * 160, K, bits,
                                 group=group), "gate+up")
    # QKV with the rotary embedding (heads of 64), one token and three
    for m in (1, 3):
        xm = synth.activations(303 + m, m, K)
        pos = np.arange(m, dtype=np.int32) + 40
        got = gwa.qmv_qkv_rope(dev_bf16(xm), dw, 256, 64, 64, 1e4,
                               torch.from_numpy(pos).cuda())
        ref = oracle.qkv_rope(xm, w.wq, w.scales, w.biases, 256, 64, K, bits,
                              64, 1e4, pos, group=group)
        for o, r in zip(got, ref):
            close(o, r, f"rope M={m}")
    torch.cuda.synchronize()


@pytest.mark.parametrize("bits,group,K", [(3, 64, 13824), (6, 128, 13824),
                                          (2, 32, 32768), (3, 64, 32768),
                                          (6, 64, 32768)])
def test_long_rows(bits, group, K):
    """K = 13824 at four tokens keeps the integer-dot kernel with ~120 KB of
    encoded activations per block; K = 32768 at four tokens exceeds its
    shared memory and runs the fp32 kernel.  Plain and gate+up."""
    M, N = 4, 40
    w = synth.qweight(700 + bits + group, N, K, bits, group)
    x = synth.activations(701, M, K)
    ws = gwa.make_workspace(M, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w), workspace=ws)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(w), workspace=ws)
    torch.cuda.synchronize()
    close(y, oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits, group),
          f"u{bits} g{group} K={K}")
    close(h, oracle.gate_up_silu(x, w.wq, w.scales, w.biases, N, K, bits,
                                 group=group), f"gate+up u{bits} K={K}")


@pytest.mark.parametrize("bits", [3, 6])
def test_gate_up_full_shape_sampled(bits):
    """The 27648 x 5120 gate+up weight at one token, the launch the formats
    bench times: 512 sampled outputs against the oracle."""
    K, I = 5120, 13824
    w = synth.qweight(900 + bits, 2 * I, K, bits, 64)
    x = synth.activations(901, 1, K)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(w))
    torch.cuda.synchronize()
    cols = np.random.default_rng(bits).choice(I, size=512, replace=False)
    ref = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, bits,
                              group=64, cols=cols)
    close(h[:, torch.from_numpy(cols).cuda()], ref, f"u{bits} full shape")


# One token of u4 / u8 codes in groups of 32 or 128: the chunk-per-lane
# kernel (a lane owns 64 inputs: half a group of 128, or two groups of 32
# with a dot per half) wherever the scale rows are whole 16-byte units;
# K = 13824 at groups of 128 (108 groups a row) takes the general kernel.
ONE_TOKEN = [(4, 32), (4, 128), (8, 32), (8, 128)]


@pytest.mark.parametrize("bits,group", ONE_TOKEN)
@pytest.mark.parametrize("N,K", [(777, 2048), (5120, 5120), (45, 13824)])
def test_one_token_chunk_kernel(bits, group, N, K):
    w = synth.qweight(800 + bits + group + N, N, K, bits, group)
    x = synth.activations(801 + K, 1, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w))
    torch.cuda.synchronize()
    close(y, oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits, group),
          f"u{bits} g{group} N={N} K={K}")


@pytest.mark.parametrize("bits,group", ONE_TOKEN)
def test_one_token_chunk_kernel_fused(bits, group):
    """Sections with biases, gate+up SiLU and QKV with the rotary embedding
    (heads of 64) at one token."""
    K = 2048
    rng = np.random.default_rng(810 + bits + group)
    sizes = [512, 128, 128]
    w = synth.qweight(811 + group, sum(sizes), K, bits, group)
    x = synth.activations(812, 1, K)
    bias = [synth.bf16_bits(rng.normal(0, 0.5, size=s).astype(np.float32))
            for s in sizes]
    dw = dev_qweight(w)
    outs = gwa.qmv_fused_sections(dev_bf16(x), dw, sizes,
                                  out_bias=[dev_bf16(b) for b in bias])
    refs = oracle.fused_sections(x, w.wq, w.scales, w.biases, sizes, K, bits,
                                 group=group, out_bias=bias)
    for o, r in zip(outs, refs):
        close(o, r, "sections")
    g = synth.qweight(813 + group, 2 * 333, K, bits, group)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(g))
    close(h, oracle.gate_up_silu(x, g.wq, g.scales, g.biases, 2 * 333, K, bits,
                                 group=group), "gate+up")
    pos = np.array([77], dtype=np.int32)
    got = gwa.qmv_qkv_rope(dev_bf16(x), dw, 512, 128, 64, 1e4,
                           torch.from_numpy(pos).cuda())
    ref = oracle.qkv_rope(x, w.wq, w.scales, w.biases, 512, 128, K, bits, 64,
                          1e4, pos, group=group)
    for o, r in zip(got, ref):
        close(o, r, "rope")
    torch.cuda.synchronize()


@pytest.mark.parametrize("bits,group", [(4, 32), (4, 128)])
def test_one_token_chunk_kernel_full_shape_sampled(bits, group):
    """The 27648 x 5120 gate+up weight at one token, the launch the formats
    bench times: 512 sampled outputs against the oracle."""
    K, I = 5120, 13824
    w = synth.qweight(820 + group, 2 * I, K, bits, group)
    x = synth.activations(821, 1, K)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(w))
    torch.cuda.synchronize()
    cols = np.random.default_rng(group).choice(I, size=512, replace=False)
    ref = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, bits,
                              group=group, cols=cols)
    close(h[:, torch.from_numpy(cols).cuda()], ref, f"u{bits} g{group} full")
