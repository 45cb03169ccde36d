"""GPU parity of the prefill-shaped path (M > 8, tcgen05 tensor cores)
against the CPU oracle, on ragged shapes and on sampled rows of the 48-layer
stack's projection shapes at M = 512."""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from bars import assert_within, tc_accumulation_bar, tc_swiglu_bar
from helpers import bf16_to_f64, dev_bf16, dev_qweight

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()


def assert_close(got, ref, what=""):
    ok, max_err, worst = oracle.within_tolerance(got, ref, TOL)
    assert ok, f"{what}: max |err| {max_err:.3g}, worst err/bound {worst:.3g}"


def status_of(ws):
    return int(ws[:4].view(torch.int32).item())


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [9, 16, 128, 130, 300])
@pytest.mark.parametrize("N,K", [(384, 512), (300, 1024), (256, 576)])
def test_qmm_affine_matches_oracle(bits, M, N, K):
    w = synth.qweight(1300 + N + bits, N, K, bits)
    x = synth.activations(1400 + M, M, K)
    ws = gwa.make_workspace(M, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w), workspace=ws)
    torch.cuda.synchronize()
    assert status_of(ws) == 0
    ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits)
    assert_close(bf16_to_f64(y), ref, f"M={M} N={N} K={K} u{bits}")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [16, 200])
def test_qmm_sections_and_bias(bits, M):
    K, secs = 1024, (256, 64, 64, 40)
    parts = [synth.qweight(1500 + i, n, K, bits) for i, n in enumerate(secs)]
    fused = synth.stack_rows(parts)
    x = synth.activations(1510 + M, M, K)
    bias = [synth.activations(1520 + i, 1, n)[0] for i, n in enumerate(secs)]
    bias[2] = None
    outs = gwa.qmv_fused_sections(
        dev_bf16(x), dev_qweight(fused), secs,
        out_bias=[dev_bf16(b) if b is not None else None for b in bias])
    refs = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases, secs,
                                 K, bits, out_bias=bias)
    for o, r in zip(outs, refs):
        assert o.is_contiguous() and o.storage_offset() == 0
        assert_close(bf16_to_f64(o), r, "qmm sections")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [16, 129])
@pytest.mark.parametrize("K,I", [(576, 200), (1024, 200), (2048, 65)])
def test_qmm_gate_up_silu(bits, M, K, I):
    # K = 576: decode kernels in token passes; K = 1024 / 2048: tensor cores
    # (64-pair tiles, the last one partial)
    w = synth.qweight(1600 + bits, 2 * I, K, bits)
    x = synth.activations(1610 + M, M, K)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(w))
    ref = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, bits)
    _, bar = tc_swiglu_bar(x, w, I)
    assert_within(bf16_to_f64(h), ref, bar, f"qmm gate_up M={M} u{bits}")


# Few tiles for the GPU: the kernel splits each tile's K blocks over a
# cluster of up to 4 CTAs (rank 0 adds the others' partial sums through
# distributed shared memory).  With K = 5120 (84 K blocks) or 13824 and at
# most a handful of 128-row tiles, every shape below fits one wave of
# 4-CTA clusters on a 152-SM GPU, so it takes the split.
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [16, 300])
@pytest.mark.parametrize("mode", ["plain", "sections", "gate_up"])
def test_qmm_cluster_k_split(bits, M, mode):
    K = 5120
    x = synth.activations(1700 + M, M, K)
    if mode == "plain":
        N = 200  # two tiles, the last one partial
        w = synth.qweight(1710 + bits, N, K, bits)
        y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w))
        ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits)
        assert_close(bf16_to_f64(y), ref, f"split plain M={M} u{bits}")
    elif mode == "sections":
        secs = (128, 64, 72)
        parts = [synth.qweight(1720 + i, n, K, bits) for i, n in enumerate(secs)]
        fused = synth.stack_rows(parts)
        bias = [synth.activations(1730 + i, 1, n)[0] for i, n in enumerate(secs)]
        outs = gwa.qmv_fused_sections(dev_bf16(x), dev_qweight(fused), secs,
                                      out_bias=[dev_bf16(b) for b in bias])
        refs = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases,
                                     secs, K, bits, out_bias=bias)
        for o, r in zip(outs, refs):
            assert_close(bf16_to_f64(o), r, f"split sections M={M} u{bits}")
    else:
        I = 100  # two 64-pair tiles
        w = synth.qweight(1740 + bits, 2 * I, K, bits)
        h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(w))
        ref = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, bits)
        # where g or u cancels (u8 sums of ~6000 in magnitude reaching 0.01)
        # its fp32 rounding moves h by more than 1e-2 |h|: the SwiGLU bar
        href, bar = tc_swiglu_bar(x, w, I)
        assert np.allclose(href, ref, rtol=1e-9, atol=1e-12)
        assert_within(bf16_to_f64(h), ref, bar, f"split gate_up M={M} u{bits}")


@pytest.mark.parametrize("bits", [4, 8])
def test_qmm_cluster_k_split_long_rows(bits):
    # one 128-row tile of a down projection's input width: four ranks of
    # 7-8 runs of 8 K blocks each, the bias blocks on the last
    M, N, K = 16, 128, 13824
    w = synth.qweight(1750 + bits, N, K, bits)
    x = synth.activations(1751, M, K)
    ws = gwa.make_workspace(M, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w), workspace=ws)
    torch.cuda.synchronize()
    assert status_of(ws) == 0
    ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits)
    assert_close(bf16_to_f64(y), ref, f"split long rows u{bits}")


def test_tensor_core_and_decode_paths_agree():
    # the first 8 tokens through the decode kernel and all 16 through the
    # tensor-core kernel
    N, K = 512, 2048
    w = dev_qweight(synth.qweight(1700, N, K, 4))
    x = dev_bf16(synth.activations(1701, 16, K))
    y16 = gwa.qmv_affine(x, w)
    y8 = gwa.qmv_affine(x[:8], w)
    assert_close(bf16_to_f64(y16[:8]), bf16_to_f64(y8), "tc vs decode")


@pytest.mark.parametrize("name,rows,K,cols", [
    ("qkv", 7168, 5120, None), ("down", 5120, 13824, None),
    ("gate_up", 27648, 5120, [0, 1, 127, 128, 5000, 13823])])
def test_stack_shapes_at_prefill_size(name, rows, K, cols):
    # the 48-layer stack's projections at M = 512 (layer 0 recipe, drawn on
    # the host), checked on sampled outputs the oracle computes one by one
    M = 512
    w = synth.qweight(synth.stack_seed(0, 0, 4) + rows, rows, K, 4)
    x = synth.activations(1800 + rows, M, K)
    dw = dev_qweight(w)
    if name == "gate_up":
        h = gwa.qmv_gate_up_silu(dev_bf16(x), dw)
        ref = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, rows, K, 4,
                                  cols=cols)
        got = bf16_to_f64(h)[:, cols]
    else:
        y = gwa.qmv_affine(dev_bf16(x), dw)
        sample = [0, 1, 127, 128, 255, 256, rows // 2, rows - 1]
        ref = oracle.qmv(x, w.wq, w.scales, w.biases, rows, K, 4, rows=sample)
        got = bf16_to_f64(y)[:, sample]
    assert_close(got, ref, f"{name} M=512")


def test_missing_workspace_is_an_error_not_a_fault():
    w = dev_qweight(synth.qweight(1900, 64, 128, 4))
    x = dev_bf16(synth.activations(1901, 32, 128))
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(gwa.GwaError) as e:
        gwa.qmv_affine(x, w, workspace=small)
    assert e.value.code == gwa.GWA_ERR_WORKSPACE
    torch.cuda.synchronize()


def scaled_weight(seed, N, K, bits, scale, bias_abs):
    """Codes as drawn; bf16 scales scale * U(1, 2), biases +-bias_abs * U(1, 2)
    (or the recipe's -8 scale + N(0, 1e-3) scaled with the scale when
    bias_abs is None)."""
    w = synth.qweight(seed, N, K, bits)
    rng = synth.rng_for(seed + 1)
    G = K // 64
    s = synth.bf16_bits((scale * rng.uniform(1, 2, (N, G))).astype(np.float32))
    if bias_abs is None:
        b = synth.bf16_bits((-8.0 * synth.bf16_values(s)
                             + scale * 0.1 * rng.standard_normal((N, G))).astype(np.float32))
    else:
        sign = np.where(rng.random((N, G)) < 0.5, -1.0, 1.0)
        b = synth.bf16_bits((sign * bias_abs * rng.uniform(1, 2, (N, G))).astype(np.float32))
    return synth.QWeight(w.wq, s, b, N, K, bits)


def assert_close_acc(got, ref, x, w, rows, what=""):
    """The output bar plus the fp32 accumulation's own rounding (bars.py)."""
    assert_within(got, ref, tc_accumulation_bar(ref, x, w, rows), what)


# Values far outside fp16's range (2^-14 .. 65504): every token and weight
# row is scaled by a power of two before the fp16 conversion, so these are as
# exact as ordinary ones.  K = 1024: the tensor-core kernel.
@pytest.mark.parametrize("M", [16, 512])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("scale,bias_abs,xmul", [
    (1e-6, None, 1.0),     # scales below fp16's normal range
    (1e3, None, 1.0),      # s * (q - 8) beyond 65504
    (0.01, 1e5, 1.0),      # |bias| far beyond 65504
    (0.01, None, 1e6),     # |x| = 1e6 scale
    (1e-6, 1e-3, 1e-30),   # tiny everything
    (1e3, 1e5, 1e6),       # large everything
])
def test_qmm_exact_outside_fp16_range(M, bits, scale, bias_abs, xmul):
    N, K = 256, 1024
    w = scaled_weight(1910 + bits, N, K, bits, scale, bias_abs)
    xv = synth.bf16_values(synth.activations(1911 + M, M, K)).astype(np.float32)
    x = synth.bf16_bits(xv * np.float32(xmul))
    ws = gwa.make_workspace(M, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w), workspace=ws)
    torch.cuda.synchronize()
    assert status_of(ws) == 0
    sample = list(range(0, N, 7)) + [N - 1]
    ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits, rows=sample)
    assert_close_acc(bf16_to_f64(y)[:, sample], ref, x, w, sample,
                     f"M={M} u{bits} scale={scale} bias={bias_abs} x*{xmul}")


def test_qmm_exact_outliers_and_mixed_rows():
    # one token with a 1e6 outlier, rows whose scales differ by 1e9
    M, N, K = 32, 256, 2048
    w = synth.qweight(1930, N, K, 4)
    s = synth.bf16_values(w.scales).copy()
    s[::2] *= np.float32(1e-5)
    s[1::4] *= np.float32(1e4)
    sb = synth.bf16_bits(s)
    bb = synth.bf16_bits(-8.0 * synth.bf16_values(sb))
    w = synth.QWeight(w.wq, sb, bb, N, K, 4)
    x = synth.activations(1931, M, K)
    x[3, 5] = synth.bf16_bits(np.array([1.0e6], np.float32))[0]
    ws = gwa.make_workspace(M, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w), workspace=ws)
    torch.cuda.synchronize()
    assert status_of(ws) == 0
    ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, 4)
    assert_close_acc(bf16_to_f64(y), ref, x, w, list(range(N)),
                     "outliers and mixed rows")
    assert gwa.pipeline_status() == 0
