"""GPU parity of fp8 (e4m3) weights against the oracle.

Reading of "saragossa", "Quantization formats" (fp8 (e4m3) beside the affine
widths, with the u8 footprint): E4M3 codes in the affine container, four a
word, lowest byte first, one bf16 scale and bias per group, w = scale *
e4m3(q) + bias.  They run on the general decode kernel in fp32 (every
product of an E4M3 value and a bf16 activation is exact).  Bars: codes and
dequantized values bit for bit; one-hot activations read each dequantized
weight exactly; outputs within 1e-2 * max(1, |ref|) (SwiGLU: plus the
propagated fp32 rounding, as for the other formats).
"""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from helpers import bf16_to_f64, dev_bf16, dev_qweight, host_u16

pytestmark = pytest.mark.gpu
FP8 = gwa.GWA_FP8_E4M3
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert FP8 == synth.FP8_E4M3 == oracle.FP8_E4M3
    gwa.build()
    gwa.load()
    assert torch.cuda.is_available()


def close(got, ref, what=""):
    ok, max_err, worst = oracle.within_tolerance(bf16_to_f64(got), ref, TOL)
    assert ok, f"{what}: max |err| {max_err:.3g}, worst {worst:.3g}"


@pytest.mark.parametrize("group", [32, 64, 128])
def test_unpack_and_dequant_bit_exact(group):
    N, K = 37, 512
    w = synth.qweight(4000 + group, N, K, FP8, group)
    dw = dev_qweight(w)
    codes = gwa.debug_unpack(dw).cpu().numpy()
    assert np.array_equal(codes, oracle.unpack(w.wq, N, K, FP8))
    wf = gwa.debug_dequant(dw).cpu().numpy().astype(np.float64)
    ref = oracle.dequant(w.wq, w.scales, w.biases, N, K, FP8, group)
    assert np.array_equal(wf, ref.astype(np.float32).astype(np.float64))


def test_every_code_value_through_the_projection():
    # one row per code byte (NaN bytes excluded), scale 1, bias 0, a one-hot
    # token: y[n] is the code's E4M3 value rounded to bf16 (exact: 4 bits);
    # the sum that holds it adds +0 terms, so code 0x80 (-0) gives +0
    codes = [c for c in range(256) if (c & 0x7f) != 0x7f]
    N, K = len(codes), 64
    by = np.zeros((N, K), np.uint8)
    by[:, 5] = codes
    wq = by.reshape(N, K // 4, 4).view(np.uint32).reshape(N, K // 4).copy()
    w = synth.QWeight(wq, np.full((N, 1), 0x3F80, np.uint16),
                      np.zeros((N, 1), np.uint16), N, K, FP8, 64)
    x = np.zeros((1, K), np.uint16)
    x[0, 5] = 0x3F80
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w))
    torch.cuda.synchronize()
    want = synth.bf16_bits(np.array([oracle.e4m3_value(c) for c in codes],
                                    np.float32) + np.float32(0.0))
    assert np.array_equal(host_u16(y)[0], want)


@pytest.mark.parametrize("M", [1, 3])
def test_one_hot_reads_dequantized_weights(M):
    N, K = 96, 512
    w = synth.qweight(4100, N, K, FP8, 64)
    deq = oracle.dequant(w.wq, w.scales, w.biases, N, K, FP8, 64)
    dw = dev_qweight(w)
    pos = list(range(64)) + [300, 511]
    for i in range(0, len(pos), M):
        batch = pos[i:i + M]
        x = np.zeros((len(batch), K), np.uint16)
        for m, k in enumerate(batch):
            x[m, k] = 0x3F80
        y = gwa.qmv_affine(dev_bf16(x), dw)
        torch.cuda.synchronize()
        want = synth.bf16_bits(deq[:, batch].T.astype(np.float32))
        assert np.array_equal(host_u16(y), want), batch


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M", [1, 3, 8, 11])
def test_plain_projection(group, M):
    N, K = 300, 1024
    w = synth.qweight(4200 + group, N, K, FP8, group)
    x = synth.activations(4201 + M, M, K)
    ws = gwa.make_workspace(M, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w), workspace=ws)
    torch.cuda.synchronize()
    close(y, oracle.qmv(x, w.wq, w.scales, w.biases, N, K, FP8, group),
          f"fp8 g{group} M={M}")


def test_sections_gate_up_and_rope():
    K, M = 512, 2
    rng = np.random.default_rng(44)
    sizes = [256, 64, 64]
    w = synth.qweight(4300, sum(sizes), K, FP8)
    x = synth.activations(4301, M, K)
    bias = [synth.bf16_bits(rng.normal(0, 0.5, size=s).astype(np.float32))
            for s in sizes]
    dw = dev_qweight(w)
    outs = gwa.qmv_fused_sections(dev_bf16(x), dw, sizes,
                                  out_bias=[dev_bf16(b) for b in bias])
    refs = oracle.fused_sections(x, w.wq, w.scales, w.biases, sizes, K, FP8,
                                 out_bias=bias)
    for o, r in zip(outs, refs):
        close(o, r, "sections")
    g = synth.qweight(4302, 2 * 160, K, FP8)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(g))
    W = oracle.dequant(g.wq, g.scales, g.biases, 320, K, FP8)
    xv = synth.bf16_values(x).astype(np.float64)
    gv, uv = xv @ W[:160].T, xv @ W[160:].T
    # fp32 rounding of g and u: each exact product enters a sequential fp32
    # sum (at most K additions, each off by 2^-24 of a partial sum bounded by
    # sum |w x|), after one rounding of each dequantized weight
    e = (K + 1) * 2.0 ** -24
    eg = e * (np.abs(xv) @ np.abs(W[:160]).T)
    eu = e * (np.abs(xv) @ np.abs(W[160:]).T)
    sig = 1.0 / (1.0 + np.exp(-gv))
    href = gv * sig * uv
    bar = (TOL * np.maximum(1.0, np.abs(href)) +
           np.abs(sig * (1 + gv * (1 - sig)) * uv) * eg + np.abs(gv * sig) * eu)
    assert (np.abs(bf16_to_f64(h) - href) <= bar).all()
    for m in (1, 3):
        xm = synth.activations(4303 + m, m, K)
        pos = np.arange(m, dtype=np.int32) + 40
        got = gwa.qmv_qkv_rope(dev_bf16(xm), dw, 256, 64, 64, 1e4,
                               torch.from_numpy(pos).cuda())
        ref = oracle.qkv_rope(xm, w.wq, w.scales, w.biases, 256, 64, K, FP8,
                              64, 1e4, pos)
        for o, r in zip(got, ref):
            close(o, r, f"rope M={m}")
    torch.cuda.synchronize()


def test_full_gate_up_shape_sampled():
    # 27648 x 5120 at one token, sampled output columns
    I, K = 13824, 5120
    g = synth.qweight(4400, 2 * I, K, FP8)
    x = synth.activations(4401, 1, K)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(g))
    torch.cuda.synchronize()
    cols = list(range(0, I, 97)) + [I - 1]
    ref = oracle.gate_up_silu(x, g.wq, g.scales, g.biases, 2 * I, K, FP8,
                              cols=cols)
    close(h[:, cols], ref, "full gate+up")


def test_other_entry_points_refuse_fp8():
    w = dev_qweight(synth.qweight(4500, 4 * 128, 512, FP8))
    ids = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(gwa.GwaError) as ei:
        gwa.moe_qmv_gather(torch.zeros((1, 512), dtype=torch.bfloat16,
                                       device="cuda"), ids,
                           gwa.expert_view(w, 4), 4, gwa.GWA_MOE_GATE_UP_SILU)
    assert "bits" in str(ei.value)
    with pytest.raises(gwa.GwaError):
        gwa.quantize_affine(torch.zeros((4, 512), dtype=torch.bfloat16,
                                        device="cuda"), bits=FP8)
