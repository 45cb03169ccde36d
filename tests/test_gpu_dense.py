"""GPU parity of the dense decode path (M <= 8) against the CPU oracle.

Bars: code unpacking and dequantized values bit-exact; outputs within
|err| <= 1e-2 * max(1, |ref|) elementwise (bf16 outputs, fp32 accumulation).
"""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from helpers import bf16_to_f64, dev_bf16, dev_qweight, host_u16

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()
    assert torch.cuda.is_available()


def assert_close(got, ref, what=""):
    ok, max_err, worst = oracle.within_tolerance(got, ref, TOL)
    assert ok, f"{what}: max |err| {max_err:.3g}, worst err/bound {worst:.3g}"


# ---------------------------------------------------------------- a1 / a2
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,K", [(768, 512), (37, 576), (1, 64), (64, 13824)])
def test_unpack_is_bit_exact(bits, N, K):
    w = synth.qweight(7 + N, N, K, bits)
    got = gwa.debug_unpack(dev_qweight(w)).cpu().numpy()
    assert np.array_equal(got, oracle.unpack(w.wq, N, K, bits))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,K", [(768, 512), (37, 576), (128, 5120)])
def test_dequant_is_bit_exact(bits, N, K):
    w = synth.qweight(9 + N, N, K, bits)
    got = gwa.debug_dequant(dev_qweight(w)).cpu().numpy()
    want = oracle.dequant(w.wq, w.scales, w.biases, N, K, bits).astype(
        np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------- a3
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 6, 8])
@pytest.mark.parametrize("N,K", [(768, 512), (259, 576), (1, 64), (45, 13824)])
def test_qmv_affine_matches_oracle(bits, M, N, K):
    w = synth.qweight(100 + N + bits, N, K, bits)
    x = synth.activations(200 + M, M, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w))
    torch.cuda.synchronize()
    ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits)
    assert y.shape == (M, N)
    assert_close(bf16_to_f64(y), ref, f"M={M} N={N} K={K} u{bits}")


def test_qmv_uneven_grid_covers_every_row():
    # N far from a multiple of the rows per CTA / per warp block
    N, K = 4099, 1024
    w = synth.qweight(301, N, K, 4)
    x = synth.activations(302, 1, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w))
    ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, 4)
    assert_close(bf16_to_f64(y), ref, "N=4099")


@pytest.mark.parametrize("bits", [4, 8])
def test_token_counts_agree(bits):
    # one token at a time (streaming kernel), two (streaming), four and eight
    # at once (staged kernel): same results within the output tolerance
    N, K = 512, 2048
    w = synth.qweight(311, N, K, bits)
    dw = dev_qweight(w)
    xh = synth.activations(312, 8, K)
    x = dev_bf16(xh)
    ref = oracle.qmv(xh, w.wq, w.scales, w.biases, N, K, bits)
    runs = {
        8: gwa.qmv_affine(x, dw),
        4: torch.cat([gwa.qmv_affine(x[i:i + 4], dw) for i in (0, 4)]),
        2: torch.cat([gwa.qmv_affine(x[i:i + 2], dw) for i in range(0, 8, 2)]),
        1: torch.cat([gwa.qmv_affine(x[i:i + 1], dw) for i in range(8)]),
    }
    for m, y in runs.items():
        assert_close(bf16_to_f64(y), ref, f"{m} tokens per call")
    # same kernel, same per-row arithmetic: bitwise equal
    y1b = torch.cat([gwa.qmv_affine(x[i:i + 1], dw) for i in range(8)])
    assert torch.equal(runs[1], y1b)


# ---------------------------------------------------------------- a4
def _guarded(rows, cols, sentinel=-12345):
    """A [rows, cols] bf16 view inside a buffer with guard bands both sides."""
    pad = 64
    buf = torch.full((rows * cols + 2 * pad,), sentinel, dtype=torch.int16,
                     device="cuda")
    view = buf[pad:pad + rows * cols].view(torch.bfloat16).view(rows, cols)
    return buf, view, pad


def _check_guards(buf, pad, sentinel=-12345):
    assert torch.all(buf[:pad] == sentinel) and torch.all(buf[-pad:] == sentinel)


@pytest.mark.parametrize("M", [1, 4])
def test_fused_qkv_tiny_config(M):
    K, secs = 512, (512, 128, 128)
    parts = [synth.qweight(synth.seed_for(0, 0, i), n, K, 4)
             for i, n in enumerate(secs)]
    fused = synth.stack_rows(parts)
    x = synth.activations(synth.seed_for(0, 0, 9), M, K)
    guards = [_guarded(M, n) for n in secs]
    outs = gwa.qmv_fused_sections(dev_bf16(x), dev_qweight(fused), secs,
                                  outs=[g[1] for g in guards])
    torch.cuda.synchronize()
    refs = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases, secs,
                                 K, 4)
    ptrs = set()
    for o, r, (buf, _, pad), n in zip(outs, refs, guards, secs):
        assert o.shape == (M, n) and o.is_contiguous()
        assert o.storage_offset() == 64            # its own buffer's start
        ptrs.add(o.data_ptr())
        assert_close(bf16_to_f64(o), r, "tiny qkv")
        _check_guards(buf, pad)
    assert len(ptrs) == 3


def test_fused_qkv_decode_config_full():
    K, secs = 5120, (5120, 1024, 1024)
    parts = [synth.qweight(synth.seed_for(1, 0, i), n, K, 4)
             for i, n in enumerate(secs)]
    fused = synth.stack_rows(parts)
    x = synth.activations(synth.seed_for(1, 0, 9), 1, K)
    q, k, v = gwa.qmv_fused_sections(dev_bf16(x), dev_qweight(fused), secs)
    refs = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases, secs,
                                 K, 4)
    for o, r in zip((q, k, v), refs):
        assert_close(bf16_to_f64(o), r, "qkv 5120")


@pytest.mark.parametrize("bits", [4, 8])
def test_fused_equals_separate_bitwise(bits):
    K, secs = 1024, (384, 64, 64, 7)
    parts = [synth.qweight(400 + i, n, K, bits) for i, n in enumerate(secs)]
    fused = dev_qweight(synth.stack_rows(parts))
    x = dev_bf16(synth.activations(410, 3, K))
    outs = gwa.qmv_fused_sections(x, fused, secs)
    for o, p in zip(outs, parts):
        sep = gwa.qmv_affine(x, dev_qweight(p))
        assert torch.equal(o, sep)


def test_sections_optional_bias():
    K, secs = 256, (96, 32, 32)
    parts = [synth.qweight(420 + i, n, K, 4) for i, n in enumerate(secs)]
    fused = synth.stack_rows(parts)
    x = synth.activations(430, 2, K)
    bias = [synth.activations(431 + i, 1, n)[0] for i, n in enumerate(secs)]
    bias[1] = None
    outs = gwa.qmv_fused_sections(
        dev_bf16(x), dev_qweight(fused), secs,
        out_bias=[dev_bf16(b) if b is not None else None for b in bias])
    refs = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases, secs,
                                 K, 4, out_bias=bias)
    for o, r in zip(outs, refs):
        assert_close(bf16_to_f64(o), r, "sections+bias")


# ---------------------------------------------------------------- a5
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [1, 3, 4, 8])
def test_gate_up_silu_small(bits, M):
    K, I = 576, 333
    w = synth.qweight(500 + bits, 2 * I, K, bits)
    x = synth.activations(510 + M, M, K)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(w))
    ref = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, bits)
    assert h.shape == (M, I)
    assert_close(bf16_to_f64(h), ref, f"gate_up M={M} u{bits}")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_gate_up_silu_config_full(M):
    # M = 1: lane-per-group kernel; 4: streaming kernel; 8: tensor-core
    # kernel, one pass
    K, I = 5120, 13824
    w = synth.stack_rows([synth.qweight(synth.seed_for(2, 0, 0), I, K, 4),
                          synth.qweight(synth.seed_for(2, 0, 1), I, K, 4)])
    x = synth.activations(synth.seed_for(2, 0, 9) + M, M, K)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(w))
    torch.cuda.synchronize()
    ref = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, 4)
    assert_close(bf16_to_f64(h), ref, f"gate_up config M={M}")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [5, 8])
@pytest.mark.parametrize("N,K", [(301, 6144), (1000, 13824), (19, 20480),
                                 (8, 7680)])
def test_rows_split_over_a_cluster(bits, M, N, K):
    # 5..8 tokens on rows longer than 5120 inputs: for u8 the tensor-core
    # decode kernel on clusters of 2 (K = 6144), 3 (7680, 13824) or 4 (20480)
    # CTAs along K, for u4 the streaming kernel in two passes; N ragged
    # against the 8-row stages and the cluster count.  The output sits
    # between guard bands: only rank 0 of a cluster writes.
    w = synth.qweight(400 + N + bits, N, K, bits)
    x = synth.activations(410 + M, M, K)
    buf, y, pad = _guarded(M, N)
    gwa.qmv_affine(dev_bf16(x), dev_qweight(w), y=y)
    torch.cuda.synchronize()
    _check_guards(buf, pad)
    ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits)
    assert_close(bf16_to_f64(y), ref, f"M={M} N={N} K={K} u{bits}")
    # deterministic: the ranks' sums are added in a fixed order
    y2 = gwa.qmv_affine(dev_bf16(x), dev_qweight(w))
    assert torch.equal(y, y2)


@pytest.mark.parametrize("bits", [4, 8])
def test_down_config_full_eight_tokens(bits):
    # the stack's down projection (13824 -> 5120) at 8 tokens (u8: one pass
    # on clusters of three CTAs), against the oracle and two 4-token calls
    N, K = 5120, 13824
    w = synth.qweight(synth.seed_for(3, 0, 3) + bits, N, K, bits)
    xh = synth.activations(synth.seed_for(3, 0, 9), 8, K)
    dw, x = dev_qweight(w), dev_bf16(xh)
    y8 = gwa.qmv_affine(x, dw)
    y4 = torch.cat([gwa.qmv_affine(x[i:i + 4], dw) for i in (0, 4)])
    torch.cuda.synchronize()
    ref = oracle.qmv(xh, w.wq, w.scales, w.biases, N, K, bits)
    assert_close(bf16_to_f64(y8), ref, f"down M=8 u{bits}")
    assert_close(bf16_to_f64(y4), ref, f"down 2x4 tokens u{bits}")


# ---------------------------------------------------------------- edges
def test_empty_inputs_are_no_ops():
    w = dev_qweight(synth.qweight(600, 16, 128, 4))
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    y = gwa.qmv_affine(x, w)
    assert y.shape == (0, 16)


def test_bad_arguments_raise_status_not_fault():
    w = dev_qweight(synth.qweight(601, 16, 128, 4))
    x = dev_bf16(synth.activations(602, 1, 128))
    bad = gwa.QWeight(w.wq, w.scales, w.biases, 16, 128, 5, 64)
    with pytest.raises(gwa.GwaError) as e:
        gwa.qmv_affine(x, bad)
    assert e.value.code == gwa.GWA_ERR_UNSUPPORTED
    xs = torch.empty(130, dtype=torch.bfloat16, device="cuda")[1:129]
    with pytest.raises(gwa.GwaError) as e:
        gwa.qmv_affine(xs.view(1, 128), w)
    assert e.value.code == gwa.GWA_ERR_MISALIGNED
    torch.cuda.synchronize()          # the context is still healthy
    assert gwa.qmv_affine(x, w).shape == (1, 16)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [1, 3, 5, 8])
def test_sections_bias_streaming_kernels(bits, M):
    # K = 1024: the one-token lane-per-group kernel (M = 1), the chunk
    # streaming kernel (M = 3) and the tensor-core kernel (M = 5, 8; ragged
    # last stage), ragged section sizes, optional biases
    K, secs = 1024, (200, 56, 56, 9)
    parts = [synth.qweight(440 + i + bits, n, K, bits)
             for i, n in enumerate(secs)]
    fused = synth.stack_rows(parts)
    x = synth.activations(450 + M, M, K)
    bias = [synth.activations(451 + i, 1, n)[0] for i, n in enumerate(secs)]
    bias[2] = None
    outs = gwa.qmv_fused_sections(
        dev_bf16(x), dev_qweight(fused), secs,
        out_bias=[dev_bf16(b) if b is not None else None for b in bias])
    refs = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases, secs,
                                 K, bits, out_bias=bias)
    for o, r in zip(outs, refs):
        assert_close(bf16_to_f64(o), r, f"sections+bias M={M} u{bits}")


@pytest.mark.parametrize("bits", [4, 8])
def test_gate_up_lane_per_group_kernel(bits):
    # K = 1536 (24 groups: two 16-lane slices per row, one partly idle),
    # I off every stage size
    K, I = 1536, 777
    w = synth.qweight(520 + bits, 2 * I, K, bits)
    x = synth.activations(530, 1, K)
    h = gwa.qmv_gate_up_silu(dev_bf16(x), dev_qweight(w))
    ref = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, bits)
    assert_close(bf16_to_f64(h), ref, f"gate_up lane-per-group u{bits}")


# One-token shares one stage longer than the shared-memory ring: 152 CTAs
# of 33 or 34 rows (u4, K = 5120: four stages of eight rows plus a short
# slot) or of 17 or 18 rows (u8: two stages plus a short slot).  Rows past
# the end of the short stage must neither be stored nor read out of it.
@pytest.mark.parametrize("bits,N", [(4, 5000), (4, 5120), (8, 2600)])
def test_one_token_short_last_slot(bits, N):
    K = 5120
    w = synth.qweight(600 + N + bits, N, K, bits)
    x = synth.activations(610 + bits, 1, K)
    y = gwa.qmv_affine(dev_bf16(x), dev_qweight(w))
    ref = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits)
    assert_close(bf16_to_f64(y), ref, f"short slot N={N} u{bits}")


def test_one_token_short_last_slot_sections():
    K, secs = 5120, (4096, 512, 512)
    parts = [synth.qweight(620 + i, n, K, 4) for i, n in enumerate(secs)]
    fused = synth.stack_rows(parts)
    bias = [synth.activations(630 + i, 1, n)[0] for i, n in enumerate(secs)]
    x = synth.activations(640, 1, K)
    outs = gwa.qmv_fused_sections(dev_bf16(x), dev_qweight(fused), secs,
                                  out_bias=[dev_bf16(b) for b in bias])
    refs = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases, secs,
                                 K, 4, out_bias=bias)
    for o, r in zip(outs, refs):
        assert_close(bf16_to_f64(o), r, "short slot sections")
