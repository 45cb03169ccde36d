"""Pins of the oracle's fp8 (e4m3) weights, independent of its C code.

The format is read from "saragossa", "Quantization formats" (fp8 (e4m3)
among the formats the loader takes, with the u8 footprint): e4m3 codes in the
affine container, w = scale * e4m3(q) + bias.  The value of a code is the OCP
FP8 E4M3 number of its byte: sign bit 7, exponent bits 6..3 with bias 7,
mantissa bits 2..0; exponent 0 gives the subnormals m/8 * 2^-6; exponent 15
with mantissa 7 is NaN; there are no infinities.  Here every one of the 256
codes is decoded again from its bit string with exact rationals, and a few are
checked against hand-written values."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import gwa_synth as synth
import oracle

FP8 = oracle.FP8_E4M3
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def decode(byte):
    """E4M3 from the bit string; None for NaN."""
    bits = format(byte, "08b")
    sign, exp, man = bits[0], int(bits[1:5], 2), int(bits[5:], 2)
    if exp == 15 and man == 7:
        return None
    if exp == 0:
        v = Fraction(man, 8) * Fraction(1, 2 ** 6)
    else:
        v = (1 + Fraction(man, 8)) * Fraction(2) ** (exp - 7)
    return -v if sign == "1" else v


def test_every_code_matches_its_bit_string():
    for b in range(256):
        want = decode(b)
        got = oracle.e4m3_value(b)
        if want is None:
            assert math.isnan(got), hex(b)
        else:
            assert got == float(want), hex(b)
            assert Fraction(got) == want  # exact, not rounded
            if want == 0:
                assert math.copysign(1.0, got) == (-1.0 if b & 0x80 else 1.0)


@pytest.mark.parametrize("byte,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x3F, 1.875), (0x40, 2.0), (0x77, 240.0), (0x7E, 448.0),
    (0xB8, -1.0), (0xFE, -448.0), (0x81, -(2.0 ** -9))])
def test_hand_written_values(byte, value):
    assert oracle.e4m3_value(byte) == value


def test_nan_codes_and_range():
    assert math.isnan(oracle.e4m3_value(0x7F))
    assert math.isnan(oracle.e4m3_value(0xFF))
    pos = [oracle.e4m3_value(b) for b in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))       # monotone, no gaps
    assert max(pos) == 448.0 and pos[1] == 2.0 ** -9
    finite = [oracle.e4m3_value(b) for b in range(256)
              if not math.isnan(oracle.e4m3_value(b))]
    assert len(finite) == 254


def test_unpack_reads_bytes_lowest_first():
    words = np.array([[0x7E01B838, 0x00FF3F40]], dtype=np.uint32)
    codes = oracle.unpack(words, 1, 8, FP8)
    assert codes.tolist() == [[0x38, 0xB8, 0x01, 0x7E, 0x40, 0x3F, 0xFF, 0x00]]


def test_dequant_is_scale_times_value_plus_bias():
    rng = np.random.default_rng(5)
    N, K = 3, 128
    codes = rng.integers(0, 256, (N, K), dtype=np.uint32)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    wq = (codes.reshape(N, K // 4, 4) << np.array([0, 8, 16, 24], np.uint32)).sum(
        axis=2, dtype=np.uint64).astype(np.uint32)
    s = synth.bf16_bits(rng.uniform(0.5, 2.0, (N, 2)).astype(np.float32))
    b = synth.bf16_bits(rng.normal(0, 1, (N, 2)).astype(np.float32))
    unit = oracle.dequant(wq, np.full((N, 2), 0x3F80, np.uint16),
                          np.zeros((N, 2), np.uint16), N, K, FP8)
    w = oracle.dequant(wq, s, b, N, K, FP8)
    sv, bv = synth.bf16_values(s), synth.bf16_values(b)
    for n in range(N):
        for k in range(K):
            v = decode(int(codes[n, k]))
            assert Fraction(unit[n, k]) == v
            exact = Fraction(float(sv[n, k // 64])) * v + Fraction(float(bv[n, k // 64]))
            assert Fraction(w[n, k]) == exact     # exact in fp64 here


def test_qmv_equals_exact_rational_sum():
    rng = np.random.default_rng(6)
    M, N, K = 2, 4, 64
    codes = rng.integers(0, 0x7F, (N, K), dtype=np.uint32) | (
        rng.integers(0, 2, (N, K), dtype=np.uint32) << 7)
    wq = (codes.reshape(N, K // 4, 4) << np.array([0, 8, 16, 24], np.uint32)).sum(
        axis=2, dtype=np.uint64).astype(np.uint32)
    s = synth.bf16_bits(rng.uniform(0.01, 0.1, (N, 1)).astype(np.float32))
    b = synth.bf16_bits(rng.normal(0, 0.01, (N, 1)).astype(np.float32))
    x = synth.activations(7, M, K)
    y = oracle.qmv(x, wq, s, b, N, K, FP8)
    xv, sv, bv = synth.bf16_values(x), synth.bf16_values(s), synth.bf16_values(b)
    for m in range(M):
        for n in range(N):
            acc = sum(Fraction(float(xv[m, k])) *
                      (Fraction(float(sv[n, 0])) * decode(int(codes[n, k])) +
                       Fraction(float(bv[n, 0]))) for k in range(K))
            assert abs(y[m, n] - float(acc)) <= 1e-12 * max(1.0, abs(float(acc)))


def test_footprint_matches_the_printed_one():
    # container bits per weight: 8-bit code + a bf16 scale and bias per 64
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "fp8_footprint.txt"))
            if ln.strip() and not ln.startswith("#")]
    for fmt, params_b, gb in rows:
        code_bits = 8
        bpw = code_bits + 32 / 64
        assert round(float(params_b) * bpw / 8) == int(gb), fmt
    # the alternative reading (an 8-bit scale per 32 codes) would not
    assert round(27 * (8 + 8 / 32) / 8) != 29


def test_other_steps_refuse_fp8():
    with pytest.raises(Exception):
        oracle.quantize_affine(np.zeros((1, 64), np.uint16), 1, 64, FP8)
