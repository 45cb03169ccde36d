"""Pins for the oracle's affine quantization (CPU only).

The step is the requantize of "Sanctum-MLX", "The April 2026 cutover" (LoRA
merge at load: dequantize, add the delta, requantize at group size 64).  The
pages give no rounding rule; the oracle takes the plainest reading (per group
scale = bf16((max - min) / (2^b - 1)), bias = min, code = rint((w - bias) /
scale) clamped, in fp32).  Each test below pins it to something other than
itself: a hand-worked group, weights built on an exact grid, the round-trip
error bound, and the degenerate and ordering properties a mistake would
break (truncation instead of rounding, max for min, a reversed bit order, a
scale left unrounded).
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "quantize_worked_example.txt")


def bf16_bits(x):
    """float32 values that are exact in bf16 -> their bit patterns."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def bits_to_f64(h):
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def to_bf16_rn(x):
    """Round float32 to bf16 bit patterns, nearest even (test-side helper)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def read_golden():
    cases, cur = [], None
    for ln in open(GOLDEN):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        key, *vals = ln.split()
        if key == "bits":
            cur = {"bits": int(vals[0])}
            cases.append(cur)
        elif key in ("scale", "bias"):
            cur[key] = int(vals[0], 16)
        elif key == "words":
            cur["words"] = [int(v, 16) for v in vals]
    return cases


@pytest.mark.parametrize("case", read_golden(), ids=lambda c: f"u{c['bits']}")
def test_hand_worked_group(case):
    vals = np.array([1 + 0.5 * (i % 16) for i in range(64)], dtype=np.float32)
    wq, sc, bi = oracle.quantize_affine(bf16_bits(vals)[None, :], 1, 64,
                                        case["bits"])
    assert int(sc[0, 0]) == case["scale"]
    assert int(bi[0, 0]) == case["bias"]
    assert [int(v) for v in wq[0]] == case["words"]


@pytest.mark.parametrize("bits", [4, 8])
def test_grid_weights_come_back_exactly(bits):
    """w = lo + s*q with s a power of two and every code 0 and 2^b-1 present
    in each group: the scale, bias and codes are recovered exactly."""
    rng = np.random.default_rng(11 + bits)
    N, K, qmax = 6, 256, (1 << bits) - 1
    q = rng.integers(0, qmax + 1, size=(N, K))
    q[:, ::64] = 0
    q[:, 1::64] = qmax
    s = 2.0 ** rng.integers(-8, 3, size=(N, K // 64))
    # lo/s + q stays an integer of magnitude <= 255: exact in bf16
    lo = rng.integers(-255, 256 - qmax, size=(N, K // 64)) * s
    w = np.repeat(lo, 64, axis=1) + np.repeat(s, 64, axis=1) * q
    wq, sc, bi = oracle.quantize_affine(bf16_bits(w.astype(np.float32)), N, K,
                                        bits)
    np.testing.assert_array_equal(bits_to_f64(sc), s)
    np.testing.assert_array_equal(bits_to_f64(bi), lo)
    np.testing.assert_array_equal(oracle.unpack(wq, N, K, bits), q)


@pytest.mark.parametrize("bits", [4, 8])
def test_round_trip_within_half_a_step(bits):
    """Random bf16 weights: |w - (s*q + bias)| <= s/2 + (2^b-1)|s - s_exact|
    (+ fp32 slack), where s_exact = (max - min) / (2^b - 1) unrounded; codes
    use the whole range."""
    rng = np.random.default_rng(100 + bits)
    N, K, qmax = 8, 512, (1 << bits) - 1
    w32 = rng.normal(0, 1, size=(N, K)).astype(np.float32) * np.float32(0.05)
    wb = to_bf16_rn(w32)
    w = bits_to_f64(wb)
    wq, sc, bi = oracle.quantize_affine(wb, N, K, bits)
    back = oracle.dequant(wq, sc, bi, N, K, bits)
    g = w.reshape(N, K // 64, 64)
    s_exact = (g.max(axis=2) - g.min(axis=2)) / qmax
    s = bits_to_f64(sc)
    bound = s / 2 + qmax * np.abs(s - s_exact) + 2.0 ** -20 * np.abs(g).max(axis=2)
    err = np.abs(back - w).reshape(N, K // 64, 64).max(axis=2)
    assert np.all(err <= bound * (1 + 1e-12)), (err / bound).max()
    codes = oracle.unpack(wq, N, K, bits).reshape(N, K // 64, 64)
    assert np.all(codes.min(axis=2) == 0)
    assert np.all(codes.max(axis=2) >= qmax - 1)
    # the scale is the bf16 rounding of the fp32 quotient
    np.testing.assert_array_equal(
        sc, to_bf16_rn((g.max(axis=2) - g.min(axis=2)).astype(np.float32)
                       / np.float32(qmax)))


@pytest.mark.parametrize("bits", [4, 8])
def test_round_half_to_even_not_truncation(bits):
    """Inputs exactly halfway between two grid points go to the even code;
    inputs just above half a step go up (truncation would keep them down)."""
    qmax = (1 << bits) - 1
    # grid lo = 0, s = 1 (max = qmax); probe values j + 0.5 and j + 0.75
    probes = [0.5, 1.5, 2.5, 3.25, 3.75, 4.5]
    vals = np.zeros(64, dtype=np.float32)
    vals[1] = qmax
    vals[2:2 + len(probes)] = probes
    wq, sc, bi = oracle.quantize_affine(bf16_bits(vals)[None, :], 1, 64, bits)
    assert bits_to_f64(sc)[0, 0] == 1.0
    codes = oracle.unpack(wq, 1, 64, bits)[0]
    assert list(codes[2:2 + len(probes)]) == [0, 2, 2, 3, 4, 4]


@pytest.mark.parametrize("bits", [4, 8])
def test_constant_and_two_valued_groups(bits):
    qmax = (1 << bits) - 1
    w = np.zeros((1, 128), dtype=np.float32)
    w[0, :64] = -3.5                      # constant group
    w[0, 64:] = np.where(np.arange(64) % 2 == 0, -1.0, 2.0)  # two values
    wq, sc, bi = oracle.quantize_affine(bf16_bits(w), 1, 128, bits)
    codes = oracle.unpack(wq, 1, 128, bits)[0]
    assert int(sc[0, 0]) == 0 and bits_to_f64(bi)[0, 0] == -3.5
    assert np.all(codes[:64] == 0)
    assert bits_to_f64(bi)[0, 1] == -1.0
    assert list(np.unique(codes[64:])) == [0, qmax]
    back = oracle.dequant(wq, sc, bi, 1, 128, bits)[0]
    assert np.all(back[:64] == -3.5)


@pytest.mark.parametrize("bits", [4, 8])
def test_codes_are_monotone_in_the_weights(bits):
    rng = np.random.default_rng(7 * bits)
    w32 = np.sort(rng.uniform(-2, 3, size=(4, 64)).astype(np.float32), axis=1)
    wb = to_bf16_rn(w32)
    wq, sc, bi = oracle.quantize_affine(wb, 4, 64, bits)
    codes = oracle.unpack(wq, 4, 64, bits).astype(int)
    assert np.all(np.diff(codes, axis=1) >= 0)
    assert np.all(codes[:, 0] == 0) and np.all(codes[:, -1] == (1 << bits) - 1)


def test_zero_minimum_is_stored_as_positive_zero():
    """-0 and +0 compare equal; whichever occurs, a zero minimum is stored
    as +0 (bits 0x0000), so the stored bias does not depend on input order."""
    vals = np.zeros((2, 64), dtype=np.float32)
    vals[:, 5] = 1.0
    vals[0, 0] = -0.0          # -0 first
    vals[1, 7] = -0.0          # +0 first, -0 later
    wq, sc, bi = oracle.quantize_affine(bf16_bits(vals), 2, 64, 4)
    assert list(bi[:, 0]) == [0, 0]

