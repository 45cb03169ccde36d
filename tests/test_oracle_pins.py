"""Pins for the CPU oracle: each test checks it against something other than
itself -- literal words written by hand, exact rational arithmetic over bit
strings, closed forms, special cases and the values the pages print.

The independent routes used here (bit-string field slicing, bf16 decoding by
sign/exponent/mantissa fields, ``fractions.Fraction`` sums) share nothing with
the oracle's shift-and-mask C code.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import gwa_synth as synth
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def fields_of_word(word: int, bits: int):
    """Codes of one packed word via its binary string: field 0 is the lowest
    `bits` bits (the low-bits-first reading of the packed layout)."""
    s = format(int(word), "032b")                    # most significant first
    msb_first = [s[i:i + bits] for i in range(0, 32, bits)]
    return [int(f, 2) for f in reversed(msb_first)]


def word_of_fields(codes, bits: int) -> int:
    """Inverse of fields_of_word, again through a binary string."""
    return int("".join(format(int(c), f"0{bits}b") for c in reversed(codes)), 2)


def fields_of_row(words, bits: int, K: int):
    """Codes of one packed row via the binary string of its whole bit
    stream (word 0 holds stream bits 0..31): code k is stream bits
    [bits*k, bits*k + bits).  Covers widths that straddle words (u3, u6)."""
    s = "".join(format(int(w), "032b") for w in reversed(list(words)))
    L = len(s)                                       # s[L-1] is stream bit 0
    return [int(s[L - bits * (k + 1):L - bits * k], 2) for k in range(K)]


def row_of_fields(codes, bits: int):
    """Inverse of fields_of_row: the row's words, again through a string."""
    s = "".join(format(int(c), f"0{bits}b") for c in reversed(list(codes)))
    assert len(s) % 32 == 0
    return [int(s[len(s) - 32 * (j + 1):len(s) - 32 * j], 2)
            for j in range(len(s) // 32)]


def bf16_fraction(h: int) -> Fraction:
    """Exact value of a bf16 bit pattern from its fields."""
    h = int(h)
    sign = -1 if (h >> 15) & 1 else 1
    e = (h >> 7) & 0xFF
    m = h & 0x7F
    assert e != 0xFF, "no inf/nan in these tests"
    if e == 0:
        return sign * Fraction(m, 128) * Fraction(1, 2**126)
    return sign * (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)


def exact_qmv(x, w: synth.QWeight):
    """y[m, n] as exact rationals, from bit strings and field-decoded bf16."""
    M = x.shape[0]
    codes = [fields_of_row(w.wq[n], w.bits, w.K) for n in range(w.N)]
    y = [[Fraction(0)] * w.N for _ in range(M)]
    for n in range(w.N):
        assert len(codes[n]) == w.K and w.wq.shape[1] * 32 == w.K * w.bits
        for m in range(M):
            acc = Fraction(0)
            for k in range(w.K):
                g = k // w.group
                wk = bf16_fraction(w.scales[n, g]) * codes[n][k] + \
                    bf16_fraction(w.biases[n, g])
                acc += bf16_fraction(x[m, k]) * wk
            y[m][n] = acc
    return y


def bf16_of_float(v: float) -> int:
    """bf16 pattern of a value that bf16 represents exactly."""
    h = int(synth.bf16_bits(np.array([v], dtype=np.float32))[0])
    assert bf16_fraction(h) == Fraction(v)
    return h


# ---------------------------------------------------------------- unpack
def test_unpack_literal_words_low_bits_first():
    # 0x76543210 holds the nibbles 0..7 from the lowest bits up.
    got = oracle.unpack(np.array([[0x76543210, 0xFEDCBA98]], np.uint32),
                        1, 16, 4)
    assert got.tolist() == [list(range(16))]
    got8 = oracle.unpack(np.array([[0x03020100, 0xFF807F01]], np.uint32),
                         1, 8, 8)
    assert got8.tolist() == [[0, 1, 2, 3, 0x01, 0x7F, 0x80, 0xFF]]


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_unpack_roundtrip_every_code_every_position(bits):
    P = 32 // bits
    levels = 1 << bits
    rows = []
    # every code value at every field position, other fields varying too
    for pos in range(P):
        for c in range(levels):
            codes = [(c + 3 * j + 1) % levels for j in range(P)]
            codes[pos] = c
            rows.append(codes)
    words = np.array([[word_of_fields(r, bits)] for r in rows], np.uint32)
    got = oracle.unpack(words, len(rows), P, bits)
    assert got.tolist() == rows
    # and the string slicer agrees with the literal layout on random words
    r = np.random.default_rng(5).integers(0, 2**32, size=(7, 3),
                                          dtype=np.uint32)
    got = oracle.unpack(r, 7, 3 * P, bits)
    want = [[c for word in row for c in fields_of_word(word, bits)]
            for row in r]
    assert got.tolist() == want


# ---------------------------------------------------------------- dequant
def test_dequant_closed_form_and_identity_case():
    K = 128
    w = synth.qweight(11, 3, K, 4)
    got = oracle.dequant(w.wq, w.scales, w.biases, 3, K, 4)
    for n in range(3):
        codes = [c for word in w.wq[n] for c in fields_of_word(word, 4)]
        for k in range(K):
            want = bf16_fraction(w.scales[n, k // 64]) * codes[k] + \
                bf16_fraction(w.biases[n, k // 64])
            assert Fraction(got[n, k]) == want      # exact in fp64
    # scale 1, bias 0: the weight is the integer code itself
    one, zero = bf16_of_float(1.0), 0
    s = np.full((3, 2), one, np.uint16)
    b = np.full((3, 2), zero, np.uint16)
    got = oracle.dequant(w.wq, s, b, 3, K, 4)
    codes = np.array([[c for word in row for c in fields_of_word(word, 4)]
                      for row in w.wq])
    assert np.array_equal(got, codes.astype(np.float64))


def test_unpack_straddling_codes_literal_words():
    """u3 code 10 occupies stream bits 30..32 and u6 code 5 bits 30..35: a
    code of all ones there sets the top two bits of word 0 and the lowest
    one (u3) or four (u6) bits of word 1, worked by hand."""
    for bits, k, w0, w1 in [(3, 10, 0xC0000000, 0x00000001),
                            (6, 5, 0xC0000000, 0x0000000F)]:
        K = 32
        words = np.zeros((1, K * bits // 32), np.uint32)
        words[0, 0], words[0, 1] = w0, w1
        want = [0] * K
        want[k] = (1 << bits) - 1
        assert list(oracle.unpack(words, 1, K, bits)[0]) == want
    # u3 codes 0..7 in order: 0b111_110_101_100_011_010_001_000 = 0xFAC688
    words = np.zeros((1, 3), np.uint32)
    words[0, 0] = 0x00FAC688
    assert list(oracle.unpack(words, 1, 32, 3)[0][:8]) == list(range(8))


@pytest.mark.parametrize("bits", [3, 6])
def test_unpack_roundtrip_straddling_widths(bits):
    """Every code value at every position of a 32-code row (3 or 6 words),
    packed through a bit string; and random rows read back by slicing."""
    K, levels = 32, 1 << bits
    rows = [[(v + k) % levels for k in range(K)] for v in range(levels)]
    words = np.array([row_of_fields(r, bits) for r in rows], np.uint32)
    got = oracle.unpack(words, len(rows), K, bits)
    assert np.array_equal(got, np.array(rows))
    r = np.random.default_rng(bits).integers(0, 2**32, size=(5, 3 * 4 * bits // 4),
                                             dtype=np.uint64).astype(np.uint32)
    Kr = r.shape[1] * 32 // bits
    got = oracle.unpack(r, 5, Kr, bits)
    want = [fields_of_row(row, bits, Kr) for row in r]
    assert np.array_equal(got, np.array(want))


# ---------------------------------------------------------------- qmv
@pytest.mark.parametrize("bits,group", [(4, 64), (8, 64), (2, 64), (4, 32),
                                        (4, 128), (2, 32), (8, 128), (3, 64),
                                        (6, 64), (3, 32), (6, 128)])
def test_qmv_matches_exact_rational_bruteforce(bits, group):
    M, N, K = 2, 5, 384            # several groups; N != K catches transposes
    w = synth.qweight(21 + bits + group, N, K, bits, group)
    x = synth.activations(31 + bits, M, K)
    got = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, bits, group)
    want = exact_qmv(x, w)
    for m in range(M):
        for n in range(N):
            ref = float(want[m][n])
            assert abs(got[m, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_qmv_integer_case_is_exact():
    # scale 1, bias 0, small integer activations: y is an integer matmul.
    M, N, K = 3, 4, 128
    r = np.random.default_rng(3)
    wq = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    xi = r.integers(-4, 5, size=(M, K))
    x = synth.bf16_bits(xi.astype(np.float32))
    s = np.full((N, 2), bf16_of_float(1.0), np.uint16)
    b = np.zeros((N, 2), np.uint16)
    got = oracle.qmv(x, wq, s, b, N, K, 4)
    codes = np.array([[c for word in row for c in fields_of_word(word, 4)]
                      for row in wq], dtype=np.int64)
    assert np.array_equal(got, (xi @ codes.T).astype(np.float64))


def test_qmv_centred_codes_cancel_to_zero():
    # every code 8 and bias = -8*scale: every weight is exactly 0.
    M, N, K = 2, 3, 256
    wq = np.full((N, K // 8), 0x88888888, np.uint32)
    s = synth.bf16_bits(np.array([[0.0078125, 0.015625, 0.01171875, 0.5]] * N,
                                 np.float32))
    b = synth.bf16_bits(-8.0 * synth.bf16_values(s))
    x = synth.activations(7, M, K)
    got = oracle.qmv(x, wq, s, b, N, K, 4)
    assert np.all(got == 0.0)


@pytest.mark.parametrize("k", [0, 7, 8, 63, 64, 65, 127, 191])
def test_qmv_one_hot_reads_one_code(k):
    # x = e_k gives y[n] = S[n, k/64] * q[n, k] + B[n, k/64]: one field of one
    # word, with the scale of the group that k falls in.
    N, K = 6, 192
    w = synth.qweight(41, N, K, 4)
    x = np.zeros((1, K), np.uint16)
    x[0, k] = bf16_of_float(1.0)
    got = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, 4)
    for n in range(N):
        q = fields_of_word(w.wq[n, k // 8], 4)[k % 8]
        want = bf16_fraction(w.scales[n, k // 64]) * q + \
            bf16_fraction(w.biases[n, k // 64])
        assert Fraction(got[0, n]) == want


def test_qmv_row_subset_equals_full():
    N, K = 40, 256
    w = synth.qweight(51, N, K, 4)
    x = synth.activations(52, 3, K)
    full = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, 4)
    rows = [39, 0, 17, 17, 5]
    sub = oracle.qmv(x, w.wq, w.scales, w.biases, N, K, 4, rows=rows)
    assert np.array_equal(sub, full[:, rows])


# ---------------------------------------------------------------- sections
def test_fused_sections_equal_separate_projections():
    K = 256
    parts = [synth.qweight(60 + i, n, K, 4) for i, n in
             enumerate((64, 16, 16))]
    fused = synth.stack_rows(parts)
    x = synth.activations(65, 2, K)
    outs = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases,
                                 (64, 16, 16), K, 4)
    for o, p in zip(outs, parts):
        sep = oracle.qmv(x, p.wq, p.scales, p.biases, p.N, K, 4)
        assert o.flags["C_CONTIGUOUS"] and o.shape == sep.shape
        assert np.array_equal(o, sep)              # same arithmetic, same order


def test_fused_sections_optional_bias_added_per_section():
    K = 128
    parts = [synth.qweight(70 + i, n, K, 4) for i, n in enumerate((8, 4))]
    fused = synth.stack_rows(parts)
    x = synth.activations(72, 1, K)
    bias = [synth.bf16_bits(np.arange(8, dtype=np.float32) * 0.25),
            synth.bf16_bits(-np.arange(4, dtype=np.float32))]
    plain = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases,
                                  (8, 4), K, 4)
    withb = oracle.fused_sections(x, fused.wq, fused.scales, fused.biases,
                                  (8, 4), K, 4, out_bias=bias)
    assert np.array_equal(withb[0] - plain[0],
                          np.arange(8, dtype=np.float64)[None, :] * 0.25)
    assert np.array_equal(withb[1] - plain[1],
                          -np.arange(4, dtype=np.float64)[None, :])


# ---------------------------------------------------------------- SiLU
def test_silu_textbook_identities():
    assert oracle.silu(0.0) == 0.0
    ln3 = math.log(3.0)
    assert abs(oracle.silu(ln3) - 0.75 * ln3) < 1e-15     # sigma(ln 3) = 3/4
    for g in (0.3, 1.7, 5.0, 12.5):
        # sigma(g) + sigma(-g) = 1  =>  silu(g) - silu(-g) = g
        assert abs(oracle.silu(g) - oracle.silu(-g) - g) < 1e-14 * max(1, g)
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15


def test_gate_up_rows_order_and_epilogue():
    # Gate rows first, then up rows: build a weight whose gate half and up
    # half give recognisably different outputs with a one-hot x.
    K, I = 128, 4
    one = bf16_of_float(1.0)
    wq = np.zeros((2 * I, K // 8), np.uint32)
    gate_codes = [1, 2, 3, 4]
    up_codes = [5, 6, 7, 9]
    for i in range(I):
        wq[i, 0] = gate_codes[i]               # field 0 of word 0 -> k = 0
        wq[I + i, 0] = up_codes[i]
    s = np.full((2 * I, 2), one, np.uint16)
    b = np.zeros((2 * I, 2), np.uint16)
    x = np.zeros((1, K), np.uint16)
    x[0, 0] = one
    h = oracle.gate_up_silu(x, wq, s, b, 2 * I, K, 4)
    for i in range(I):
        g, u = gate_codes[i], up_codes[i]
        assert abs(h[0, i] - g / (1 + math.exp(-g)) * u) < 1e-13


def test_gate_up_equals_silu_of_halves():
    K, I = 192, 24
    w = synth.qweight(81, 2 * I, K, 4)
    x = synth.activations(82, 3, K)
    y = oracle.qmv(x, w.wq, w.scales, w.biases, 2 * I, K, 4)
    h = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, 4)
    g, u = y[:, :I], y[:, I:]
    want = g / (1.0 + np.exp(-g)) * u
    assert np.allclose(h, want, rtol=1e-14, atol=1e-14)
    cols = [3, 0, 23]
    hs = oracle.gate_up_silu(x, w.wq, w.scales, w.biases, 2 * I, K, 4,
                             cols=cols)
    assert np.array_equal(hs, h[:, cols])


# ---------------------------------------------------------------- MoE
def _experts(seed, E, N, K, bits=4):
    return synth.stack_rows([synth.qweight(seed + e, N, K, bits)
                             for e in range(E)])


def test_moe_gate_up_is_a_loop_of_gate_up_calls():
    E, I, K, M, topk = 6, 8, 128, 3, 2
    w = _experts(100, E, 2 * I, K)
    x = synth.activations(120, M, K)
    ids, _ = synth.routing(121, M, topk, E)
    h = oracle.moe_gate_up_silu(x, ids, w.wq, w.scales, w.biases, E, 2 * I,
                                K, 4)
    rows = 2 * I
    for t in range(M):
        for j in range(topk):
            e = ids[t, j]
            sl = slice(e * rows, (e + 1) * rows)
            want = oracle.gate_up_silu(x[t:t + 1], w.wq[sl], w.scales[sl],
                                       w.biases[sl], rows, K, 4)
            assert np.array_equal(h[t, j], want[0])


def test_moe_down_is_a_routed_sum_of_qmv_calls():
    E, N, K, M, topk = 5, 16, 64, 2, 3
    w = _experts(200, E, N, K)
    ids, r = synth.routing(220, M, topk, E)
    hin = synth.activations(221, M * topk, K).reshape(M, topk, K)
    y = oracle.moe_down_combine(hin, ids, r, w.wq, w.scales, w.biases, E, N,
                                K, 4)
    for t in range(M):
        want = np.zeros(N)
        for j in range(topk):
            e = ids[t, j]
            sl = slice(e * N, (e + 1) * N)
            want += float(r[t, j]) * oracle.qmv(
                hin[t, j][None], w.wq[sl], w.scales[sl], w.biases[sl], N, K,
                4)[0]
        assert np.allclose(y[t], want, rtol=1e-13, atol=1e-13)


def test_moe_top1_with_unit_weight_is_plain_qmv():
    E, N, K = 4, 12, 128
    w = _experts(300, E, N, K)
    ids = np.array([[2], [0]], np.int32)
    r = np.ones((2, 1), np.float32)
    hin = synth.activations(301, 2, K).reshape(2, 1, K)
    y = oracle.moe_down_combine(hin, ids, r, w.wq, w.scales, w.biases, E, N,
                                K, 4)
    for t, e in enumerate((2, 0)):
        sl = slice(e * N, (e + 1) * N)
        want = oracle.qmv(hin[t, 0][None], w.wq[sl], w.scales[sl],
                          w.biases[sl], N, K, 4)[0]
        assert np.array_equal(y[t], want)


def test_moe_rejects_out_of_range_expert():
    E, N, K = 2, 4, 64
    w = _experts(400, E, N, K)
    ids = np.array([[2]], np.int32)
    with pytest.raises(ValueError):
        oracle.moe_down_combine(np.zeros((1, 1, K), np.uint16), ids,
                                np.ones((1, 1), np.float32), w.wq, w.scales,
                                w.biases, E, N, K, 4)


# ---------------------------------------------------------------- the pages
def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_bits_per_weight_matches_printed_table():
    # One bf16 scale and one bf16 bias per 64 weights: footprint of the arrays
    # the oracle consumes, per weight, must equal the printed bpw.
    for quant, bits, bpw in _rows("bpw_table.txt"):
        bits, bpw = int(bits), float(bpw)
        w = synth.qweight(1, 4, 256, bits)
        per_weight = 8 * w.nbytes / (4 * 256)
        assert per_weight == bpw, quant


def test_fused_qkv_packed_shape_matches_page():
    for hidden, q_out, kv_out, bits, rows, wpr in _rows("fused_qkv_shape.txt"):
        hidden, q_out, kv_out, bits = map(int, (hidden, q_out, kv_out, bits))
        parts = [synth.qweight(2, n, hidden, bits)
                 for n in (q_out, kv_out, kv_out)]
        fused = synth.stack_rows(parts)
        assert fused.wq.shape == (int(rows), int(wpr)) == \
            (q_out + 2 * kv_out, hidden // 8)
