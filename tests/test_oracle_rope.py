"""Pins for the oracle's rotary position embedding (CPU only).

The step is the fused RoPE of "The Cathedral Doubled Itself", "The kernel
that worked and the kernel that won't" (applied to the materialized Q and K;
designed, not shipped there).  The pages give no formula; the oracle uses the
textbook rotate-half form.  Pinned by a hand-worked head (which fixes the
pairing, the frequency exponent and the signs), identity at position 0, the
rotation's invariants (pair norms, composition of positions, dot products
that depend only on the position difference) and the Q/K/V composition.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "rope_worked_example.txt")


def read_golden():
    d, base, rows = None, None, []
    for ln in open(GOLDEN):
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        parts = ln.split()
        if parts[0] == "head_dim":
            d = int(parts[1])
        elif parts[0] == "base":
            base = float(parts[1])
        else:
            vals = [float(v) for v in parts]
            rows.append((int(vals[0]), vals[1:1 + d], vals[1 + d:1 + 2 * d]))
    return d, base, rows


def test_hand_worked_head():
    d, base, rows = read_golden()
    for pos, x, want in rows:
        got = oracle.rope(np.array([x]), d, base, [pos])[0]
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_position_zero_is_the_identity():
    rng = np.random.default_rng(1)
    y = rng.normal(size=(3, 256))
    np.testing.assert_array_equal(oracle.rope(y, 128, 1e6, [0, 0, 0]), y)


def rot(y, d, base, pos):
    return oracle.rope(y, d, base, pos)


@pytest.mark.parametrize("d,base", [(128, 10000.0), (64, 1e6)])
def test_pair_norms_are_preserved(d, base):
    rng = np.random.default_rng(d)
    y = rng.normal(size=(4, 3 * d))
    pos = [1, 17, 4095, 32767]
    out = rot(y, d, base, pos)
    h = d // 2
    y, out = y.reshape(4, 3, d), out.reshape(4, 3, d)
    n_in = y[..., :h] ** 2 + y[..., h:] ** 2
    n_out = out[..., :h] ** 2 + out[..., h:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


def test_positions_compose():
    rng = np.random.default_rng(2)
    y = rng.normal(size=(1, 128))
    twice = rot(rot(y, 128, 1e4, [300]), 128, 1e4, [77])
    once = rot(y, 128, 1e4, [377])
    np.testing.assert_allclose(twice, once, rtol=0, atol=1e-11)


def test_scores_depend_only_on_the_position_difference():
    rng = np.random.default_rng(3)
    q = rng.normal(size=(1, 128))
    k = rng.normal(size=(1, 128))
    base = 1e6

    def score(pq, pk):
        return float((rot(q, 128, base, [pq]) @ rot(k, 128, base, [pk]).T)[0, 0])

    ref = score(40, 13)
    for shift in (1, 500, 20000):
        assert abs(score(40 + shift, 13 + shift) - ref) <= 1e-9 * (1 + abs(ref))
    assert abs(score(41, 13) - ref) > 1e-6  # and it does depend on it


def test_qkv_rope_rotates_q_and_k_only():
    import gwa_synth as synth
    K, d = 512, 64
    w = synth.qweight(5, 128 + 64 + 64, K, 4)
    x = synth.activations(6, 2, K)
    pos = [3, 9]
    q, k, v = oracle.qkv_rope(x, w.wq, w.scales, w.biases, 128, 64, K, 4, d,
                              1e4, pos)
    q0, k0, v0 = oracle.fused_sections(x, w.wq, w.scales, w.biases,
                                       [128, 64, 64], K, 4)
    np.testing.assert_array_equal(v, v0)
    np.testing.assert_array_equal(q, oracle.rope(q0, d, 1e4, pos))
    np.testing.assert_array_equal(k, oracle.rope(k0, d, 1e4, pos))
    assert not np.allclose(q, q0)
