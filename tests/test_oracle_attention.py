"""Pins for the oracle's attention over a 4-bit value cache (CPU only).

The step is sdpa_dequant_v ("Sanctum-MLX", six-changes table row 5 and the
paragraph after it); the value format is the library's affine reading
(v = scale * code + bias per group of head dimensions).  Each test pins the
oracle to a closed form: a hand-worked two-key case, a single visible key,
equal scores, the causal mask, the GQA head mapping and the score scale.
"""
import math
import os

import numpy as np
import pytest

import gwa_synth as synth
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "attention_worked_example.txt")


def bf16(a):
    return synth.bf16_bits(np.asarray(a, dtype=np.float32))


def pack_codes(codes, bits=4):
    """codes [..., D] -> words [..., D*bits/32], lowest bits first."""
    codes = np.asarray(codes, dtype=np.uint64)
    per = 32 // bits
    c = codes.reshape(codes.shape[:-1] + (codes.shape[-1] // per, per))
    words = np.zeros(c.shape[:-1], dtype=np.uint64)
    for j in range(per):
        words |= c[..., j] << np.uint64(bits * j)
    return words.astype(np.uint32)


def random_cache(seed, B, Hkv, T, D, bits=4, group=64):
    rng = np.random.default_rng(seed)
    k = bf16(rng.normal(0, 1, size=(B, Hkv, T, D)))
    codes = rng.integers(0, 1 << bits, size=(B, Hkv, T, D))
    vq = pack_codes(codes, bits)
    vs = bf16(rng.uniform(0.01, 0.05, size=(B, Hkv, T, D // group)))
    vb = bf16(rng.normal(0, 0.2, size=(B, Hkv, T, D // group)))
    return k, codes, vq, vs, vb


def dequant_rows(codes, vs, vb, group=64):
    s = np.repeat(synth.bf16_values(vs).astype(np.float64), group, axis=-1)
    b = np.repeat(synth.bf16_values(vb).astype(np.float64), group, axis=-1)
    return s * codes + b


def test_hand_worked_two_keys():
    vals = {}
    for ln in open(GOLDEN):
        ln = ln.strip()
        if ln and not ln.startswith("#"):
            key, v = ln.split()
            vals[key] = float(v)
    D = int(vals["D"])
    q = np.zeros((1, 1, 1, D), dtype=np.float32); q[..., 0] = 1
    k = np.zeros((1, 1, 2, D), dtype=np.float32); k[0, 0, 1, 0] = 1
    codes = np.zeros((1, 1, 2, D), dtype=np.int64)
    codes[0, 0, 0] = int(vals["codes0"]); codes[0, 0, 1] = int(vals["codes1"])
    ones = bf16(np.ones((1, 1, 2, 1))); zeros = bf16(np.zeros((1, 1, 2, 1)))
    out = oracle.sdpa_dequant_v(bf16(q), bf16(k), pack_codes(codes), ones,
                                zeros, 1, 1, 1, D, 1, 2,
                                scale=math.log(vals["scale_ln"]), causal=False)
    np.testing.assert_allclose(out, vals["out"], rtol=0, atol=1e-12)


def test_single_visible_key_returns_its_value():
    B, Hq, Hkv, T, D = 1, 2, 1, 1, 128
    k, codes, vq, vs, vb = random_cache(1, B, Hkv, T, D)
    q = bf16(np.random.default_rng(2).normal(size=(B, Hq, 1, D)))
    out = oracle.sdpa_dequant_v(q, k, vq, vs, vb, B, Hq, 1, D, Hkv, T)
    want = dequant_rows(codes, vs, vb)[0, 0, 0]
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h, 0], want, rtol=0, atol=1e-12)
    # and it agrees with the weight dequantization the projections use
    flat = oracle.dequant(vq.reshape(1, -1), vs.reshape(1, -1),
                          vb.reshape(1, -1), 1, D, 4)[0]
    np.testing.assert_allclose(out[0, 0, 0], flat, rtol=0, atol=1e-12)


def test_equal_scores_average_the_visible_values():
    B, Hq, Hkv, T, D = 1, 1, 1, 9, 64
    k, codes, vq, vs, vb = random_cache(3, B, Hkv, T, D)
    q = bf16(np.zeros((B, Hq, 1, D)))
    out = oracle.sdpa_dequant_v(q, k, vq, vs, vb, B, Hq, 1, D, Hkv, T)
    want = dequant_rows(codes, vs, vb)[0, 0].mean(axis=0)
    np.testing.assert_allclose(out[0, 0, 0], want, rtol=0, atol=1e-12)


def test_causal_mask_hides_later_keys():
    B, Hq, Hkv, T, D, Lq = 1, 1, 1, 5, 64, 2
    k, codes, vq, vs, vb = random_cache(4, B, Hkv, T, D)
    q = bf16(np.zeros((B, Hq, Lq, D)))
    # make the last key dominate any query that can see it
    k2 = synth.bf16_values(k).copy(); k2[0, 0, T - 1] = 0
    out = oracle.sdpa_dequant_v(q, bf16(k2), vq, vs, vb, B, Hq, Lq, D, Hkv, T)
    vals = dequant_rows(codes, vs, vb)[0, 0]
    # query 0 sees keys 0..T-2, query 1 sees all T (scores all 0: the mean)
    np.testing.assert_allclose(out[0, 0, 0], vals[:T - 1].mean(axis=0), atol=1e-12)
    np.testing.assert_allclose(out[0, 0, 1], vals.mean(axis=0), atol=1e-12)
    nc = oracle.sdpa_dequant_v(q, bf16(k2), vq, vs, vb, B, Hq, Lq, D, Hkv, T,
                               causal=False)
    np.testing.assert_allclose(nc[0, 0, 0], vals.mean(axis=0), atol=1e-12)


def test_gqa_head_mapping():
    B, Hq, Hkv, T, D = 2, 6, 2, 3, 64
    k, codes, vq, vs, vb = random_cache(5, B, Hkv, T, D)
    q = bf16(np.zeros((B, Hq, 1, D)))
    out = oracle.sdpa_dequant_v(q, k, vq, vs, vb, B, Hq, 1, D, Hkv, T)
    vals = dequant_rows(codes, vs, vb)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(out[b, h, 0], vals[b, h // 3].mean(axis=0),
                                       atol=1e-12)


def test_scale_acts_like_scaling_the_query():
    B, Hq, Hkv, T, D = 1, 1, 1, 6, 64
    k, codes, vq, vs, vb = random_cache(6, B, Hkv, T, D)
    qf = np.random.default_rng(7).normal(size=(B, Hq, 1, D)).astype(np.float32)
    a = oracle.sdpa_dequant_v(bf16(qf), k, vq, vs, vb, B, Hq, 1, D, Hkv, T,
                              scale=0.5)
    b = oracle.sdpa_dequant_v(bf16(qf * 2), k, vq, vs, vb, B, Hq, 1, D, Hkv, T,
                              scale=0.25)   # q * 2 is exact in bf16
    np.testing.assert_allclose(a, b, rtol=1e-12)
    # and a larger scale sharpens: the output moves toward the top key's value
    vals = dequant_rows(codes, vs, vb)[0, 0]
    scores = (synth.bf16_values(k)[0, 0].astype(np.float64) @
              synth.bf16_values(bf16(qf))[0, 0, 0].astype(np.float64))
    top = vals[np.argmax(scores)]
    sharp = oracle.sdpa_dequant_v(bf16(qf), k, vq, vs, vb, B, Hq, 1, D, Hkv, T,
                                  scale=200.0)
    np.testing.assert_allclose(sharp[0, 0, 0], top, atol=1e-6)
