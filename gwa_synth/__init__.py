"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the projection itself: it draws packed
words, bf16 scales/biases, activations and MoE routings with the value
distributions of the workloads below, and hands the same arrays to both the
CUDA library and the CPU oracle.

Recipe (every draw from numpy's PCG64 with an explicit seed):
  * activations x: bf16(N(0, 1)); for the edge-case tests also N(0, 1)
    with outlier channels (1e2 .. 1e4), N(0, 1) scaled by 2^U{-14..8} per
    element, and groups of zeros and bf16 subnormals;
  * packed weights: uniform random uint32 words, so every b-bit field of every
    word is an independent uniform code in 0 .. 2^b - 1;
  * scales: bf16(U(0.005, 0.02)), one per row per group of 64 inputs;
  * biases: bf16(-8 * scale + N(0, 1e-3)) with the stored (bf16) scale;
  * MoE: top-k expert ids drawn uniformly without replacement per token;
    routing weights are the softmax of N(0, 1) logits over the k selected
    slots (fp32).

bf16 values are carried as their uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

GROUP = 64


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def seed_for(config: int, layer: int = 0, tensor: int = 0) -> int:
    """Seed of one tensor: 1000*config + 10*layer + tensor."""
    return 1000 * int(config) + 10 * int(layer) + int(tensor)


def bf16_bits(a) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (uint16), round to nearest even.

    Only used to encode inputs; NaN does not occur in these draws."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_values(h) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


@dataclass
class QWeight:
    """One affine group-quantized weight in the packed layout.

    wq:     uint32 [rows, K*bits/32]  (codes packed along the input axis)
    scales: uint16 (bf16 bits) [rows, K/64]
    biases: uint16 (bf16 bits) [rows, K/64]
    """
    wq: np.ndarray
    scales: np.ndarray
    biases: np.ndarray
    N: int
    K: int
    bits: int
    group: int = GROUP

    @property
    def nbytes(self) -> int:
        return self.wq.nbytes + self.scales.nbytes + self.biases.nbytes


def activations(seed: int, M: int, K: int) -> np.ndarray:
    """x bf16 [M, K] ~ N(0, 1)."""
    r = rng_for(seed)
    return bf16_bits(r.standard_normal((M, K), dtype=np.float32))


def activations_outliers(seed: int, M: int, K: int, values=(1e3,),
                         count: int = 3) -> np.ndarray:
    """x bf16 [M, K] ~ N(0, 1) with `count` entries of each row set to
    +-v for v cycling over `values` (outlier channels), at positions drawn
    without replacement."""
    r = rng_for(seed)
    x = r.standard_normal((M, K), dtype=np.float32)
    for m in range(M):
        pos = r.choice(K, size=count, replace=False)
        sign = np.where(r.random(count) < 0.5, -1.0, 1.0)
        for i, k in enumerate(pos):
            x[m, k] = sign[i] * values[i % len(values)]
    return bf16_bits(x)


def activations_wide(seed: int, M: int, K: int, lo: int = -14,
                     hi: int = 8) -> np.ndarray:
    """x bf16 [M, K]: N(0, 1) times 2^e, e uniform on lo..hi per element, so
    every group of 64 spans far more than 2^8 in magnitude."""
    r = rng_for(seed)
    x = r.standard_normal((M, K), dtype=np.float32)
    e = r.integers(lo, hi + 1, size=(M, K))
    return bf16_bits(np.ldexp(x, e).astype(np.float32))


def activations_edge(seed: int, M: int, K: int) -> np.ndarray:
    """x bf16 [M, K] of edge values, cycling over the groups of 64: a group
    of zeros (both signs), a group of bf16 subnormals, normal values with a
    few subnormals and zeros among them, and plain N(0, 1)."""
    r = rng_for(seed)
    h = bf16_bits(r.standard_normal((M, K), dtype=np.float32))
    G = K // GROUP
    for m in range(M):
        for g in range(G):
            sl = slice(g * GROUP, (g + 1) * GROUP)
            kind = (g + m) % 4
            if kind == 0:
                h[m, sl] = np.where(r.random(GROUP) < 0.5, 0x0000, 0x8000)
            elif kind == 1:
                sub = r.integers(1, 0x80, size=GROUP).astype(np.uint16)
                h[m, sl] = sub | np.where(r.random(GROUP) < 0.5, 0, 0x8000
                                          ).astype(np.uint16)
            elif kind == 2:
                idx = r.choice(GROUP, size=12, replace=False)
                seg = h[m, sl].copy()
                seg[idx[:6]] = r.integers(1, 0x80, size=6).astype(np.uint16)
                seg[idx[6:]] = 0
                h[m, sl] = seg
    return h


def packed_words(rng: np.random.Generator, N: int, K: int,
                 bits: int) -> np.ndarray:
    wpr = K * bits // 32
    return rng.integers(0, 2**32, size=(N, wpr), dtype=np.uint32)


def scale_bias(rng: np.random.Generator, N: int, K: int, group: int = GROUP):
    G = K // group
    s = bf16_bits(rng.uniform(0.005, 0.02, size=(N, G)).astype(np.float32))
    noise = rng.normal(0.0, 1e-3, size=(N, G)).astype(np.float32)
    b = bf16_bits(-8.0 * bf16_values(s) + noise)
    return s, b


# `bits` of fp8 (e4m3) weights: 8-bit codes in the same container
FP8_E4M3 = 0x108


def qweight(seed: int, N: int, K: int, bits: int = 4,
            group: int = GROUP) -> QWeight:
    """A seeded packed weight of N output rows and K inputs.  fp8 weights
    (bits = FP8_E4M3): uniform random code bytes other than the two NaN
    codes (0x7f, 0xff become 0x7e, 0xfe), the same scales, biases
    N(0, 1e-3) (the codes are signed)."""
    width = 8 if bits == FP8_E4M3 else bits
    if K % group or (K * width) % 32:
        raise ValueError("K must be a multiple of the group and of 32/bits")
    r = rng_for(seed)
    wq = packed_words(r, N, K, width)
    s, b = scale_bias(r, N, K, group)
    if bits == FP8_E4M3:
        by = wq.view(np.uint8)
        by[(by & 0x7f) == 0x7f] -= 1
        b = bf16_bits(r.normal(0.0, 1e-3, size=s.shape).astype(np.float32))
    return QWeight(wq, s, b, N, K, bits, group)


def stack_rows(parts) -> QWeight:
    """Concatenate weights along the output axis (host side)."""
    K, bits, group = parts[0].K, parts[0].bits, parts[0].group
    if any(p.K != K or p.bits != bits or p.group != group for p in parts):
        raise ValueError("parts must share K, bits and group")
    return QWeight(np.concatenate([p.wq for p in parts]),
                   np.concatenate([p.scales for p in parts]),
                   np.concatenate([p.biases for p in parts]),
                   sum(p.N for p in parts), K, bits, group)


def routing(seed: int, M: int, topk: int, E: int):
    """Top-k expert ids (int32 [M, topk], distinct per token) and routing
    weights (float32 [M, topk], softmax of N(0,1) logits over the slots)."""
    r = rng_for(seed)
    ids = np.stack([r.choice(E, size=topk, replace=False)
                    for _ in range(M)]).astype(np.int32).reshape(M, topk)
    logits = r.standard_normal((M, topk)).astype(np.float64)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# ---------------------------------------------------------------- on device
def device_qweight(seed: int, N: int, K: int, bits: int = 4,
                   group: int = GROUP, device="cuda"):
    """The same recipe drawn on the GPU with torch's generator, for weights
    too large to draw on the host (the 48-layer stack).  Returns the raw
    tensors (wq int32 [N, K*bits/32], scales/biases bfloat16 [N, K/group]);
    a test copies a sampled layer back to the host for the oracle."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    width = 8 if bits == FP8_E4M3 else bits
    wpr = K * width // 32
    wq = torch.randint(0, 2**32, (N, wpr), generator=g, device=device,
                       dtype=torch.int64).to(torch.int32)
    G = K // group
    s = (torch.rand((N, G), generator=g, device=device) * 0.015 + 0.005)
    s = s.to(torch.bfloat16)
    noise = torch.randn((N, G), generator=g, device=device) * 1e-3
    if bits == FP8_E4M3:  # no NaN codes; signed codes, small biases
        by = wq.view(torch.uint8)
        by -= ((by & 0x7f) == 0x7f).to(torch.uint8)
        return wq, s, noise.to(torch.bfloat16)
    b = (-8.0 * s.float() + noise).to(torch.bfloat16)
    return wq, s, b


def stack_layer_shapes(hidden=5120, q=5120, kv=1024, intermediate=13824):
    """(name, rows, K) of the four projections of one dense layer:
    fused QKV, o_proj, fused gate+up, down."""
    return [("qkv", q + 2 * kv, hidden), ("o", hidden, q),
            ("gate_up", 2 * intermediate, hidden),
            ("down", hidden, intermediate)]


def stack_seed(layer: int, proj: int, bits: int) -> int:
    return seed_for(3, layer, proj) + 100000 * bits


# Workload shapes (sizes only).
TINY_QKV = dict(M=1, K=512, sections=(512, 128, 128), bits=4)
QKV_5120 = dict(M=1, K=5120, sections=(5120, 1024, 1024), bits=4)
GATE_UP_5120 = dict(K=5120, I=13824, bits=4)
STACK_LAYER = dict(hidden=5120, qkv=(5120, 1024, 1024), o=5120,
                   intermediate=13824, layers=48)
MOE_2048 = dict(hidden=2048, experts=256, I=512, topk=8, bits=4)
