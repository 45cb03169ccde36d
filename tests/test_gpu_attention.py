"""GPU parity of the attention over a quantized value cache
(gwa_sdpa_dequant_v; "Sanctum-MLX", six-changes table row 5) against the
oracle: plain fp64 softmax attention with the values dequantized by the
library's affine format.  Outputs within |err| <= 1e-2 * max(1, |ref|).
Cases span one key, key counts that are not multiples of the splits, GQA
groups of 1 to 8 query heads, several query positions under the causal mask,
head widths 64/128/256, u4 and u8 values, and batches.
"""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from helpers import dev_bf16

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()
    assert torch.cuda.is_available()


def cache(seed, B, Hkv, T, D, bits):
    rng = np.random.default_rng(seed)
    k = synth.bf16_bits(rng.normal(0, 1, size=(B, Hkv, T, D)).astype(np.float32))
    vq = rng.integers(0, 2**32, size=(B, Hkv, T, D * bits // 32), dtype=np.uint32)
    vs = synth.bf16_bits(rng.uniform(0.01, 0.05, size=(B, Hkv, T, D // 64)).astype(np.float32))
    vb = synth.bf16_bits((-synth.bf16_values(vs) * (2 ** bits - 1) / 2 +
                          rng.normal(0, 0.05, size=vs.shape)).astype(np.float32))
    return k, vq, vs, vb


def run(B, Hq, Hkv, Lq, T, D, bits=4, causal=True, seed=0, qscale=1.0):
    rng = np.random.default_rng(1000 + seed)
    q = synth.bf16_bits((rng.normal(0, 1, size=(B, Hq, Lq, D)) * qscale).astype(np.float32))
    k, vq, vs, vb = cache(seed, B, Hkv, T, D, bits)
    got = gwa.sdpa_dequant_v(
        dev_bf16(q), dev_bf16(k),
        torch.from_numpy(vq.view(np.int32)).cuda(), dev_bf16(vs), dev_bf16(vb),
        bits=bits, causal=causal)
    torch.cuda.synchronize()
    ref = oracle.sdpa_dequant_v(q, k, vq, vs, vb, B, Hq, Lq, D, Hkv, T,
                                bits=bits, causal=causal)
    ok, max_err, worst = oracle.within_tolerance(
        got.float().cpu().numpy().astype(np.float64), ref, TOL)
    assert ok, f"max |err| {max_err:.3g}, worst {worst:.3g}"


@pytest.mark.parametrize("T", [1, 7, 64, 1000, 4097])
def test_decode_gqa(T):
    # one query per head, 40 query heads over 8 KV heads, heads of 128
    run(1, 40, 8, 1, T, 128, seed=T)


@pytest.mark.parametrize("Lq,T", [(4, 4), (4, 300), (9, 50)])
def test_causal_queries(Lq, T):
    run(1, 8, 2, Lq, T, 128, seed=Lq + T)


@pytest.mark.parametrize("D", [64, 256])
def test_head_widths(D):
    run(2, 4, 4, 1, 333, D, seed=D)


def test_u8_values_and_batches():
    run(3, 16, 2, 2, 513, 128, bits=8, seed=5)


def test_not_causal_and_sharp_scores():
    run(1, 4, 1, 3, 200, 128, causal=False, seed=6, qscale=4.0)


def test_decode_full_cache():
    # the bench's 32768-key decode over 8 KV heads of 128 (40 query heads)
    run(1, 40, 8, 1, 32768, 128, seed=32768)
