"""GPU parity of the affine quantization kernel against the CPU oracle.

The code is an integer decided in floating point; kernel and oracle both
decide it in IEEE fp32 (the reading of the requantize step of "Sanctum-MLX",
"The April 2026 cutover"), so codes, scales and biases must agree bit for
bit.  Sizes span several warps' worth of groups with ragged ends, the edge
groups the rule has (constant, two-valued, zero minimum of either sign, halfway
values, extreme and subnormal ranges), and the full gate+up shape on sampled
rows.
"""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import oracle
from helpers import dev_bf16, host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()
    assert torch.cuda.is_available()


def to_bf16_rn(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def check_exact(w_u16, bits):
    N, K = w_u16.shape
    got = gwa.quantize_affine(dev_bf16(w_u16), bits=bits)
    torch.cuda.synchronize()
    wq, sc, bi = oracle.quantize_affine(w_u16, N, K, bits)
    np.testing.assert_array_equal(got.wq.cpu().numpy().view(np.uint32), wq)
    np.testing.assert_array_equal(host_u16(got.scales), sc)
    np.testing.assert_array_equal(host_u16(got.biases), bi)
    return got


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,K", [(1, 64), (3, 128), (37, 640), (130, 5120),
                                 (5, 13824)])
def test_matches_the_oracle_bit_for_bit(bits, N, K):
    rng = np.random.default_rng(1000 * bits + N + K)
    w = to_bf16_rn(rng.normal(0, 0.05, size=(N, K)).astype(np.float32))
    check_exact(w, bits)


@pytest.mark.parametrize("bits", [4, 8])
def test_edge_groups(bits):
    qmax = (1 << bits) - 1
    rng = np.random.default_rng(77 + bits)
    groups = []
    groups.append(np.full(64, -3.5))                                 # constant
    groups.append(np.where(np.arange(64) % 2 == 0, -1.0, 2.0))       # two values
    z = np.zeros(64); z[3] = 1.0; z[0] = -0.0; groups.append(z)      # -0 first
    z = np.zeros(64); z[3] = 1.0; z[9] = -0.0; groups.append(z)      # +0 first
    h = np.zeros(64); h[1] = qmax; h[2:8] = [0.5, 1.5, 2.5, 3.25, 3.75, 4.5]
    groups.append(h)                                                 # halfway
    groups.append(rng.normal(0, 1, 64) * 1e30)                       # huge
    groups.append(rng.normal(0, 1, 64) * 1e-37)                      # tiny scale
    groups.append(np.abs(rng.normal(0, 1, 64)) * 1e-39)              # subnormals
    groups.append(-np.abs(rng.normal(0, 1, 64)) - 5.0)               # negative
    m = rng.normal(0, 1, 64); m[0] = 1e20; m[1] = -1e-20; groups.append(m)
    w = to_bf16_rn(np.stack(groups).astype(np.float32)).reshape(1, -1)
    check_exact(w, bits)


@pytest.mark.parametrize("bits", [4, 8])
def test_full_gate_up_shape_on_sampled_rows(bits):
    N, K = 27648, 5120
    g = torch.Generator(device="cuda").manual_seed(31 + bits)
    w = (torch.randn((N, K), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    got = gwa.quantize_affine(w, bits=bits)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 1, N // 2, N - 2, N - 1],
                                     np.random.default_rng(5).integers(0, N, 40)]))
    idx = torch.from_numpy(rows).cuda()
    w_rows = host_u16(w.index_select(0, idx))
    wq, sc, bi = oracle.quantize_affine(w_rows, len(rows), K, bits)
    np.testing.assert_array_equal(
        got.wq.index_select(0, idx).cpu().numpy().view(np.uint32), wq)
    np.testing.assert_array_equal(host_u16(got.scales.index_select(0, idx)), sc)
    np.testing.assert_array_equal(host_u16(got.biases.index_select(0, idx)), bi)


@pytest.mark.parametrize("bits", [4, 8])
def test_quantized_weights_feed_the_projection(bits):
    """Quantize on the GPU, project with the result: the output matches the
    oracle's projection with the oracle's quantization of the same weights."""
    N, K = 256, 1024
    rng = np.random.default_rng(3 + bits)
    w = to_bf16_rn(rng.normal(0, 0.05, size=(N, K)).astype(np.float32))
    x = to_bf16_rn(rng.normal(0, 1, size=(2, K)).astype(np.float32))
    qw = gwa.quantize_affine(dev_bf16(w), bits=bits)
    y = gwa.qmv_affine(dev_bf16(x), qw)
    torch.cuda.synchronize()
    wq, sc, bi = oracle.quantize_affine(w, N, K, bits)
    ref = oracle.qmv(x, wq, sc, bi, N, K, bits)
    ok, max_err, worst = oracle.within_tolerance(
        y.float().cpu().numpy().astype(np.float64), ref, 1e-2)
    assert ok, (max_err, worst)


def test_empty_weight():
    out = gwa.quantize_affine(torch.empty((0, 128), dtype=torch.bfloat16,
                                          device="cuda"), bits=4)
    assert out.wq.shape == (0, 16) and out.scales.shape == (0, 2)
