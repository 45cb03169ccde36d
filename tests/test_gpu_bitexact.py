"""Code unpacking and dequantization pinned bit for bit through the
production kernels, not only the debug exports.

With one-hot activations (token m has 1.0 at input k_m and zeros elsewhere)
a projection returns, exactly, each row's dequantized weight at k_m rounded
to bf16: the integer-dot kernels form s * q + b with one rounding (fmaf), the
tensor-core kernels form s * q and the bias term exactly and add them in
fp32, and every other group contributes exact zeros.  So for every kernel
route:
  * scale 1, bias 0:         y[m, n] == q[n, k_m]             (the code itself)
  * bf16 scales and biases:  y[m, n] == bf16_rn(fp32(s q + b)) (the oracle's
                             dequantized value, exact in fp32 here, rounded)
checked against oracle.unpack / oracle.dequant.  The positions k_m sweep
every slot of a word and of a group.  Gate+up: a gate bias of 32 makes
SiLU(g) = g exactly in fp32 (e^-g < 2^-25), so h = g * u pins both halves'
codes.  MoE down: top-1 with route weight 1.
"""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from helpers import dev_bf16, dev_qweight, host_u16

pytestmark = pytest.mark.gpu
ONE = 0x3F80  # bf16 1.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()
    assert torch.cuda.is_available()


def unit_affine(w):
    """The same codes with scale 1 and bias 0."""
    G = w.K // w.group
    return synth.QWeight(w.wq, np.full((w.N, G), ONE, np.uint16),
                         np.zeros((w.N, G), np.uint16), w.N, w.K, w.bits,
                         w.group)


def one_hot(positions, K):
    x = np.zeros((len(positions), K), np.uint16)
    for m, k in enumerate(positions):
        x[m, k] = ONE
    return x


def expected(w, positions):
    """bf16 bits of the dequantized weights at the given inputs, [M, N]."""
    deq = oracle.dequant(w.wq, w.scales, w.biases, w.N, w.K, w.bits, w.group)
    cols = deq[:, positions].T.astype(np.float32)  # fp32: s q + b is exact here
    return synth.bf16_bits(cols)


def sweep(K, group, M, extra=()):
    """Batches of M one-hot positions covering every slot of the first group
    (so every slot of a word) and a few in later groups."""
    pos = list(range(min(group, K))) + [k for k in extra if k < K]
    return [pos[i:i + M] for i in range(0, len(pos), M)]


def check_plain(w, M, what, ws_tokens=None):
    dw = dev_qweight(w)
    for batch in sweep(w.K, w.group, M, extra=(w.K // 2 + 3, w.K - 1)):
        x = one_hot(batch, w.K)
        ws = gwa.make_workspace(len(batch), w.K)
        y = gwa.qmv_affine(dev_bf16(x), dw, workspace=ws)
        torch.cuda.synchronize()
        got = host_u16(y)
        want = expected(w, batch)
        bad = np.argwhere(got != want)
        assert bad.size == 0, (f"{what}: {len(bad)} mismatches, first at "
                               f"token {bad[0][0]} (k={batch[bad[0][0]]}) row "
                               f"{bad[0][1]}: got {got[tuple(bad[0])]:#06x} "
                               f"want {want[tuple(bad[0])]:#06x}")


# kernel routes by token count and shape (see the dispatcher): one token
# (chunk per lane), 2..4 (streaming), 5..8 (tensor-core decode), 5..8 with u8
# rows longer than 5120 (clusters along K), K off 512 (staged), M > 8
# (tcgen05; K off 512 falls back to the decode kernels in passes)
ROUTES = [
    ("one-token", 1, 128, 1024),
    ("streaming", 4, 128, 1024),
    ("streaming-3", 3, 64, 1024),
    ("mma", 8, 128, 1024),
    ("staged", 4, 67, 576),
    ("staged-1", 1, 67, 576),
    ("tcgen05", 16, 256, 1024),
]


@pytest.mark.parametrize("route,M,N,K", ROUTES)
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("unit", [True, False])
def test_one_hot_reads_dequantized_weights(route, M, N, K, bits, unit):
    w = synth.qweight(7100 + N + bits, N, K, bits)
    if unit:
        w = unit_affine(w)
        # the oracle's codes are the expected outputs themselves
        codes = oracle.unpack(w.wq, N, K, bits)
        assert np.array_equal(synth.bf16_values(expected(w, [0, 1]))[0],
                              codes[:, 0].astype(np.float32))
    check_plain(w, M, f"{route} u{bits} unit={unit}")


@pytest.mark.parametrize("M", [6, 8])
def test_one_hot_cluster_split(M):
    # u8 rows longer than 5120 inputs at 5..8 tokens: clusters along K; the
    # positions straddle the CTAs' K ranges
    K, N = 13824, 64
    w = synth.qweight(7200, N, K, 8)
    dw = dev_qweight(w)
    pos = [0, 1, 2, 3, 4607, 4608, 4609, 9215, 9216, 13823, 6000, 77]
    for i in range(0, len(pos), M):
        batch = pos[i:i + M]
        y = gwa.qmv_affine(dev_bf16(one_hot(batch, K)), dw)
        torch.cuda.synchronize()
        assert np.array_equal(host_u16(y), expected(w, batch)), f"cluster {batch}"


@pytest.mark.parametrize("bits,group,M", [(2, 64, 1), (3, 64, 2), (6, 64, 3),
                                          (2, 32, 4), (3, 128, 1), (6, 128, 4),
                                          (4, 32, 1), (4, 128, 1), (8, 32, 2),
                                          (8, 128, 3)])
def test_one_hot_general_widths(bits, group, M):
    N, K = 96, 768
    w = synth.qweight(7300 + bits * 10 + group, N, K, bits, group)
    check_plain(w, M, f"u{bits} g{group} M={M}")
    check_plain(unit_affine(w), M, f"u{bits} g{group} M={M} unit")


def gate_up_weight(seed, I, K, bits):
    """Gate rows: scale 1, bias 32 (so SiLU(g) = g exactly in fp32); up
    rows: scale 1, bias 0."""
    w = synth.qweight(seed, 2 * I, K, bits)
    G = K // 64
    s = np.full((2 * I, G), ONE, np.uint16)
    b = np.zeros((2 * I, G), np.uint16)
    b[:I] = 0x4200  # bf16 32.0
    return synth.QWeight(w.wq, s, b, 2 * I, K, bits)


def expected_gate_up(w, positions):
    I = w.N // 2
    deq = oracle.dequant(w.wq, w.scales, w.biases, w.N, w.K, w.bits)
    g = deq[:I, positions].T
    u = deq[I:, positions].T
    return synth.bf16_bits((g * u).astype(np.float32))  # exact in fp32


@pytest.mark.parametrize("M", [1, 3, 8, 16])
@pytest.mark.parametrize("bits", [4, 8])
def test_one_hot_gate_up(M, bits):
    I, K = 128, 1024
    w = gate_up_weight(7400 + bits, I, K, bits)
    dw = dev_qweight(w)
    for batch in sweep(K, 64, M, extra=(700,)):
        ws = gwa.make_workspace(len(batch), K)
        h = gwa.qmv_gate_up_silu(dev_bf16(one_hot(batch, K)), dw, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(host_u16(h), expected_gate_up(w, batch)), \
            f"gate+up M={M} u{bits} {batch}"


@pytest.mark.parametrize("M", [1, 2, 8])
@pytest.mark.parametrize("H", [512, 4096])
def test_one_hot_moe(M, H):
    # gate+up: every token routed to one expert; down: top-1, weight 1
    E, I = 4, 64
    parts = [gate_up_weight(7500 + e, I, H, 4) for e in range(E)]
    gu = synth.stack_rows(parts)
    ids = (np.arange(M, dtype=np.int32) % E).reshape(M, 1)
    dgu = gwa.expert_view(dev_qweight(gu), E)
    for batch in sweep(H, 64, M, extra=(H - 1,)):
        bm = len(batch)
        h = gwa.moe_qmv_gather(dev_bf16(one_hot(batch, H)),
                               torch.from_numpy(ids[:bm].copy()).cuda(), dgu, E,
                               gwa.GWA_MOE_GATE_UP_SILU)
        torch.cuda.synchronize()
        got = host_u16(h).reshape(bm, I)
        for t in range(bm):
            want = expected_gate_up(parts[int(ids[t, 0])], [batch[t]])[0]
            assert np.array_equal(got[t], want), f"moe gate+up H={H} k={batch[t]}"
    dn = synth.stack_rows([synth.qweight(7600 + e, H, I, 4) for e in range(E)])
    ddn = gwa.expert_view(dev_qweight(dn), E)
    for batch in sweep(I, 64, M):
        bm = len(batch)
        y = gwa.moe_qmv_gather(dev_bf16(one_hot(batch, I).reshape(bm, 1, I)),
                               torch.from_numpy(ids[:bm].copy()).cuda(), ddn, E,
                               gwa.GWA_MOE_DOWN_COMBINE,
                               route_w=torch.ones((bm, 1), device="cuda"))
        torch.cuda.synchronize()
        got = host_u16(y)
        for t in range(bm):
            e = int(ids[t, 0])
            part = synth.QWeight(dn.wq[e * H:(e + 1) * H],
                                 dn.scales[e * H:(e + 1) * H],
                                 dn.biases[e * H:(e + 1) * H], H, I, 4)
            assert np.array_equal(got[t], expected(part, [batch[t]])[0]), \
                f"moe down H={H} k={batch[t]}"
