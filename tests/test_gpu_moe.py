"""GPU parity of the top-k MoE expert gather (gate+up SiLU and down+combine)
against the CPU oracle, at the MoE workload's shapes (hidden 2048, 256
experts, expert intermediate 512, top-8, M = 1..8) and on edge cases."""
import numpy as np
import pytest
import torch

import group_wise_affine_gb300 as gwa
import gwa_synth as synth
import oracle
from helpers import bf16_to_f64, dev_bf16, dev_qweight

pytestmark = pytest.mark.gpu
TOL = 1e-2
H, E, I, TOPK = 2048, 256, 512, 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gwa.build()
    gwa.load()


def assert_close(got, ref, what=""):
    ok, max_err, worst = oracle.within_tolerance(got, ref, TOL)
    assert ok, f"{what}: max |err| {max_err:.3g}, worst err/bound {worst:.3g}"


def experts(seed, n_exp, rows, K, bits=4):
    return synth.stack_rows([synth.qweight(seed + e, rows, K, bits)
                             for e in range(n_exp)])


@pytest.fixture(scope="module")
def moe_weights():
    gu = experts(1_000_000, E, 2 * I, H)
    dn = experts(2_000_000, E, H, I)
    return (gu, dn, gwa.expert_view(dev_qweight(gu), E),
            gwa.expert_view(dev_qweight(dn), E))


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
def test_gate_up_config(moe_weights, M):
    gu, _, dgu, _ = moe_weights
    x = synth.activations(synth.seed_for(4, 2, M), M, H)
    ids, _ = synth.routing(synth.seed_for(4, 3, M), M, TOPK, E)
    out = gwa.moe_qmv_gather(dev_bf16(x), torch.from_numpy(ids).cuda(), dgu,
                             E, gwa.GWA_MOE_GATE_UP_SILU)
    ref = oracle.moe_gate_up_silu(x, ids, gu.wq, gu.scales, gu.biases, E,
                                  2 * I, H, 4)
    assert out.shape == (M, TOPK, I)
    assert_close(bf16_to_f64(out), ref, f"moe gate_up M={M}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_down_combine_config(moe_weights, M):
    _, dn, _, ddn = moe_weights
    ids, rw = synth.routing(synth.seed_for(4, 4, M), M, TOPK, E)
    hin = synth.activations(synth.seed_for(4, 5, M), M * TOPK, I).reshape(
        M, TOPK, I)
    out = gwa.moe_qmv_gather(dev_bf16(hin), torch.from_numpy(ids).cuda(), ddn,
                             E, gwa.GWA_MOE_DOWN_COMBINE,
                             route_w=torch.from_numpy(rw).cuda())
    ref = oracle.moe_down_combine(hin, ids, rw, dn.wq, dn.scales, dn.biases,
                                  E, H, I, 4)
    assert out.shape == (M, H)
    assert_close(bf16_to_f64(out), ref, f"moe down M={M}")


def test_chain_gate_up_then_down(moe_weights):
    gu, dn, dgu, ddn = moe_weights
    M = 4
    x = synth.activations(synth.seed_for(4, 6, 0), M, H)
    ids, rw = synth.routing(synth.seed_for(4, 7, 0), M, TOPK, E)
    dids = torch.from_numpy(ids).cuda()
    h = gwa.moe_qmv_gather(dev_bf16(x), dids, dgu, E,
                           gwa.GWA_MOE_GATE_UP_SILU)
    y = gwa.moe_qmv_gather(h, dids, ddn, E, gwa.GWA_MOE_DOWN_COMBINE,
                           route_w=torch.from_numpy(rw).cuda())
    # the oracle runs its own chain: its fp64 h, rounded to bf16, feeds down
    href = oracle.moe_gate_up_silu(x, ids, gu.wq, gu.scales, gu.biases, E,
                                   2 * I, H, 4)
    hbits = synth.bf16_bits(href.astype(np.float32))
    yref = oracle.moe_down_combine(hbits, ids, rw, dn.wq, dn.scales,
                                   dn.biases, E, H, I, 4)
    assert_close(bf16_to_f64(y), yref, "chain")


@pytest.mark.parametrize("bits", [4, 8])
def test_repeated_experts_and_ragged_shapes(bits):
    # ids repeat across and within tokens; K and rows off the tile sizes
    n_exp, K, I2, N = 6, 576, 2 * 75, 133
    gu = experts(700, n_exp, I2, K, bits)
    dn = experts(720, n_exp, N, 192, bits)
    ids = np.array([[3, 3, 5], [5, 1, 3], [0, 5, 5]], np.int32)
    M, topk = ids.shape
    x = synth.activations(730, M, K)
    out = gwa.moe_qmv_gather(dev_bf16(x), torch.from_numpy(ids).cuda(),
                             gwa.expert_view(dev_qweight(gu), n_exp), n_exp, 0)
    ref = oracle.moe_gate_up_silu(x, ids, gu.wq, gu.scales, gu.biases, n_exp,
                                  I2, K, bits)
    assert_close(bf16_to_f64(out), ref, "gate_up repeats")
    rw = np.array([[0.5, 0.25, 0.25], [0.1, 0.2, 0.7], [1.0, 0.0, -0.5]],
                  np.float32)
    hin = synth.activations(731, M * topk, 192).reshape(M, topk, 192)
    y = gwa.moe_qmv_gather(dev_bf16(hin), torch.from_numpy(ids).cuda(),
                           gwa.expert_view(dev_qweight(dn), n_exp), n_exp, 1,
                           route_w=torch.from_numpy(rw).cuda())
    yref = oracle.moe_down_combine(hin, ids, rw, dn.wq, dn.scales, dn.biases,
                                   n_exp, N, 192, bits)
    assert_close(bf16_to_f64(y), yref, "down repeats")


def test_top1_unit_weight_matches_plain_projection():
    n_exp, N, K = 4, 256, 512
    dn = experts(800, n_exp, N, K)
    ids = np.array([[2], [0], [2]], np.int32)
    hin = synth.activations(801, 3, K).reshape(3, 1, K)
    y = gwa.moe_qmv_gather(dev_bf16(hin), torch.from_numpy(ids).cuda(),
                           gwa.expert_view(dev_qweight(dn), n_exp), n_exp, 1,
                           route_w=torch.ones((3, 1), device="cuda"))
    for t, e in enumerate((2, 0, 2)):
        sl = slice(e * N, (e + 1) * N)
        part = synth.QWeight(dn.wq[sl], dn.scales[sl], dn.biases[sl], N, K, 4)
        plain = gwa.qmv_affine(dev_bf16(hin[t, 0][None]), dev_qweight(part))
        assert_close(bf16_to_f64(y[t:t + 1]), bf16_to_f64(plain), "top1")


def test_out_of_range_expert_sets_status_and_contributes_zero():
    n_exp, K, I2 = 3, 128, 64
    gu = experts(900, n_exp, I2, K)
    ids = np.array([[1, 7], [-1, 2]], np.int32)
    x = synth.activations(901, 2, K)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gwa.moe_qmv_gather(dev_bf16(x), torch.from_numpy(ids).cuda(),
                             gwa.expert_view(dev_qweight(gu), n_exp), n_exp, 0,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    o = bf16_to_f64(out)
    assert np.all(o[0, 1] == 0) and np.all(o[1, 0] == 0)
    good = np.array([[1], [2]], np.int32)
    ref = oracle.moe_gate_up_silu(x, good, gu.wq, gu.scales, gu.biases, n_exp,
                                  I2, K, 4)
    assert_close(o[0, 0], ref[0, 0])
    assert_close(o[1, 1], ref[1, 0])
    # down: the bad slots are skipped, the rest combine as usual
    dn = experts(910, n_exp, 96, K)
    hin = synth.activations(911, 4, K).reshape(2, 2, K)
    rw = np.array([[0.6, 0.4], [0.3, 0.7]], np.float32)
    status.zero_()
    y = gwa.moe_qmv_gather(dev_bf16(hin), torch.from_numpy(ids).cuda(),
                           gwa.expert_view(dev_qweight(dn), n_exp), n_exp, 1,
                           route_w=torch.from_numpy(rw).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    y0 = oracle.moe_down_combine(hin[0:1, 0:1], np.array([[1]], np.int32),
                                 rw[0:1, 0:1], dn.wq, dn.scales, dn.biases,
                                 n_exp, 96, K, 4)
    y1 = oracle.moe_down_combine(hin[1:2, 1:2], np.array([[2]], np.int32),
                                 rw[1:2, 1:2], dn.wq, dn.scales, dn.biases,
                                 n_exp, 96, K, 4)
    assert_close(bf16_to_f64(y[0:1]), y0, "down bad slot 0")
    assert_close(bf16_to_f64(y[1:2]), y1, "down bad slot 1")


def _valid_refs(ids, n_exp):
    """ids with out-of-range entries replaced by expert 0, and the mask of
    the valid slots (the oracle takes only valid ids)."""
    valid = (ids >= 0) & (ids < n_exp)
    return np.where(valid, ids, 0).astype(np.int32), valid


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K", [512, 1024, 2048])
def test_streaming_repeats_invalid_ragged(bits, K):
    # K/64 = 8, 16, 32 groups (one 8-, 16- or 32-lane slice per row); ids
    # repeat within and across tokens and include out-of-range entries;
    # rows per expert off every stage size
    n_exp, I2, N = 7, 2 * 75, 133
    gu = experts(1000 + K + bits, n_exp, I2, K, bits)
    dn = experts(1100 + K + bits, n_exp, N, K, bits)
    ids = np.array([[3, 3, 5, 9], [5, 1, 3, -2], [0, 5, 5, 6]], np.int32)
    M, topk = ids.shape
    good, valid = _valid_refs(ids, n_exp)
    dids = torch.from_numpy(ids).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = synth.activations(1200 + K, M, K)
    out = gwa.moe_qmv_gather(dev_bf16(x), dids,
                             gwa.expert_view(dev_qweight(gu), n_exp), n_exp, 0,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    ref = oracle.moe_gate_up_silu(x, good, gu.wq, gu.scales, gu.biases, n_exp,
                                  I2, K, bits)
    ref[~valid] = 0.0
    o = bf16_to_f64(out)
    assert np.all(o[~valid] == 0)
    assert_close(o, ref, f"gate_up stream K={K} u{bits}")
    rw = synth.bf16_values(synth.activations(1300 + K, M, topk)).copy()
    hin = synth.activations(1400 + K, M * topk, K).reshape(M, topk, K)
    status.zero_()
    y = gwa.moe_qmv_gather(dev_bf16(hin), dids,
                           gwa.expert_view(dev_qweight(dn), n_exp), n_exp, 1,
                           route_w=torch.from_numpy(rw).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    yref = oracle.moe_down_combine(hin, good, np.where(valid, rw, 0.0), dn.wq,
                                   dn.scales, dn.biases, n_exp, N, K, bits)
    assert_close(bf16_to_f64(y), yref, f"down stream K={K} u{bits}")


def test_streaming_is_deterministic(moe_weights):
    _, _, dgu, ddn = moe_weights
    M = 8
    ids, rw = synth.routing(synth.seed_for(4, 8, 0), M, TOPK, E)
    dids = torch.from_numpy(ids).cuda()
    x = dev_bf16(synth.activations(synth.seed_for(4, 9, 0), M, H))
    h1 = gwa.moe_qmv_gather(x, dids, dgu, E, gwa.GWA_MOE_GATE_UP_SILU)
    h2 = gwa.moe_qmv_gather(x, dids, dgu, E, gwa.GWA_MOE_GATE_UP_SILU)
    assert torch.equal(h1, h2)
    r = torch.from_numpy(rw).cuda()
    y1 = gwa.moe_qmv_gather(h1, dids, ddn, E, gwa.GWA_MOE_DOWN_COMBINE,
                            route_w=r)
    y2 = gwa.moe_qmv_gather(h1, dids, ddn, E, gwa.GWA_MOE_DOWN_COMBINE,
                            route_w=r)
    assert torch.equal(y1, y2)


def test_long_rows_use_the_staged_kernels():
    # K = 2560 (40 groups) is past the streaming kernel's slice
    n_exp, K, I2, N = 3, 2560, 2 * 40, 72
    gu = experts(1500, n_exp, I2, K)
    dn = experts(1510, n_exp, N, K)
    ids = np.array([[2, 0], [1, 2]], np.int32)
    M, topk = ids.shape
    x = synth.activations(1520, M, K)
    out = gwa.moe_qmv_gather(dev_bf16(x), torch.from_numpy(ids).cuda(),
                             gwa.expert_view(dev_qweight(gu), n_exp), n_exp, 0)
    ref = oracle.moe_gate_up_silu(x, ids, gu.wq, gu.scales, gu.biases, n_exp,
                                  I2, K, 4)
    assert_close(bf16_to_f64(out), ref, "gate_up long rows")
    rw = np.array([[0.75, 0.25], [0.5, 0.5]], np.float32)
    hin = synth.activations(1521, M * topk, K).reshape(M, topk, K)
    y = gwa.moe_qmv_gather(dev_bf16(hin), torch.from_numpy(ids).cuda(),
                           gwa.expert_view(dev_qweight(dn), n_exp), n_exp, 1,
                           route_w=torch.from_numpy(rw).cuda())
    yref = oracle.moe_down_combine(hin, ids, rw, dn.wq, dn.scales, dn.biases,
                                   n_exp, N, K, 4)
    assert_close(bf16_to_f64(y), yref, "down long rows")
