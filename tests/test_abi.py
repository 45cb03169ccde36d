"""The C ABI without a GPU: the library builds, loads, exports every entry
point include/gwa.h declares, and rejects bad arguments with a status code
before touching the device."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gwa.h")

needs_nvcc = pytest.mark.skipif(
    shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
    reason="nvcc not available")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gwa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import group_wise_affine_gb300 as gwa
    gwa.build()
    return gwa.load()


def test_header_declares_the_four_projections():
    names = declared_functions()
    for want in ("gwa_qmv_affine", "gwa_qmv_fused_sections",
                 "gwa_qmv_gate_up_silu", "gwa_moe_qmv_gather",
                 "gwa_last_error", "gwa_workspace_bytes"):
        assert want in names


@needs_nvcc
def test_library_exports_every_declared_symbol(lib):
    import group_wise_affine_gb300 as gwa
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(gwa.EXPORTS) <= set(declared_functions())


def _qw(gwa, bits=4, group=64, N=16, K=128, wq=0x1000, sc=0x2000, bi=0x3000):
    # fake device addresses: validation must reject before any dereference
    return gwa._QW(wq, sc, bi, N, K, bits, group)


@needs_nvcc
@pytest.mark.parametrize("kw,code", [
    (dict(bits=5), 2), (dict(bits=7), 2), (dict(group=48), 2),
    (dict(group=256), 2),
    (dict(K=100), 1), (dict(K=0), 1), (dict(N=-1), 1),
    (dict(wq=0x1004), 3), (dict(sc=0x2001), 3),
])
def test_bad_weight_is_rejected_without_a_gpu(lib, kw, code):
    import group_wise_affine_gb300 as gwa
    rc = lib.gwa_qmv_affine(0x4000, 1, _qw(gwa, **kw), 0x5000, None, 0, None)
    assert rc == code
    assert lib.gwa_last_error().decode()


@needs_nvcc
def test_bad_activations_and_sections_are_rejected(lib):
    import group_wise_affine_gb300 as gwa
    w = _qw(gwa)
    assert lib.gwa_qmv_affine(0x4008, 1, w, 0x5000, None, 0, None) == 3
    assert lib.gwa_qmv_affine(None, 1, w, 0x5000, None, 0, None) == 1
    assert lib.gwa_qmv_affine(0x4000, -1, w, 0x5000, None, 0, None) == 1
    sizes = (ctypes.c_int64 * 3)(8, 4, 3)          # adds to 15, not 16
    outs = (ctypes.c_void_p * 3)(0x6000, 0x7000, 0x8000)
    rc = lib.gwa_qmv_fused_sections(0x4000, 1, w, 3,
                                    ctypes.cast(sizes, ctypes.c_void_p),
                                    ctypes.cast(outs, ctypes.c_void_p), None,
                                    None, 0, None)
    assert rc == 1 and "add up" in lib.gwa_last_error().decode()
    assert lib.gwa_qmv_fused_sections(0x4000, 1, w, 9,
                                      ctypes.cast(sizes, ctypes.c_void_p),
                                      ctypes.cast(outs, ctypes.c_void_p), None,
                                      None, 0, None) == 1
    odd = _qw(gwa, N=15)
    assert lib.gwa_qmv_gate_up_silu(0x4000, 1, odd, 0x5000, None, 0, None) == 1


@needs_nvcc
def test_moe_arguments_are_checked(lib):
    import group_wise_affine_gb300 as gwa
    w = _qw(gwa, N=8)
    call = lambda **k: lib.gwa_moe_qmv_gather(
        k.get("x", 0x4000), k.get("M", 1), k.get("topk", 2),
        k.get("ids", 0x9000), k.get("rw", 0xA000), w, k.get("E", 4),
        k.get("mode", 0), k.get("out", 0xB000), None, None)
    assert call(mode=2) == 1
    assert call(topk=0) == 1
    assert call(E=0) == 1
    assert call(M=9) == 2
    assert call(mode=1, rw=None) == 1
    assert call(ids=0x9002) == 3


@needs_nvcc
def test_empty_problems_are_no_ops(lib):
    import group_wise_affine_gb300 as gwa
    # M == 0 or N == 0: nothing to do, nothing enqueued, no device needed
    assert lib.gwa_qmv_affine(0x4000, 0, _qw(gwa), 0x5000, None, 0, None) == 0
    assert lib.gwa_qmv_affine(0x4000, 1, _qw(gwa, N=0), None, None, 0,
                              None) == 0
    assert lib.gwa_workspace_bytes(1, 5120) == 0


def test_binding_refuses_mismatched_sizes_before_any_call():
    # Size checks run before any pointer is taken, so CPU tensors suffice.
    import torch
    import group_wise_affine_gb300 as gwa
    N, K = 8, 128
    wq = torch.zeros((N, K // 8), dtype=torch.int32)
    s = torch.zeros((N, K // 64), dtype=torch.bfloat16)
    w = gwa.QWeight(wq, s, s, N, K, 4, 64)
    x = torch.zeros((1, K), dtype=torch.bfloat16)
    bad = gwa.QWeight(wq, s, s, N * 4, K, 4, 64)        # claims 4x the rows
    with pytest.raises(ValueError):
        gwa.qmv_affine(x, bad, y=torch.zeros((1, 4 * N), dtype=torch.bfloat16))
    with pytest.raises(ValueError):                     # output too small
        gwa.qmv_affine(x, w, y=torch.zeros((1, N - 1), dtype=torch.bfloat16))
    with pytest.raises(ValueError):                     # stacked experts: N per expert
        gwa.moe_qmv_gather(x, torch.zeros((1, 2), dtype=torch.int32), w, 4, 0,
                           out=torch.zeros((1, 2, N // 2),
                                           dtype=torch.bfloat16))
    per_expert = gwa.expert_view(w, 4)
    assert per_expert.N == 2


@needs_nvcc
def test_quantize_arguments_are_checked(lib):
    q = lambda **k: lib.gwa_quantize_affine(
        k.get("w", 0x4000), k.get("N", 8), k.get("K", 128), k.get("bits", 4),
        k.get("group", 64), k.get("wq", 0x1000), k.get("sc", 0x2000),
        k.get("bi", 0x3000), None)
    assert q(bits=3) == 2
    assert q(group=32) == 2
    assert q(K=100) == 1
    assert q(N=-1) == 1
    assert q(w=None) == 1
    assert q(w=0x4008) == 3
    assert q(wq=0x1004) == 3
    assert q(sc=0x2001) == 3
    assert q(N=0) == 0   # nothing to do, no device needed


@needs_nvcc
def test_qkv_rope_arguments_are_checked(lib):
    import group_wise_affine_gb300 as gwa
    w = _qw(gwa, N=256, K=128)   # q 128 + 2 * kv 64
    call = lambda **k: lib.gwa_qmv_qkv_rope(
        0x4000, k.get("M", 1), w, k.get("q", 128), k.get("kv", 64),
        k.get("d", 64), k.get("base", 10000.0), k.get("pos", 0x9000),
        0x5000, 0x6000, 0x7000, None, None, 0, None)
    assert call(d=63) == 1          # odd head_dim
    assert call(d=512) == 1         # too wide
    assert call(q=96) == 1          # q + 2 kv != N
    assert call(kv=48, q=160) == 1  # not a multiple of head_dim
    assert call(base=0.0) == 1
    assert call(pos=None) == 1
    assert call(pos=0x9002) == 3
    assert call(M=0) == 0           # nothing to do, no device needed


@needs_nvcc
def test_formats_outside_the_tuned_kernels_are_refused_where_unsupported(lib):
    import group_wise_affine_gb300 as gwa
    # experts and quantization: u4/u8 at group 64 only
    w2 = _qw(gwa, bits=2, N=8)
    assert lib.gwa_moe_qmv_gather(0x4000, 1, 2, 0x9000, None, w2, 4, 0,
                                  0xB000, None, None) == 2
    assert lib.gwa_quantize_affine(0x4000, 8, 128, 4, 32, 0x1000, 0x2000,
                                   0x3000, None) == 2
    # u2 and groups of 32 / 128 are accepted by the projections (empty call)
    for bits, group in ((2, 64), (4, 32), (8, 128)):
        assert lib.gwa_qmv_affine(0x4000, 0, _qw(gwa, bits=bits, group=group),
                                  0x5000, None, 0, None) == 0



@needs_nvcc
def test_attention_arguments_are_checked(lib):
    call = lambda **a: lib.gwa_sdpa_dequant_v(
        a.get("q", 0x4000), a.get("B", 1), a.get("Hq", 8), a.get("Lq", 1),
        a.get("D", 128), 0x5000, a.get("Hkv", 2), a.get("T", 16),
        a.get("vq", 0x6000), 0x7000, 0x8000, a.get("bits", 4),
        a.get("group", 64), 0.1, a.get("causal", 1), 0x9000, None, 0, None)
    assert call(D=96) == 2
    assert call(bits=2) == 2
    assert call(group=32) == 2
    assert call(Hq=6, Hkv=4) == 1        # Hq not a multiple of Hkv
    assert call(T=0) == 1
    assert call(Lq=20, T=16) == 1        # causal: a query would see no key
    assert call(q=None) == 1
    assert call(vq=0x6004) == 3
    assert call(q=0x4008) == 3           # q and k need 16 bytes
    assert call() == 5                   # no workspace
    assert call(Lq=0) == 0               # nothing to do
    assert lib.gwa_sdpa_workspace_bytes(1, 8, 2, 1, 16, 128) > 0
