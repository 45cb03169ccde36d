"""Python binding of libgwa.so: affine group-quantized projections on GB300.

Argument marshalling only: every function below checks tensor placement and
dtypes, passes raw device pointers, sizes and the current CUDA stream to the
C ABI (``include/gwa.h``) and raises ``GwaError`` on a non-zero status.  All
arithmetic runs in the library's sm_103a kernels.  There is no fallback: if
``_build/libgwa.so`` is missing, every call raises.

Names mirror the C entry points without the ``gwa_`` prefix:
``qmv_affine``, ``qmv_fused_sections``, ``qmv_gate_up_silu``,
``qmv_qkv_rope``, ``moe_qmv_gather``, ``quantize_affine``, ``sdpa_dequant_v``,
``workspace_bytes``, ``last_error``,
``debug_unpack``, ``debug_dequant``.

Weights: ``wq`` int32 [N, K*bits/32] (the packed uint32 words; fp8 weights,
``bits=GWA_FP8_E4M3``, hold four 8-bit codes a word), ``scales`` and
``biases`` bfloat16 [N, K/group].  Activations and outputs are bfloat16.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgwa.so")

GWA_OK = 0
GWA_ERR_INVALID_ARG = 1
GWA_ERR_UNSUPPORTED = 2
GWA_ERR_MISALIGNED = 3
GWA_ERR_CUDA = 4
GWA_ERR_WORKSPACE = 5
GWA_NOALLOC_SCRATCH_BYTES = 8 << 20
GWA_MOE_GATE_UP_SILU = 0
GWA_MOE_DOWN_COMBINE = 1
# ``bits`` of fp8 (e4m3) weights: 8-bit E4M3 codes in the affine container
GWA_FP8_E4M3 = 0x108


def code_bits(bits: int) -> int:
    """Stream bits of one code of a format (fp8: 8)."""
    return 8 if bits == GWA_FP8_E4M3 else bits

EXPORTS = ("gwa_qmv_affine", "gwa_qmv_fused_sections", "gwa_qmv_gate_up_silu",
           "gwa_workspace_bytes", "gwa_moe_qmv_gather", "gwa_last_error",
           "gwa_pipeline_status", "gwa_debug_unpack", "gwa_debug_dequant",
           "gwa_qmv_affine_noalloc", "gwa_quantize_affine", "gwa_qmv_qkv_rope",
           "gwa_qkv_rope_workspace_bytes", "gwa_sdpa_dequant_v",
           "gwa_sdpa_workspace_bytes", "gwa_debug_bounded_wait")


class GwaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"gwa status {code}: {msg}")
        self.code = code


class _QW(ctypes.Structure):
    _fields_ = [("wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("bits", ctypes.c_int32),
                ("group", ctypes.c_int32)]


_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA sources into _build/libgwa.so (nvcc, sm_103a)."""
    from . import builder
    return builder.build(force=force)


def load(path: str = LIB_PATH):
    """Load libgwa.so and declare its signatures; raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with group_wise_affine_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, i64, i32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                        ctypes.c_size_t)
    lib.gwa_qmv_affine.argtypes = [vp, i64, _QW, vp, vp, sz, vp]
    lib.gwa_qmv_fused_sections.argtypes = [vp, i64, _QW, i32, vp, vp, vp, vp,
                                           sz, vp]
    lib.gwa_qmv_gate_up_silu.argtypes = [vp, i64, _QW, vp, vp, sz, vp]
    lib.gwa_workspace_bytes.argtypes = [i64, i64]
    lib.gwa_workspace_bytes.restype = sz
    lib.gwa_moe_qmv_gather.argtypes = [vp, i64, i32, vp, vp, _QW, i32, i32, vp,
                                       vp, vp]
    lib.gwa_last_error.argtypes = []
    lib.gwa_last_error.restype = ctypes.c_char_p
    lib.gwa_qmv_affine_noalloc.argtypes = [vp, i64, _QW, vp, vp]
    lib.gwa_qmv_affine_noalloc.restype = ctypes.c_int
    lib.gwa_pipeline_status.argtypes = [vp, i32]
    lib.gwa_pipeline_status.restype = ctypes.c_int
    lib.gwa_quantize_affine.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp,
                                        vp]
    lib.gwa_qmv_qkv_rope.argtypes = [vp, i64, _QW, i64, i64, i32,
                                     ctypes.c_double, vp, vp, vp, vp, vp, vp,
                                     sz, vp]
    lib.gwa_qmv_qkv_rope.restype = ctypes.c_int
    lib.gwa_qkv_rope_workspace_bytes.argtypes = [i64, i64, i32]
    lib.gwa_qkv_rope_workspace_bytes.restype = sz
    lib.gwa_sdpa_dequant_v.argtypes = [vp, i64, i32, i32, i32, vp, i32, i64, vp,
                                       vp, vp, i32, i32, ctypes.c_float, i32,
                                       vp, vp, sz, vp]
    lib.gwa_sdpa_dequant_v.restype = ctypes.c_int
    lib.gwa_sdpa_workspace_bytes.argtypes = [i64, i32, i32, i32, i64, i32]
    lib.gwa_sdpa_workspace_bytes.restype = sz
    lib.gwa_quantize_affine.restype = ctypes.c_int
    lib.gwa_debug_unpack.argtypes = [_QW, vp, vp]
    lib.gwa_debug_dequant.argtypes = [_QW, vp, vp]
    lib.gwa_debug_bounded_wait.argtypes = [ctypes.c_uint32, vp, vp]
    for f in ("gwa_qmv_affine", "gwa_qmv_fused_sections",
              "gwa_qmv_gate_up_silu", "gwa_moe_qmv_gather",
              "gwa_debug_unpack", "gwa_debug_dequant",
              "gwa_debug_bounded_wait"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def last_error() -> str:
    return load().gwa_last_error().decode()


def pipeline_status(reset: bool = True) -> int:
    """Pipeline waits that ran out of time since the last reset (synchronizes
    the device)."""
    out = ctypes.c_uint32(0)
    _check(load().gwa_pipeline_status(ctypes.byref(out), int(reset)))
    return int(out.value)


def _check(rc: int) -> None:
    if rc != GWA_OK:
        raise GwaError(rc, last_error())


@dataclass
class QWeight:
    """A packed weight on the device (caller-owned tensors)."""
    wq: torch.Tensor       # int32 [N, K*bits/32]
    scales: torch.Tensor   # bfloat16 [N, K/group]
    biases: torch.Tensor   # bfloat16 [N, K/group]
    N: int
    K: int
    bits: int = 4
    group: int = 64

    def c(self) -> _QW:
        return _QW(_ptr(self.wq), _ptr(self.scales), _ptr(self.biases),
                   self.N, self.K, self.bits, self.group)

    @property
    def nbytes(self) -> int:
        return (self.wq.numel() * 4 + self.scales.numel() * 2
                + self.biases.numel() * 2)


def qweight(wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
            bits: int = 4, group: int = 64) -> QWeight:
    N = wq.shape[0]
    K = wq.shape[-1] * 32 // code_bits(bits)
    return QWeight(wq, scales, biases, N, K, bits, group)


def fuse_rows(parts: Sequence[QWeight]) -> QWeight:
    """Concatenate weights along the output axis, once, on the device (the
    fused QKV / gate+up weight).  The caller may drop the parts afterwards."""
    K, bits, group = parts[0].K, parts[0].bits, parts[0].group
    if any(p.K != K or p.bits != bits or p.group != group for p in parts):
        raise ValueError("parts must share K, bits and group")
    return QWeight(torch.cat([p.wq for p in parts]).contiguous(),
                   torch.cat([p.scales for p in parts]).contiguous(),
                   torch.cat([p.biases for p in parts]).contiguous(),
                   sum(p.N for p in parts), K, bits, group)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ws(workspace: Optional[torch.Tensor]):
    if workspace is None:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def _bf16(x: torch.Tensor, name: str) -> torch.Tensor:
    if x.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {x.dtype}")
    return x


def _check_weight(w: QWeight, copies: int = 1) -> None:
    """The library cannot see buffer sizes: refuse tensors whose sizes do not
    match (N, K, bits, group), so a wrong shape raises instead of reading
    past the end of a buffer.  `copies` = number of stacked experts."""
    if (w.bits not in (2, 3, 4, 6, 8, GWA_FP8_E4M3) or w.group <= 0
            or w.K % w.group):
        return                                   # the C ABI reports these
    words = copies * w.N * w.K * code_bits(w.bits) // 32
    groups = copies * w.N * (w.K // w.group)
    if w.wq.dtype != torch.int32 or w.wq.numel() != words:
        raise ValueError(f"wq must be int32 with {words} elements "
                         f"(got {w.wq.dtype}, {w.wq.numel()})")
    for name, t in (("scales", w.scales), ("biases", w.biases)):
        if t.dtype != torch.bfloat16 or t.numel() != groups:
            raise ValueError(f"{name} must be bfloat16 with {groups} elements "
                             f"(got {t.dtype}, {t.numel()})")


def _check_out(t: torch.Tensor, numel: int, name: str) -> None:
    if t.dtype != torch.bfloat16 or t.numel() != numel:
        raise ValueError(f"{name} must be bfloat16 with {numel} elements")


def expert_view(stacked: QWeight, num_experts: int) -> QWeight:
    """The same stacked tensors, described per expert (N = rows per expert)."""
    if stacked.N % num_experts:
        raise ValueError("rows do not divide evenly into experts")
    return QWeight(stacked.wq, stacked.scales, stacked.biases,
                   stacked.N // num_experts, stacked.K, stacked.bits,
                   stacked.group)


def workspace_bytes(M: int, K: int) -> int:
    return int(load().gwa_workspace_bytes(M, K))


def make_workspace(M: int, K: int, device=None) -> Optional[torch.Tensor]:
    n = workspace_bytes(M, K)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def qmv_affine(x: torch.Tensor, w: QWeight, y: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] . dequant(w)^T (bf16 out, fp32 accumulation)."""
    x = _bf16(x, "x")
    _check_weight(w)
    M = x.numel() // w.K
    if y is None:
        y = torch.empty((M, w.N), dtype=torch.bfloat16, device=x.device)
    _check_out(y, M * w.N, "y")
    if workspace is None and M > 8:
        workspace = make_workspace(M, w.K, x.device)
    wp, wn = _ws(workspace)
    _check(load().gwa_qmv_affine(_ptr(x), M, w.c(), _ptr(y), wp, wn,
                                 _stream(stream)))
    return y


def qmv_affine_noalloc(x: torch.Tensor, w: QWeight, y: torch.Tensor,
                       stream=None) -> torch.Tensor:
    """gwa_qmv_affine_noalloc: the same projection without a workspace, for
    callers that cannot allocate device memory on this path (the library's
    built-in scratch is used instead; see include/gwa.h).  `y` is required,
    since creating it here would allocate."""
    x = _bf16(x, "x")
    _check_weight(w)
    M = x.numel() // w.K
    _check_out(y, M * w.N, "y")
    _check(load().gwa_qmv_affine_noalloc(_ptr(x), M, w.c(), _ptr(y),
                                         _stream(stream)))
    return y


def qmv_fused_sections(x: torch.Tensor, w: QWeight, sections: Sequence[int],
                       outs: Optional[List[torch.Tensor]] = None,
                       out_bias: Optional[Sequence[Optional[torch.Tensor]]] = None,
                       workspace: Optional[torch.Tensor] = None,
                       stream=None) -> List[torch.Tensor]:
    """One pass over the row-concatenated weight, each section written to its
    own contiguous [M, size] buffer (e.g. Q, K, V)."""
    x = _bf16(x, "x")
    _check_weight(w)
    M = x.numel() // w.K
    n = len(sections)
    if outs is None:
        outs = [torch.empty((M, s), dtype=torch.bfloat16, device=x.device)
                for s in sections]
    if len(outs) != n:
        raise ValueError("one output per section")
    for i, (o, size) in enumerate(zip(outs, sections)):
        _check_out(o, M * size, f"outs[{i}]")
    if out_bias is not None:
        for i, (b, size) in enumerate(zip(out_bias, sections)):
            if b is not None:
                _check_out(b, size, f"out_bias[{i}]")
    sizes = (ctypes.c_int64 * n)(*sections)
    optrs = (ctypes.c_void_p * n)(*[_ptr(o) for o in outs])
    bptrs = None
    if out_bias is not None:
        bptrs = (ctypes.c_void_p * n)(*[_ptr(b) for b in out_bias])
    if workspace is None and M > 8:
        workspace = make_workspace(M, w.K, x.device)
    wp, wn = _ws(workspace)
    _check(load().gwa_qmv_fused_sections(
        _ptr(x), M, w.c(), n, ctypes.cast(sizes, ctypes.c_void_p),
        ctypes.cast(optrs, ctypes.c_void_p),
        ctypes.cast(bptrs, ctypes.c_void_p) if bptrs is not None else None,
        wp, wn, _stream(stream)))
    return list(outs)


def qmv_qkv_rope(x: torch.Tensor, w: QWeight, q_size: int, kv_size: int,
                 head_dim: int, rope_base: float, positions: torch.Tensor,
                 outs: Optional[List[torch.Tensor]] = None,
                 out_bias: Optional[Sequence[Optional[torch.Tensor]]] = None,
                 workspace: Optional[torch.Tensor] = None,
                 stream=None) -> List[torch.Tensor]:
    """gwa_qmv_qkv_rope: the fused QKV projection into contiguous Q, K, V,
    with the rotary embedding of Q and K at ``positions`` (int32 [M] on the
    device)."""
    x = _bf16(x, "x")
    _check_weight(w)
    M = x.numel() // w.K
    sections = (q_size, kv_size, kv_size)
    if positions.dtype != torch.int32 or positions.numel() < M:
        raise ValueError("positions must be int32 with one entry per token")
    if outs is None:
        outs = [torch.empty((M, s), dtype=torch.bfloat16, device=x.device)
                for s in sections]
    if len(outs) != 3:
        raise ValueError("three outputs: Q, K, V")
    for i, (o, size) in enumerate(zip(outs, sections)):
        _check_out(o, M * size, f"outs[{i}]")
    bptrs = None
    if out_bias is not None:
        for i, (b, size) in enumerate(zip(out_bias, sections)):
            if b is not None:
                _check_out(b, size, f"out_bias[{i}]")
        bptrs = (ctypes.c_void_p * 3)(*[_ptr(b) for b in out_bias])
    # one token of a u4/u8 group-64 weight needs none (its kernel forms its
    # own (cos, sin)); every other case takes a table in the workspace
    tuned = w.bits in (4, 8) and w.group == 64
    if workspace is None and (M > 1 or not tuned):
        n = int(load().gwa_qkv_rope_workspace_bytes(M, w.K, head_dim))
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    wp, wn = _ws(workspace)
    _check(load().gwa_qmv_qkv_rope(
        _ptr(x), M, w.c(), q_size, kv_size, head_dim, float(rope_base),
        _ptr(positions), _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]),
        ctypes.cast(bptrs, ctypes.c_void_p) if bptrs is not None else None,
        wp, wn, _stream(stream)))
    return list(outs)


def qmv_gate_up_silu(x: torch.Tensor, w: QWeight,
                     h: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """h[M, I] = SiLU(x Wg^T) * (x Wu^T) over a fused [gate; up] weight."""
    x = _bf16(x, "x")
    _check_weight(w)
    M = x.numel() // w.K
    if h is None:
        h = torch.empty((M, w.N // 2), dtype=torch.bfloat16, device=x.device)
    _check_out(h, M * (w.N // 2), "h")
    if workspace is None and M > 8:
        workspace = make_workspace(M, w.K, x.device)
    wp, wn = _ws(workspace)
    _check(load().gwa_qmv_gate_up_silu(_ptr(x), M, w.c(), _ptr(h), wp, wn,
                                       _stream(stream)))
    return h


def moe_qmv_gather(x: torch.Tensor, expert_ids: torch.Tensor, w: QWeight,
                   num_experts: int, mode: int,
                   route_w: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
    """Top-k expert projection over stacked experts (w.N rows per expert).

    mode 0 (gate+up SiLU): x [M, K] -> out [M, topk, w.N/2].
    mode 1 (down + combine): x [M, topk, K], route_w fp32 [M, topk]
    -> out [M, w.N].  w.N is the row count of ONE expert (see
    ``expert_view``); wq holds num_experts * w.N rows."""
    x = _bf16(x, "x")
    _check_weight(w, copies=num_experts)
    if expert_ids.dtype != torch.int32 or expert_ids.dim() != 2:
        raise TypeError("expert_ids must be int32 [M, topk]")
    M, topk = expert_ids.shape
    if x.numel() != (M if mode == GWA_MOE_GATE_UP_SILU else M * topk) * w.K:
        raise ValueError("x has the wrong number of elements for this mode")
    if route_w is not None and (route_w.dtype != torch.float32
                                or route_w.numel() != M * topk):
        raise TypeError("route_w must be float32 [M, topk]")
    if status is not None and (status.dtype != torch.int32
                               or status.numel() < 1):
        raise TypeError("status must be an int32 tensor")
    if out is None:
        shape = (M, topk, w.N // 2) if mode == GWA_MOE_GATE_UP_SILU else \
            (M, w.N)
        out = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
    _check_out(out, M * topk * (w.N // 2) if mode == GWA_MOE_GATE_UP_SILU
               else M * w.N, "out")
    _check(load().gwa_moe_qmv_gather(_ptr(x), M, topk, _ptr(expert_ids),
                                     _ptr(route_w), w.c(), num_experts, mode,
                                     _ptr(out), _ptr(status),
                                     _stream(stream)))
    return out


def quantize_affine(w: torch.Tensor, bits: int = 4, group: int = 64,
                    out: Optional[QWeight] = None, stream=None) -> QWeight:
    """gwa_quantize_affine: bf16 weights w [N, K] -> packed QWeight (codes,
    bf16 scales and biases per 64 inputs).  Allocates the outputs unless
    ``out`` (N, K, bits and group matching) is given."""
    w = _bf16(w, "w")
    if w.dim() != 2:
        raise ValueError("w must be [N, K]")
    N, K = w.shape
    if out is None:
        dev = w.device
        out = QWeight(
            torch.empty((N, max(K * bits // 32, 0)), dtype=torch.int32,
                        device=dev),
            torch.empty((N, max(K // group, 0)), dtype=torch.bfloat16,
                        device=dev),
            torch.empty((N, max(K // group, 0)), dtype=torch.bfloat16,
                        device=dev),
            N, K, bits, group)
    elif (out.N, out.K, out.bits, out.group) != (N, K, bits, group):
        raise ValueError("out does not match w's shape, bits and group")
    _check(load().gwa_quantize_affine(_ptr(w), N, K, bits, group,
                                      _ptr(out.wq), _ptr(out.scales),
                                      _ptr(out.biases), _stream(stream)))
    return out


def sdpa_dequant_v(q: torch.Tensor, k: torch.Tensor, vq: torch.Tensor,
                   vs: torch.Tensor, vb: torch.Tensor, bits: int = 4,
                   group: int = 64, scale: Optional[float] = None,
                   causal: bool = True, out: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
    """gwa_sdpa_dequant_v: softmax attention of q [B, Hq, Lq, D] over bf16
    keys k [B, Hkv, T, D] and quantized values (vq int32 [B, Hkv, T,
    D*bits/32], vs / vb bfloat16 [B, Hkv, T, D/64]); returns bf16
    [B, Hq, Lq, D]."""
    q, k = _bf16(q, "q"), _bf16(k, "k")
    _bf16(vs, "vs")
    _bf16(vb, "vb")
    B, Hq, Lq, D = q.shape
    Bk, Hkv, T, Dk = k.shape
    if Bk != B or Dk != D:
        raise ValueError("k must be [B, Hkv, T, D] with q's B and D")
    if vq.dtype != torch.int32 or tuple(vq.shape) != (B, Hkv, T, D * bits // 32):
        raise ValueError("vq must be int32 [B, Hkv, T, D*bits/32]")
    for name, t in (("vs", vs), ("vb", vb)):
        if tuple(t.shape) != (B, Hkv, T, D // group):
            raise ValueError(f"{name} must be [B, Hkv, T, D/group]")
    for name, t in (("q", q), ("k", k), ("vq", vq), ("vs", vs), ("vb", vb)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out is None:
        out = torch.empty((B, Hq, Lq, D), dtype=torch.bfloat16, device=q.device)
    _check_out(out, B * Hq * Lq * D, "out")
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    if workspace is None:
        n = int(load().gwa_sdpa_workspace_bytes(B, Hq, Hkv, Lq, T, D))
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    wp, wn = _ws(workspace)
    _check(load().gwa_sdpa_dequant_v(
        _ptr(q), B, Hq, Lq, D, _ptr(k), Hkv, T, _ptr(vq), _ptr(vs), _ptr(vb),
        bits, group, float(scale), int(bool(causal)), _ptr(out), wp, wn,
        _stream(stream)))
    return out


def debug_unpack(w: QWeight, stream=None) -> torch.Tensor:
    codes = torch.empty((w.N, w.K), dtype=torch.uint8, device=w.wq.device)
    _check(load().gwa_debug_unpack(w.c(), _ptr(codes), _stream(stream)))
    return codes


def debug_bounded_wait(limit_us: int, device=None, stream=None) -> torch.Tensor:
    """gwa_debug_bounded_wait: int32[4] (gave up, waited us) for the plain
    and the sleeping bounded wait, each made to run out after limit_us."""
    out = torch.full((4,), -1, dtype=torch.int32,
                     device=device if device is not None else "cuda")
    _check(load().gwa_debug_bounded_wait(int(limit_us), _ptr(out),
                                         _stream(stream)))
    return out


def debug_dequant(w: QWeight, stream=None) -> torch.Tensor:
    wf = torch.empty((w.N, w.K), dtype=torch.float32, device=w.wq.device)
    _check(load().gwa_debug_dequant(w.c(), _ptr(wf), _stream(stream)))
    return wf
