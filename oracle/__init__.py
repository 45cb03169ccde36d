"""Plain fp64 CPU oracle for affine group-quantized projections.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library (``group_wise_affine_gb300``) never imports it, and it imports nothing
from the product library: the two meet only through the seeded inputs.

The arithmetic lives in ``oracle.c`` (plain C, fp64, summed in input order);
this module compiles it with gcc on first use and wraps each routine with
numpy marshalling.  The few steps written here in Python are plain array
operations: splitting the fused output at the section boundaries ("The
Cathedral Doubled Itself", "The two fusions": one matmul over the
output-axis concatenation, split back into Q, K, V on the last axis) and the
optional per-output additive bias.

Every bf16 quantity is carried as its uint16 bit pattern.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile oracle.c into ``_build/liboracle.so`` (OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = ctypes.c_double
        lib.orc_e4m3_value.argtypes = [ctypes.c_uint32]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_silu.argtypes = [ctypes.c_double]
        lib.orc_silu.restype = ctypes.c_double
        lib.orc_max_threads.argtypes = []
        lib.orc_max_threads.restype = _int
        lib.orc_unpack.argtypes = [_u32p, _i64, _i64, _int, _u8p]
        lib.orc_dequant.argtypes = [_u32p, _u16p, _u16p, _i64, _i64, _int,
                                    _int, _f64p]
        lib.orc_qmv.argtypes = [_u16p, _i64, _u32p, _u16p, _u16p, _i64, _i64,
                                _int, _int, ctypes.c_void_p, _i64, _f64p, _int]
        lib.orc_gate_up_silu.argtypes = [_u16p, _i64, _u32p, _u16p, _u16p,
                                         _i64, _i64, _int, _int,
                                         ctypes.c_void_p, _i64, _f64p, _int]
        lib.orc_moe_gate_up_silu.argtypes = [_u16p, _i64, _i64, _i32p, _u32p,
                                             _u16p, _u16p, _i64, _i64, _i64,
                                             _int, _int, _f64p, _int]
        lib.orc_moe_down_combine.argtypes = [_u16p, _i64, _i64, _i32p, _f32p,
                                             _u32p, _u16p, _u16p, _i64, _i64,
                                             _i64, _int, _int, _f64p, _int]
        lib.orc_quantize_affine.argtypes = [_u16p, _i64, _i64, _int, _int,
                                            _u32p, _u16p, _u16p]
        lib.orc_rope.argtypes = [_f64p, _i64, _i64, _i64, ctypes.c_double,
                                 _i32p]
        lib.orc_sdpa_dequant_v.argtypes = [_u16p, _i64, _i64, _i64, _i64, _u16p,
                                           _i64, _i64, _u32p, _u16p, _u16p,
                                           _int, _int, ctypes.c_double, _int,
                                           _f64p]
        for name in ("orc_unpack", "orc_dequant", "orc_qmv",
                     "orc_gate_up_silu", "orc_moe_gate_up_silu",
                     "orc_moe_down_combine", "orc_quantize_affine",
                     "orc_rope", "orc_sdpa_dequant_v"):
            getattr(lib, name).restype = _int
        _lib = lib
        return lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    """OpenMP threads the oracle uses when ``nthreads`` is 0."""
    return int(_load().orc_max_threads())


def bf16_to_f64(h) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    h = _c(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def silu(g: float) -> float:
    return float(_load().orc_silu(float(g)))


# bits value selecting 8-bit OCP FP8 E4M3 codes (see oracle.c)
FP8_E4M3 = 0x108


def code_width(bits: int) -> int:
    """Bits a code takes in the packed stream."""
    return 8 if bits == FP8_E4M3 else bits


def e4m3_value(byte: int) -> float:
    """The OCP FP8 E4M3 number a byte stands for (NaN for S.1111.111)."""
    return float(_load().orc_e4m3_value(int(byte) & 0xff))


def unpack(wq, N: int, K: int, bits: int) -> np.ndarray:
    """Integer codes [N, K] (uint8) of a packed weight [N, K*bits/32]."""
    wq = _c(wq, np.uint32)
    out = np.empty((N, K), dtype=np.uint8)
    _check(_load().orc_unpack(wq, N, K, bits, out), "unpack")
    return out


def dequant(wq, scales, biases, N: int, K: int, bits: int,
            group: int = 64) -> np.ndarray:
    """Dequantized weights w = scale*q + bias, float64 [N, K]."""
    out = np.empty((N, K), dtype=np.float64)
    _check(_load().orc_dequant(_c(wq, np.uint32), _c(scales, np.uint16),
                               _c(biases, np.uint16), N, K, bits, group, out),
           "dequant")
    return out


def _rows_arg(rows):
    if rows is None:
        return None, None
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, r.ctypes.data_as(ctypes.c_void_p)


def qmv(x, wq, scales, biases, N: int, K: int, bits: int, group: int = 64,
        rows=None, nthreads: int = 0) -> np.ndarray:
    """y[m, i] = sum_k x[m,k] * w[rows[i], k] in fp64; x is bf16 [M, K].

    ``rows=None`` computes every output row.  Returns float64 [M, n_rows]."""
    x = _c(x, np.uint16).reshape(-1, K)
    M = x.shape[0]
    r, rp = _rows_arg(rows)
    n_rows = N if r is None else r.shape[0]
    y = np.empty((M, n_rows), dtype=np.float64)
    _check(_load().orc_qmv(x, M, _c(wq, np.uint32), _c(scales, np.uint16),
                           _c(biases, np.uint16), N, K, bits, group, rp,
                           n_rows, y, nthreads), "qmv")
    return y


def fused_sections(x, wq, scales, biases, section_sizes, K: int, bits: int,
                   group: int = 64, out_bias=None, nthreads: int = 0):
    """One projection over the output-axis concatenation, split back into one
    contiguous array per section; ``out_bias`` (optional, one bf16 vector per
    section) is added after the split."""
    N = int(sum(section_sizes))
    y = qmv(x, wq, scales, biases, N, K, bits, group, nthreads=nthreads)
    outs, start = [], 0
    for i, size in enumerate(section_sizes):
        part = np.array(y[:, start:start + size], dtype=np.float64, order="C")
        if out_bias is not None and out_bias[i] is not None:
            part = part + bf16_to_f64(out_bias[i])[None, :]
        outs.append(part)
        start += size
    return outs


def gate_up_silu(x, wq, scales, biases, N2: int, K: int, bits: int,
                 group: int = 64, cols=None, nthreads: int = 0) -> np.ndarray:
    """h[m, i] = SiLU(gate) * up over a fused [gate; up] weight of 2*I rows."""
    x = _c(x, np.uint16).reshape(-1, K)
    M = x.shape[0]
    r, rp = _rows_arg(cols)
    n_cols = N2 // 2 if r is None else r.shape[0]
    h = np.empty((M, n_cols), dtype=np.float64)
    _check(_load().orc_gate_up_silu(x, M, _c(wq, np.uint32),
                                    _c(scales, np.uint16),
                                    _c(biases, np.uint16), N2, K, bits, group,
                                    rp, n_cols, h, nthreads), "gate_up_silu")
    return h


def moe_gate_up_silu(x, ids, wq, scales, biases, E: int, N2: int, K: int,
                     bits: int, group: int = 64,
                     nthreads: int = 0) -> np.ndarray:
    """h[t, j, :] = SiLU(Wg[e] x_t) * (Wu[e] x_t), e = ids[t, j]; fp64."""
    x = _c(x, np.uint16).reshape(-1, K)
    ids = _c(ids, np.int32)
    M, topk = ids.shape
    h = np.empty((M, topk, N2 // 2), dtype=np.float64)
    _check(_load().orc_moe_gate_up_silu(x, M, topk, ids, _c(wq, np.uint32),
                                        _c(scales, np.uint16),
                                        _c(biases, np.uint16), E, N2, K, bits,
                                        group, h, nthreads),
           "moe_gate_up_silu")
    return h


def moe_down_combine(hin, ids, route_w, wq, scales, biases, E: int, N: int,
                     K: int, bits: int, group: int = 64,
                     nthreads: int = 0) -> np.ndarray:
    """y[t, :] = sum_j r[t,j] * (Wd[e] hin[t,j,:]), e = ids[t,j]; fp64."""
    ids = _c(ids, np.int32)
    M, topk = ids.shape
    hin = _c(hin, np.uint16).reshape(M, topk, K)
    y = np.empty((M, N), dtype=np.float64)
    _check(_load().orc_moe_down_combine(hin, M, topk, ids,
                                        _c(route_w, np.float32),
                                        _c(wq, np.uint32),
                                        _c(scales, np.uint16),
                                        _c(biases, np.uint16), E, N, K, bits,
                                        group, y, nthreads),
           "moe_down_combine")
    return y


def quantize_affine(w, N: int, K: int, bits: int, group: int = 64):
    """Affine group quantization of bf16 weights w [N, K] (uint16 bit
    patterns): returns (wq uint32 [N, K*bits/32], scales, biases uint16
    [N, K/group]).  Per group: scale = bf16_rn((max - min) / (2^bits - 1)),
    bias = min, code = clamp(rint((w - bias) / scale)) in fp32 (see
    oracle.c for the reading and its source)."""
    w = _c(w, np.uint16)
    wq = np.empty((N, K * bits // 32), dtype=np.uint32)
    sc = np.empty((N, K // group), dtype=np.uint16)
    bi = np.empty((N, K // group), dtype=np.uint16)
    _check(_load().orc_quantize_affine(w, N, K, bits, group, wq, sc, bi),
           "quantize_affine")
    return wq, sc, bi


def rope(y, head_dim: int, base: float, positions) -> np.ndarray:
    """Rotary embedding (rotate-half pairing) of y [M, width] (fp64, width a
    multiple of head_dim) at positions[m]; returns a new array."""
    out = np.array(y, dtype=np.float64, order="C", copy=True)
    M, width = out.shape
    pos = _c(positions, np.int32)
    _check(_load().orc_rope(out, M, width, head_dim, float(base), pos), "rope")
    return out


def qkv_rope(x, wq, scales, biases, q_size: int, kv_size: int, K: int,
             bits: int, head_dim: int, base: float, positions, out_bias=None,
             group: int = 64):
    """The fused QKV projection split into Q, K, V (optional additive bias
    per output), then RoPE on Q and K.  Returns [Q, K, V] (fp64)."""
    q, k, v = fused_sections(x, wq, scales, biases, [q_size, kv_size, kv_size],
                             K, bits, group=group, out_bias=out_bias)
    return [rope(q, head_dim, base, positions), rope(k, head_dim, base, positions),
            v]


def sdpa_dequant_v(q, k, vq, vs, vb, B: int, Hq: int, Lq: int, D: int,
                   Hkv: int, T: int, bits: int = 4, group: int = 64,
                   scale: float = None, causal: bool = True) -> np.ndarray:
    """Softmax attention of q [B, Hq, Lq, D] over bf16 keys k [B, Hkv, T, D]
    and affine-quantized values (codes vq [B, Hkv, T, D*bits/32], bf16 scales
    and biases vs, vb [B, Hkv, T, D/group]); fp64 out [B, Hq, Lq, D]."""
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((B, Hq, Lq, D), dtype=np.float64)
    _check(_load().orc_sdpa_dequant_v(
        _c(q, np.uint16), B, Hq, Lq, D, _c(k, np.uint16), Hkv, T,
        _c(vq, np.uint32), _c(vs, np.uint16), _c(vb, np.uint16), bits, group,
        float(scale), int(bool(causal)), out), "sdpa_dequant_v")
    return out


def within_tolerance(got, ref, rel: float = 1e-2):
    """The output bar: |got - ref| <= rel * max(1, |ref|), elementwise.

    Returns (ok, max_abs_err, worst_ratio) where worst_ratio is the largest
    |err| / (rel * max(1, |ref|))."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bound = rel * np.maximum(1.0, np.abs(ref))
    ratio = err / bound
    if err.size == 0:
        return True, 0.0, 0.0
    return bool(np.all(ratio <= 1.0)), float(err.max()), float(ratio.max())
