"""Test bars shared by the GPU tests (the arithmetic of the tolerances, not
of the method)."""
import numpy as np

import gwa_synth as synth

TOL = 1e-2


def tc_accumulation_term(x, w, rows):
    """The fp32 accumulation's own rounding on the tensor-core kernel, per
    output [M, len(rows)].

    Operands reach the tensor cores exactly, but the products are summed in
    fp32: each of the MMA's K steps (kext/16, twice for u8's two code halves)
    rounds at most 2^-23 of the magnitude of what it adds up.  The terms
    summed are x * s(q - c) per input and b' X per group (b' = b + c s, c = 8
    or 136, X a group sum), all bounded by |x| (|b| + 2 c |s|) per input."""
    K = w.K
    G = K // 64
    c = 8.0 if w.bits == 4 else 136.0
    s = np.abs(synth.bf16_values(w.scales[rows]).astype(np.float64))
    b = np.abs(synth.bf16_values(w.biases[rows]).astype(np.float64))
    per_input = np.repeat(b + 2.0 * c * s, 64, axis=1)      # [rows, K]
    xa = np.abs(synth.bf16_values(x).astype(np.float64))
    mag = xa @ per_input.T
    kext = K + ((3 * G + 127) // 128) * 128
    steps = (kext // 16) * (2 if w.bits == 8 else 1)
    return steps * 2.0**-23 * mag


def tc_accumulation_bar(ref, x, w, rows):
    """1e-2 * max(1, |ref|) plus the fp32 accumulation's own rounding on the
    tensor-core kernel (tc_accumulation_term).  Where an output cancels to
    far below its terms (a large common weight offset, as with u8 biases of
    -8 s), that rounding is above 1e-2 |y|."""
    return TOL * np.maximum(1.0, np.abs(ref)) + tc_accumulation_term(x, w, rows)


def tc_swiglu_bar(x, w, I):
    """Reference h = SiLU(g) * u in fp64 for a gate+up weight of 2I rows on
    the tensor-core kernel, and its bar: 1e-2 * max(1, |h|) plus the fp32
    rounding of g and u (tc_accumulation_term) carried through the epilogue,
    |SiLU'(g) u| e_g + |SiLU(g)| e_u.  That term matters where one factor
    cancels to far below its terms while the other is large."""
    import oracle
    W = oracle.dequant(w.wq, w.scales, w.biases, w.N, w.K, w.bits)
    xv = synth.bf16_values(x).astype(np.float64)
    g = xv @ W[:I].T
    u = xv @ W[I:].T
    eg = tc_accumulation_term(x, w, np.arange(I))
    eu = tc_accumulation_term(x, w, np.arange(I, 2 * I))
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    dsilu = sig * (1.0 + g * (1.0 - sig))
    h = silu * u
    bar = TOL * np.maximum(1.0, np.abs(h)) + np.abs(dsilu * u) * eg + np.abs(silu) * eu
    return h, bar


def assert_within(got, ref, bar, what=""):
    err = np.abs(got - ref)
    worst = float((err / bar).max()) if err.size else 0.0
    assert worst <= 1.0, f"{what}: max |err| {err.max():.3g}, worst err/bar {worst:.3g}"
