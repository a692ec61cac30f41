"""Parity bar shared by the GPU tests: the CUDA output against the fp64 oracle.

Tolerance for bf16/fp16 outputs: max |o - ref| <= 1e-2 and
||o - ref||_2 / ||ref||_2 <= 5e-3 over the compared elements, and no NaN/Inf.
The bf16 half-ulp near |O| ~ 2-4 is 7.8e-3, so the absolute bar is the
one-rounding bound of the output plus the fp32/bf16-P accumulation error.
"""
import numpy as np

MAX_ABS = 1e-2
REL_L2 = 5e-3


def compare(out, ref, max_abs=MAX_ABS, rel_l2=REL_L2):
    """Return (max_abs_err, rel_l2_err); raise AssertionError past the bar."""
    o = np.asarray(out, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert o.shape == r.shape, (o.shape, r.shape)
    assert np.isfinite(o).all(), f"non-finite outputs: {np.count_nonzero(~np.isfinite(o))}"
    if o.size == 0:
        return 0.0, 0.0
    err = np.abs(o - r)
    mae = float(err.max())
    nr = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(o - r) / nr) if nr > 0 else float(np.linalg.norm(o - r))
    assert mae <= max_abs, f"max abs err {mae:.3e} > {max_abs:.1e}"
    assert rel <= rel_l2, f"rel L2 err {rel:.3e} > {rel_l2:.1e}"
    return mae, rel


def rounding_bound(ref, vmax, dtype_bits=8):
    """Arithmetic bar for softmax temperatures far from 1/sqrt(D), where one
    key can carry most of the weight: P is rounded to the input type before
    P@V (relative error <= 2^-dtype_bits per element, bf16: 8 mantissa bits
    incl. the implicit one -> 2^-8 for a worst-case sum of same-sign
    errors) and O is rounded once (half an ulp of max|O|).  Returns the
    max-abs bar; the relative-L2 bar stays REL_L2."""
    omax = float(np.max(np.abs(ref))) if np.size(ref) else 0.0
    half_ulp_o = 2.0 ** (np.floor(np.log2(max(omax, 1e-30))) - dtype_bits) if omax > 0 else 0.0
    return float(vmax) * 2.0 ** -dtype_bits + half_ulp_o + 1e-3
