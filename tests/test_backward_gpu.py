"""Backward pass on the GPU (fa_backward) against the fp64 oracle's gradients
of sum(O * dO) (tessera #90, flash-attention backward commit note).

The forward output and log-sum-exp come from fa_prefill_fwd_lse on the same
inputs, as a training step would use them.  Bar, per gradient tensor:
relative L2 error <= 1e-2 and max |error| <= 1.5e-2 * max |reference|, no
NaN/Inf.  The kernel rounds P and dS to the input type as MMA operands
(relative 2^-9 for bf16 per term), forms Delta from the rounded O, and rounds
each gradient once; the oracle is exact in fp64.  Measured on GB300: relative
L2 about 2.4e-3 (bf16) and 3e-4 (fp16), max error at most 5.4e-3 of max |ref|."""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle

pytestmark = pytest.mark.gpu
REL_L2 = 1e-2
MAX_REL = 1.5e-2


def grad_compare(got, ref, name):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, name
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    scale = np.abs(ref).max()
    if scale == 0:
        assert np.abs(got).max() == 0, name
        return 0.0
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max() / scale
    assert rel <= REL_L2, f"{name}: relative L2 {rel:.3e}"
    assert mx <= MAX_REL, f"{name}: max error {mx:.3e} of max |ref|"
    return rel


def run_backward(fa, q, k, v, dout, scale, causal):
    dev = torch.device("cuda", 0)
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    o, lse = fa.prefill(qd, kd, vd, scale, causal, lse=True)
    dq, dk, dv = fa.backward(qd, kd, vd, o, dd, lse, scale, causal)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, f"device error word {detail:#x}"
    return [t.float().cpu().numpy() for t in (dq, dk, dv)]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt", [
    (1, 2, 1, 128, 128, 64, True, torch.bfloat16),
    (2, 4, 2, 300, 500, 128, True, torch.bfloat16),     # Sq != Sk, ragged tails
    (1, 4, 4, 257, 257, 64, False, torch.float16),
    (1, 8, 2, 1024, 1024, 128, True, torch.bfloat16),   # GQA: dk/dv sum 4 heads
    (1, 4, 1, 500, 200, 128, True, torch.bfloat16),     # Sq > Sk: rows with no key
    (2, 2, 1, 77, 900, 64, False, torch.bfloat16),
    (1, 4, 2, 700, 300, 128, False, torch.float16),    # D = 128 fp16, no mask
    (1, 6, 2, 384, 384, 128, True, torch.bfloat16),     # G = 3 query heads per kv head
])
def test_backward_against_oracle(fa, B, Hq, Hkv, Sq, Sk, D, causal, dt):
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed=Sq + Sk + D)
    dout = torch.randn(B, Sq, Hq, D, generator=torch.Generator().manual_seed(Sq)).to(dt)
    scale = 1 / math.sqrt(D)
    dq, dk, dv = run_backward(fa, q, k, v, dout, scale, causal)
    rq, rk, rv = oracle.attention_bwd(q, k, v, dout, scale, causal)
    grad_compare(dq, rq, "dq")
    grad_compare(dk, rk, "dk")
    grad_compare(dv, rv, "dv")


def test_backward_gqa_causal_2k(fa):
    B, Hq, Hkv, S, D = 1, 16, 2, 2048, 128
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, S, S, D, torch.bfloat16, seed=7)
    dout = torch.randn(B, S, Hq, D, generator=torch.Generator().manual_seed(8)).to(torch.bfloat16)
    dq, dk, dv = run_backward(fa, q, k, v, dout, 1 / math.sqrt(D), True)
    rq, rk, rv = oracle.attention_bwd(q, k, v, dout, 1 / math.sqrt(D), True)
    grad_compare(dq, rq, "dq")
    grad_compare(dk, rk, "dk")
    grad_compare(dv, rv, "dv")


@pytest.mark.parametrize("D", [64, 128])
def test_backward_empty_sides(fa, D):
    """No keys: dQ is zero.  No query rows: the dK/dV kernel runs items with
    no query steps (at D = 128 the 128-row sub-tile kernel), whose epilogue
    writes zero gradients."""
    dev = torch.device("cuda", 0)
    q = torch.randn(1, 10, 4, D, device=dev).to(torch.bfloat16)
    kz = torch.empty(1, 0, 2, D, device=dev, dtype=torch.bfloat16)
    lse = torch.full((1, 4, 10), -math.inf, device=dev)
    dq, dk, dv = fa.backward(q, kz, kz, torch.zeros_like(q), q, lse, 0.1, True)
    torch.cuda.synchronize()
    assert torch.equal(dq, torch.zeros_like(dq)) and dk.numel() == 0
    qz = torch.empty(1, 0, 4, D, device=dev, dtype=torch.bfloat16)
    k = torch.randn(1, 7, 2, D, device=dev).to(torch.bfloat16)
    lz = torch.empty(1, 4, 0, device=dev)
    dq, dk, dv = fa.backward(qz, k, k, qz, qz, lz, 0.1, False)
    torch.cuda.synchronize()
    assert torch.equal(dk, torch.zeros_like(dk)) and torch.equal(dv, torch.zeros_like(dv))
