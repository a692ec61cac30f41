"""Log-sum-exp output on the GPU (fa_prefill_fwd_lse / fa_decode_fwd_lse)
against the fp64 oracle's lse on the same seeded inputs.

lse = log sum_j exp(scale * <q, k_j>) over a row's visible keys; -inf for a
row that sees none (the per-row statistic of the flash-attention backward's
"_pre" pass in tessera #90; rocm-libraries #13108 leaves it out of its first
decode milestone).

Bar: |lse - lse_ref| <= 1e-3 where finite, and -inf exactly where the oracle
has -inf.  The kernel's error comes from fp32 score accumulation in the tensor
cores (about 2^-23 |s| per term, |s| of a few units here), the approximate
exp2 of P (relative 2^-22) summed in fp32, and one approximate log2: about
1e-5 in total, so 1e-3 leaves margin while still catching a wrong base,
scale or missing term (each of those moves lse by O(1)).
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle

pytestmark = pytest.mark.gpu
LSE_ATOL = 1e-3


def lse_compare(got, ref):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "-inf pattern differs"
    assert not np.isnan(got).any()
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin]).max() if fin.any() else 0.0
    assert err <= LSE_ATOL, f"max |lse - ref| = {err}"
    return err


def run_prefill_lse(fa, q, k, v, scale, causal):
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out, lse = fa.prefill(qd, kd, vd, scale, causal, lse=True)
    plain = fa.prefill(qd, kd, vd, scale, causal)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, f"device error word {detail:#x}"
    # the lse variant runs the same kernel: O is bit-identical
    assert torch.equal(out, plain)
    return out, lse.cpu().numpy()


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt,scale", [
    (1, 2, 1, 128, 128, 64, True, torch.bfloat16, 1 / 8),        # tiny causal GQA
    (2, 8, 8, 1000, 1536, 64, False, torch.float16, 1 / 8),      # ragged non-causal fp16
    (2, 4, 2, 300, 200, 128, True, torch.bfloat16, 0.088),       # Sq > Sk: rows with no key
    (1, 4, 1, 77, 333, 128, True, torch.bfloat16, 0.088),        # Sq < Sk causal
    (1, 2, 1, 129, 257, 64, False, torch.bfloat16, 0.0),         # scale 0: lse = log(Sk)
    (1, 2, 2, 200, 300, 64, True, torch.bfloat16, -0.125),       # negative scale
])
def test_prefill_lse_full(fa, B, Hq, Hkv, Sq, Sk, D, causal, dt, scale):
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed=Sq + Sk)
    _, lse = run_prefill_lse(fa, q, k, v, scale, causal)
    _, ref = oracle.attention(q, k, v, scale, causal, return_lse=True)
    lse_compare(lse, ref)
    if scale == 0.0:
        assert np.allclose(lse, math.log(Sk), atol=1e-4)


def test_prefill_lse_gqa_causal_8k_sampled(fa):
    s = fa_inputs.GQA_CAUSAL_8K
    q, k, v = fa_inputs.prefill_inputs_for(s, seed=0)
    _, lse = run_prefill_lse(fa, q, k, v, s.scale, s.causal)
    rows = fa_inputs.sample_rows(s.B, s.Hq, s.Hkv, s.Sq, n=1024, seed=0)
    _, ref = oracle.attention(q, k, v, s.scale, s.causal, rows=rows, return_lse=True)
    r = rows.numpy()
    lse_compare(lse[r[:, 0], r[:, 1], r[:, 2]], ref)


def test_prefill_lse_no_keys(fa):
    dev = torch.device("cuda", 0)
    q = torch.randn(2, 10, 4, 64, device=dev).to(torch.bfloat16)
    k = torch.empty(2, 0, 2, 64, device=dev, dtype=torch.bfloat16)
    lse = torch.zeros(2, 4, 10, device=dev)
    out, lse = fa.prefill(q, k, k, 0.1, False, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.zeros_like(out))
    assert torch.isneginf(lse).all()


def run_decode_lse(fa, q, kc, vc, L, scale):
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), kc.to(dev), vc.to(dev)
    vl = torch.tensor([L], dtype=torch.int32, device=dev)
    out, lse = fa.decode(qd, kd, vd, vl, scale, lse=True)
    plain = fa.decode(qd, kd, vd, vl, scale)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, f"device error word {detail:#x}"
    assert torch.equal(out, plain)
    return lse.cpu().numpy()


@pytest.mark.parametrize("L", [0, 1, 31, 2733, 65536])
def test_decode_lse(fa, L):
    s = fa_inputs.DECODE_1TOK
    q, kc, vc, L = fa_inputs.decode_inputs_for(s, seed=3, L=L)
    lse = run_decode_lse(fa, q, kc, vc, L, s.scale)
    _, ref = oracle.decode(q, kc, vc, L, s.scale, return_lse=True)
    lse_compare(lse, ref)


def test_decode_lse_zero_capacity(fa):
    dev = torch.device("cuda", 0)
    q = torch.randn(2, 1, 8, 128, device=dev).to(torch.bfloat16)
    kc = torch.empty(2, 0, 2, 128, device=dev, dtype=torch.bfloat16)
    vl = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = fa.decode(q, kc, kc, vl, 0.1, lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.zeros_like(out)) and torch.isneginf(lse).all()
