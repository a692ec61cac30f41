"""Seeded random small shapes through every entry point, against the fp64
oracle.  The hand-picked parity cases cover the edges one at a time; these
draw the shape parameters together (batch, GQA ratio, ragged Sq / Sk, D,
causal, dtype, scale, valid lengths, page sizes), so a combination no one
thought of still gets compared element by element.  The draws are fixed by
their seeds, so a failure reproduces."""
import math
import random

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare
from tests.test_lse_gpu import lse_compare

pytestmark = pytest.mark.gpu
DTYPES = (torch.bfloat16, torch.float16)


def _prefill_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        hkv = rng.choice([1, 2, 4])
        g = rng.choice([1, 2, 3, 5, 8])
        out.append((rng.choice([1, 2]), hkv * g, hkv, rng.randint(1, 600), rng.randint(1, 700),
                    rng.choice([64, 128]), rng.random() < 0.6, rng.choice(DTYPES),
                    rng.random() < 0.25))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt,odd_scale", _prefill_cases(12, 101))
def test_random_prefill(fa, B, Hq, Hkv, Sq, Sk, D, causal, dt, odd_scale):
    scale = 0.07 if odd_scale else 1 / math.sqrt(D)
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed=Sq * 7 + Sk)
    dev = torch.device("cuda", 0)
    o, lse = fa.prefill(q.to(dev), k.to(dev), v.to(dev), scale, causal, lse=True)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, hex(detail)
    ref, ref_lse = oracle.attention(q, k, v, scale, causal, return_lse=True)
    compare(o.float().cpu().numpy(), ref)
    lse_compare(lse.cpu().numpy(), ref_lse)


def _varlen_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        nseq = rng.randint(1, 5)
        lq = [rng.choice([0, rng.randint(1, 400)]) for _ in range(nseq)]
        lk = [x if rng.random() < 0.6 else rng.randint(0, 450) for x in lq]
        hkv = rng.choice([1, 2])
        out.append((lq, lk, hkv * rng.choice([1, 2, 4]), hkv, rng.choice([64, 128]),
                    rng.random() < 0.6, rng.choice(DTYPES)))
    return out


@pytest.mark.parametrize("lq,lk,Hq,Hkv,D,causal,dt", _varlen_cases(5, 202))
def test_random_varlen(fa, lq, lk, Hq, Hkv, D, causal, dt):
    scale = 1 / math.sqrt(D)
    q, k, v, cq, ck = fa_inputs.varlen_inputs(lq, lk, Hq, Hkv, D, dt, seed=sum(lq) + 3)
    dev = torch.device("cuda", 0)
    o = fa.prefill_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev),
                          max(lq), scale, causal)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, hex(detail)
    if q.shape[0] == 0:  # no query row drawn: nothing to write, no error
        assert o.numel() == 0
        return
    compare(o.float().cpu().numpy(),
            oracle.attention_varlen(q, k, v, cq.tolist(), ck.tolist(), scale, causal))


def _decode_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        hkv = rng.choice([1, 2, 4])
        cap = rng.randint(1, 3000)
        out.append((rng.randint(1, 3), hkv * rng.randint(1, 20), hkv, cap,
                    rng.choice([64, 128]), rng.randint(1, cap)))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,cap,D,L", _decode_cases(6, 303))
def test_random_decode(fa, B, Hq, Hkv, cap, D, L):
    scale = 1 / math.sqrt(D)
    q, kc, vc, L = fa_inputs.decode_inputs(B, Hq, Hkv, cap, D, seed=cap + L, L=L)
    dev = torch.device("cuda", 0)
    vl = torch.tensor([L], dtype=torch.int32, device=dev)
    o = fa.decode(q.to(dev), kc.to(dev), vc.to(dev), vl, scale)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, hex(detail)
    got = o.float().cpu().numpy().reshape(B, Hq, D)
    compare(got, oracle.decode(q, kc, vc, L, scale))


def _paged_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        B = rng.randint(1, 6)
        page = rng.choice([32, 64, 128, 256])  # a positive multiple of 32 (fa.h)
        max_pages = rng.randint(1, 12)
        lens = [rng.randint(0, page * max_pages) for _ in range(B)]
        hkv = rng.choice([1, 2])
        out.append((B, hkv * rng.choice([1, 2, 4, 8]), hkv, rng.choice([64, 128]), page,
                    max_pages, lens))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,D,page_size,max_pages,lens", _paged_cases(4, 404))
def test_random_paged_decode(fa, B, Hq, Hkv, D, page_size, max_pages, lens):
    from tests.test_paged_decode_gpu import paged_inputs, run_paged
    q, kp, vp, table, L = paged_inputs(B, Hq, Hkv, D, page_size, max_pages, lens,
                                       seed=sum(lens) + B)
    scale = 1 / math.sqrt(D)
    o, _ = run_paged(fa, q, kp, vp, table, L, scale)
    compare(o, oracle.decode_paged(q, kp, vp, table.tolist(), L.tolist(), scale))


def _backward_cases(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        hkv = rng.choice([1, 2])
        out.append((rng.choice([1, 2]), hkv * rng.choice([1, 2, 3, 4]), hkv,
                    rng.randint(1, 400), rng.randint(1, 400), rng.choice([64, 128]),
                    rng.random() < 0.6, rng.choice(DTYPES)))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt", _backward_cases(6, 505))
def test_random_backward(fa, B, Hq, Hkv, Sq, Sk, D, causal, dt):
    from tests.test_backward_gpu import grad_compare, run_backward
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed=Sq + 2 * Sk)
    dout = torch.randn(B, Sq, Hq, D, generator=torch.Generator().manual_seed(Sk)).to(dt)
    scale = 1 / math.sqrt(D)
    got = run_backward(fa, q, k, v, dout, scale, causal)
    ref = oracle.attention_bwd(q, k, v, dout, scale, causal)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        grad_compare(g, r, name)
