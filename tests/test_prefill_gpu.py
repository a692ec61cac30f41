"""Prefill parity on the GPU: the tcgen05 path (through the C ABI) against the
fp64 oracle on the same seeded inputs.  Small workloads compare every output
element; the two large ones compare 4096 seeded (b, head, row) samples that
always include rows 0, 1, 127, 128, 255, 256, Sq-1 and the first/last head of
every GQA group."""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare, rounding_bound

pytestmark = pytest.mark.gpu


def run_prefill(fa, q, k, v, scale, causal):
    dev = torch.device("cuda", 0)
    out = fa.prefill(q.to(dev), k.to(dev), v.to(dev), scale, causal)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, f"device error word {detail:#x}"
    return out.float().cpu().numpy()


def full_check(fa, B, Hq, Hkv, Sq, Sk, D, causal, dtype, scale, seed=0, derived_bar=False):
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dtype, seed)
    o = run_prefill(fa, q, k, v, scale, causal)
    ref = oracle.attention(q, k, v, scale, causal)
    if derived_bar:
        bits = 8 if dtype == torch.bfloat16 else 11
        return compare(o, ref, max_abs=rounding_bound(ref, v.abs().max().item(), bits))
    return compare(o, ref)


def test_tiny_causal_gqa(fa):
    s = fa_inputs.TINY_CAUSAL_GQA
    full_check(fa, s.B, s.Hq, s.Hkv, s.Sq, s.Sk, s.D, s.causal, s.dtype, s.scale)


def test_ragged_noncausal_fp16(fa):
    s = fa_inputs.RAGGED_NONCAUSAL
    full_check(fa, s.B, s.Hq, s.Hkv, s.Sq, s.Sk, s.D, s.causal, s.dtype, s.scale)


EDGE = [
    # B, Hq, Hkv, Sq, Sk, D, causal, dtype
    (1, 1, 1, 1, 1, 64, True, torch.bfloat16),
    (1, 2, 1, 1, 1, 128, False, torch.float16),
    (1, 2, 1, 130, 130, 64, True, torch.bfloat16),      # ragged tail past one tile
    (2, 4, 2, 300, 200, 128, True, torch.bfloat16),     # Sq > Sk: fully masked rows
    (1, 4, 4, 77, 333, 128, True, torch.float16),       # Sq < Sk, bottom-right causal
    (1, 8, 2, 257, 513, 64, False, torch.bfloat16),     # ragged both ways
    (3, 6, 3, 256, 256, 128, True, torch.bfloat16),     # exact tile multiples
    (1, 32, 2, 384, 384, 128, True, torch.float16),     # G = 16
    (2, 3, 1, 640, 129, 64, False, torch.float16),      # Sk just past one tile
    (1, 2, 2, 1024, 1024, 128, False, torch.bfloat16),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt", EDGE)
def test_edge_shapes(fa, B, Hq, Hkv, Sq, Sk, D, causal, dt):
    full_check(fa, B, Hq, Hkv, Sq, Sk, D, causal, dt, 1 / math.sqrt(D), seed=B + Sq)


@pytest.mark.parametrize("scale", [0.0, -0.125, 0.5])
def test_unusual_scales(fa, scale):
    """scale 0 (uniform weights), a negative scale, and 4x the usual
    temperature (one key can dominate: the derived rounding bar applies)."""
    full_check(fa, 1, 4, 2, 200, 300, 64, True, torch.bfloat16, scale, seed=7,
               derived_bar=abs(scale) > 0.2)


def test_no_keys_gives_zero(fa):
    dev = torch.device("cuda", 0)
    q = torch.randn(2, 10, 4, 64, device=dev).to(torch.bfloat16)
    k = torch.empty(2, 0, 2, 64, device=dev, dtype=torch.bfloat16)
    out = torch.full_like(q, 3.0)
    fa.prefill(q, k, k, 0.1, False, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.zeros_like(out))


def sampled_check(fa, shape, n=4096):
    q, k, v = fa_inputs.prefill_inputs_for(shape, seed=0)
    dev = torch.device("cuda", 0)
    out = fa.prefill(q.to(dev), k.to(dev), v.to(dev), shape.scale, shape.causal)
    torch.cuda.synchronize()
    assert fa.fa_device_error()[0] == fa.FA_OK
    rows = fa_inputs.sample_rows(shape.B, shape.Hq, shape.Hkv, shape.Sq, n=n, seed=0)
    r = rows.to(dev)
    got = out[r[:, 0], r[:, 2], r[:, 1], :].float().cpu().numpy()
    assert torch.isfinite(out).all().item()
    ref = oracle.attention(q, k, v, shape.scale, shape.causal, rows=rows)
    return compare(got, ref)


def test_mha_causal_4k_sampled(fa):
    sampled_check(fa, fa_inputs.MHA_CAUSAL)


def test_gqa_causal_8k_sampled(fa):
    sampled_check(fa, fa_inputs.GQA_CAUSAL_8K)


def test_repeated_calls_are_identical(fa):
    s = fa_inputs.TINY_CAUSAL_GQA
    q, k, v = fa_inputs.prefill_inputs(2, 8, 2, 700, 700, 128, torch.bfloat16, 11)
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    a = fa.prefill(qd, kd, vd, 0.09, True)
    b = fa.prefill(qd, kd, vd, 0.09, True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_work_counter_across_calls_and_streams(fa):
    """Persistent CTAs claim work items from a per-stream counter that the last
    CTA of each launch zeroes again.  Launches on one stream, interleaved with
    launches on a second stream, must each cover every item exactly once: the
    outputs are bit-identical (each item's arithmetic does not depend on which
    CTA runs it) and match the oracle."""
    q, k, v = fa_inputs.prefill_inputs(1, 16, 4, 1500, 1500, 64, torch.bfloat16, 21)
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    side = torch.cuda.Stream()
    main_outs, side_outs = [], []
    for _ in range(4):
        main_outs.append(fa.prefill(qd, kd, vd, 0.125, True))
        with torch.cuda.stream(side):
            side_outs.append(fa.prefill(qd, kd, vd, 0.125, True, stream=side))
    torch.cuda.synchronize()
    for o in main_outs[1:] + side_outs:
        assert torch.equal(o, main_outs[0])
    compare(main_outs[0].float().cpu().numpy(), oracle.attention(q, k, v, 0.125, True))
    assert fa.fa_device_error()[0] == fa.FA_OK


def test_output_aligned_to_16_bytes_only(fa):
    """At D = 128 the epilogue uses 32-byte stores when O's base is 32-byte
    aligned and 16-byte stores otherwise (the ABI asks for 16).  An output
    view 16 bytes into a buffer takes the second path; both must give the
    same bits, and match the oracle."""
    dev = torch.device("cuda", 0)
    B, Hq, Hkv, S, D = 1, 8, 2, 640, 128
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, S, S, D, torch.bfloat16, seed=41)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    n = q.numel()
    buf = torch.empty(n + 8, dtype=torch.bfloat16, device=dev)
    assert buf.data_ptr() % 32 == 0
    out16 = buf[8:8 + n].view(q.shape)  # 16 bytes past a 32-byte boundary
    assert out16.data_ptr() % 32 == 16
    fa.prefill(qd, kd, vd, 1 / math.sqrt(D), True, out=out16)
    out32 = fa.prefill(qd, kd, vd, 1 / math.sqrt(D), True)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, hex(detail)
    assert torch.equal(out16, out32)
    compare(out16.float().cpu().numpy(), oracle.attention(q, k, v, 1 / math.sqrt(D), True))
