"""Decode parity on the GPU: the CUDA split-KV path (through the C ABI) against
the fp64 oracle on the same seeded inputs, with NaN-poisoned unused capacity
(rocm-libraries #13108, review finding on unused V-cache NaNs)."""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare

pytestmark = pytest.mark.gpu


def run_decode(fa, q, kc, vc, L, scale):
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), kc.to(dev), vc.to(dev)
    vl = torch.tensor([L], dtype=torch.int32, device=dev)
    out = fa.decode(qd, kd, vd, vl, scale)
    torch.cuda.synchronize()
    st, detail = fa.fa_device_error()
    assert st == fa.FA_OK, f"device error word {detail:#x}"
    return out.float().cpu().numpy().reshape(q.shape[0], -1, q.shape[-1])


def test_worked_example_nan_tail_capacity_128_length_1(fa):
    """Capacity 128, valid length 1, V tail = bf16 0x7fc0: O equals V[0]."""
    q, kc, vc, L = fa_inputs.decode_inputs(1, 8, 2, 128, 128, seed=0, L=1, poison_k=False)
    o = run_decode(fa, q, kc, vc, L, 1 / math.sqrt(128))
    v0 = vc[0, 0].float().numpy()
    for h in range(8):
        assert np.array_equal(o[0, h], v0[h // 4]), h


def test_single_token_decode_seeded_length(fa):
    s = fa_inputs.DECODE_1TOK
    q, kc, vc, L = fa_inputs.decode_inputs_for(s, seed=0)
    o = run_decode(fa, q, kc, vc, L, s.scale)
    ref = oracle.decode(q, kc, vc, L, s.scale)
    compare(o, ref)


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 127, 1000, 4097, 65535, 65536])
def test_single_token_decode_lengths(fa, L):
    s = fa_inputs.DECODE_1TOK
    q, kc, vc, L = fa_inputs.decode_inputs_for(s, seed=1, L=L)
    o = run_decode(fa, q, kc, vc, L, s.scale)
    compare(o, oracle.decode(q, kc, vc, L, s.scale))


@pytest.mark.parametrize("L,expect", [(0, "zero"), (-7, "zero"), (5000, "cap")])
def test_valid_length_is_clamped(fa, L, expect):
    q, kc, vc, _ = fa_inputs.decode_inputs(1, 8, 2, 3000, 128, seed=2, L=3000)
    o = run_decode(fa, q, kc, vc, L, 0.1)
    if expect == "zero":
        assert np.array_equal(o, np.zeros_like(o))
    else:
        compare(o, oracle.decode(q, kc, vc, 3000, 0.1))


@pytest.mark.parametrize("B,Hq,Hkv,cap,D,L", [
    (3, 8, 2, 700, 128, 513),     # batch > 1
    (1, 32, 2, 900, 128, 900),    # G = 16: one full head block
    (2, 40, 2, 300, 64, 251),     # G = 20: two head blocks, D = 64
    (1, 4, 4, 200, 64, 77),       # MHA
    (2, 6, 1, 100, 128, 100),     # G = 6, no tail
    (1, 16, 2, 500, 128, 333),    # G = 8: one full 8-row block
])
def test_decode_shapes(fa, B, Hq, Hkv, cap, D, L):
    q, kc, vc, L = fa_inputs.decode_inputs(B, Hq, Hkv, cap, D, seed=3, L=L)
    scale = 1 / math.sqrt(D)
    compare(run_decode(fa, q, kc, vc, L, scale), oracle.decode(q, kc, vc, L, scale))


def test_decode_negative_scale(fa):
    q, kc, vc, L = fa_inputs.decode_inputs(1, 8, 2, 500, 128, seed=4, L=333)
    compare(run_decode(fa, q, kc, vc, L, -0.09), oracle.decode(q, kc, vc, L, -0.09))


def test_decode_zero_capacity(fa):
    dev = torch.device("cuda", 0)
    q = torch.randn(1, 1, 8, 128, device=dev).to(torch.bfloat16)
    kc = torch.empty(1, 0, 2, 128, device=dev, dtype=torch.bfloat16)
    vl = torch.zeros(1, dtype=torch.int32, device=dev)
    out = fa.decode(q, kc, kc, vl, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.zeros_like(out))


def test_decode_repeated_calls_and_side_stream(fa):
    s = fa_inputs.DECODE_1TOK
    q, kc, vc, L = fa_inputs.decode_inputs_for(s, seed=5, L=20000)
    ref = oracle.decode(q, kc, vc, L, s.scale)
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), kc.to(dev), vc.to(dev)
    vl = torch.tensor([L], dtype=torch.int32, device=dev)
    side = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(side):
        for _ in range(3):
            outs.append(fa.decode(qd, kd, vd, vl, s.scale, stream=side))
    torch.cuda.synchronize()
    for o in outs:
        compare(o.float().cpu().numpy().reshape(1, 8, 128), ref)
    assert fa.fa_device_error()[0] == fa.FA_OK
