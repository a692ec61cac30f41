"""Host-to-host prefill through the C ABI (fa_prefill_fwd_host).

CPU: the library's piece plan (fa_prefill_host_pieces) covers every query row
of every sequence once, heaviest piece first, and each piece, taken as a
bottom-right aligned prefill of its own, gives every row exactly the keys it
sees in the whole problem.  GPU: host tensors in, host tensor out, matching
the oracle and bit-identical to fa_prefill_fwd on device copies.
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from tests.parity import compare


@pytest.fixture(scope="module")
def lib():
    from attention_fa_fwd_04_gb300 import build
    build.build()
    import attention_fa_fwd_04_gb300 as fa
    fa.load()
    return fa


def _visible(i, Sq, Sk, causal):
    """Number of keys row i sees (bottom-right causal alignment)."""
    if not causal:
        return Sk
    return min(Sk, max(0, i + (Sk - Sq) + 1))


@pytest.mark.parametrize("B,Sq,Sk,causal,n", [
    (1, 8192, 8192, True, 16), (2, 700, 900, True, 8), (1, 1000, 600, True, 3),
    (3, 1000, 1536, False, 4), (1, 128, 128, True, 8), (2, 1, 5, True, 2), (1, 300, 0, True, 2),
    (1, 257, 257, False, 1)])
def test_pieces_cover_rows_and_keep_each_rows_keys(lib, B, Sq, Sk, causal, n):
    pieces = lib.fa_prefill_host_pieces(B, Sq, Sk, causal, n)
    rows = {b: [] for b in range(B)}
    work = []
    for b, s0, s1, sk in pieces:
        assert 0 <= b < B and 0 <= s0 < s1 <= Sq and 0 <= sk <= Sk
        assert s0 % 256 == 0
        rows[b].extend(range(s0, s1))
        for r in range(s1 - s0):  # the piece as a prefill of its own
            assert _visible(r, s1 - s0, sk, causal) == _visible(s0 + r, Sq, Sk, causal)
        work.append((s1 - s0) * sk)
    for b in range(B):
        assert sorted(rows[b]) == list(range(Sq))
    assert work == sorted(work, reverse=True)  # heaviest first
    assert len(pieces) <= B * max(1, n)


def test_no_rows_no_pieces_and_bad_arguments(lib):
    assert lib.fa_prefill_host_pieces(2, 0, 100, True, 8) == []
    with pytest.raises(ValueError):
        lib.fa_prefill_host_pieces(1, 10, 10, True, 0)


def test_host_prefill_rejects_invalid_arguments(lib):
    fa = lib
    buf = np.zeros(64, dtype=np.uint16)  # never touched: every call is rejected or empty
    p = buf.ctypes.data
    assert fa.fa_prefill_fwd_host(p, p, p, p, 1, 4, 2, 4, 4, 64, 0.1, 1, fa.FA_BF16, 0,
                                  0) == fa.FA_ERR_INVALID_ARG       # n_pieces < 1
    assert fa.fa_prefill_fwd_host(0, p, p, p, 1, 4, 2, 4, 4, 64, 0.1, 1, fa.FA_BF16, 4,
                                  0) == fa.FA_ERR_INVALID_ARG       # null q
    assert fa.fa_prefill_fwd_host(p, p, p, p, 1, 4, 3, 4, 4, 64, 0.1, 1, fa.FA_BF16, 4,
                                  0) == fa.FA_ERR_INVALID_ARG       # Hq % Hkv
    assert fa.fa_prefill_fwd_host(p, p, p, p, 0, 4, 2, 4, 4, 64, 0.1, 1, fa.FA_BF16, 4,
                                  0) == fa.FA_OK                    # empty batch


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt,n", [
    (2, 8, 2, 700, 900, 128, True, torch.bfloat16, 3),
    (1, 4, 4, 1000, 600, 64, True, torch.bfloat16, 16),
    (1, 4, 2, 1000, 1536, 64, False, torch.float16, 4),
    (1, 2, 1, 300, 0, 64, True, torch.bfloat16, 2)])
def test_host_prefill_matches_oracle_and_device_prefill(fa, B, Hq, Hkv, Sq, Sk, D, causal, dt,
                                                         n):
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed=Sq + Sk)
    scale = 1 / math.sqrt(D)
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    op = torch.empty(q.shape, dtype=dt).pin_memory()
    ref = oracle.attention(q, k, v, scale, causal)
    dev = torch.device("cuda", 0)
    dense = fa.prefill(q.to(dev), k.to(dev), v.to(dev), scale, causal).cpu()
    for _ in range(2):  # the per-device streams and events are reused across calls
        op.fill_(float("nan"))
        fa.prefill_host(qp, kp, vp, op, scale, causal, n_pieces=n)
        torch.cuda.synchronize()
        compare(op.float().numpy(), ref)
        assert torch.equal(op, dense)
    assert fa.fa_device_error()[0] == fa.FA_OK
