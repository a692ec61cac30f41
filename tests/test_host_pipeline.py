"""Host-to-host prefill (attention_fa_fwd_04_gb300.host_pipeline).

CPU: the row pieces cover every query row once, and each piece, taken as a
bottom-right aligned prefill of its own, gives every row exactly the keys it
sees in the whole problem.  GPU: HostPrefill from pinned host tensors matches
the oracle.
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from attention_fa_fwd_04_gb300.host_pipeline import prefill_row_chunks
from tests.parity import compare


def _visible(i, Sq, Sk, causal):
    """Number of keys row i sees (bottom-right causal alignment)."""
    if not causal:
        return Sk
    return min(Sk, max(0, i + (Sk - Sq) + 1))


@pytest.mark.parametrize("Sq,Sk,causal,n", [
    (8192, 8192, True, 8), (700, 900, True, 8), (1000, 600, True, 3), (1000, 1536, False, 4),
    (128, 128, True, 8), (1, 5, True, 2), (300, 0, True, 2), (257, 257, False, 1)])
def test_row_pieces_cover_rows_and_keep_each_rows_keys(Sq, Sk, causal, n):
    pieces = prefill_row_chunks(Sq, Sk, causal, n)
    rows = []
    for s0, s1, sk in pieces:
        assert 0 <= s0 < s1 <= Sq and 0 <= sk <= Sk
        assert s0 % 256 == 0
        rows.extend(range(s0, s1))
        for r in range(s1 - s0):  # the piece as a prefill of its own
            assert _visible(r, s1 - s0, sk, causal) == _visible(s0 + r, Sq, Sk, causal)
    assert rows == list(range(Sq))
    assert len(pieces) <= max(1, n)


def test_no_rows_no_pieces():
    assert prefill_row_chunks(0, 100, True, 8) == []


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Sk,D,causal,dt", [
    (2, 8, 2, 700, 900, 128, True, torch.bfloat16),
    (1, 4, 4, 1000, 600, 64, True, torch.bfloat16),
    (1, 4, 2, 1000, 1536, 64, False, torch.float16)])
def test_host_prefill_matches_oracle(fa, B, Hq, Hkv, Sq, Sk, D, causal, dt):
    from attention_fa_fwd_04_gb300.host_pipeline import HostPrefill
    q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed=Sq + Sk)
    scale = 1 / math.sqrt(D)
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    op = torch.empty(q.shape, dtype=dt).pin_memory()
    hp = HostPrefill(B, Hq, Hkv, Sq, Sk, D, dt, causal, n_chunks=3)
    ref = oracle.attention(q, k, v, scale, causal)
    for _ in range(2):  # the object is reused across calls
        op.zero_()
        hp(qp, kp, vp, op, scale)
        torch.cuda.synchronize()
        compare(op.float().numpy(), ref)
    assert np.isfinite(op.float().numpy()).all()
    assert fa.fa_device_error()[0] == fa.FA_OK
